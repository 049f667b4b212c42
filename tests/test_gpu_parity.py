"""Parity of libmuon (through its C ABI) with the float64 oracle on the GPU.

Sizes here are ones the oracle finishes in seconds while spanning several
128 x 256 tensor-core tiles, 64 x 64 element-wise tiles and ragged tails.
The single fp32 256 x 512 matrix and the chained default-size cases are
gated at relF(W) <= 1e-3; the small shapes made to reach ragged tiles use
the size-scaled weight gate (w_gate="scaled", see gpu_helpers).
"""
import warnings

import numpy as np
import pytest
import torch

from gpu_helpers import (check_against_oracle, gpu_step, oracle_step, relF,
                         to_np)
from newton_schulz_06_gb300 import Muon, mode_code
from newton_schulz_06_gb300.inputs import random_case, workload, make_state

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


def case(rows, cols, seed, **kw):
    W, G, M = random_case(rows, cols, seed, device=DEV, **kw)
    return [W, G, M]


def test_single_matrix_256x512_f32():
    """The single fp32 matrix workload: G, M ~ N(0,1), W ~ N(0, 0.02)."""
    wl = workload("single_256x512_f32")
    Ws, Gs, Ms = make_state(wl, DEV)
    trip = [Ws[0], Gs[0], Ms[0]]
    inp, wexp, oexp, _ = gpu_step([trip])
    ref = oracle_step(inp[0])
    errs = check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref)
    print("256x512 f32", errs)


@pytest.mark.parametrize("rows,cols", [(8, 16), (16, 8), (100, 37), (37, 100),
                                       (130, 130), (200, 333), (333, 200),
                                       (257, 129), (576, 1024), (1024, 576),
                                       (384, 1000)])
def test_ragged_shapes_bf16(rows, cols):
    trip = case(rows, cols, 1)
    inp, wexp, oexp, _ = gpu_step([trip])
    ref = oracle_step(inp[0])
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")


@pytest.mark.parametrize("nesterov", [False, True])
def test_f32_grad_bf16_weight_nesterov_flag(nesterov):
    trip = case(192, 320, 2, g_dtype=torch.float32)
    inp, wexp, oexp, _ = gpu_step([trip], nesterov=nesterov)
    ref = oracle_step(inp[0], nesterov=nesterov)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")


def test_grouped_matches_oracle_and_standalone_bitexact():
    shapes = [(256, 768), (768, 256), (512, 512), (130, 390), (64, 64)]
    trips = [case(r, c, 10 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    inp, wexp, oexp, _ = gpu_step(trips)
    for i, tr in enumerate(trips):
        ref = oracle_step(inp[i])
        check_against_oracle(tr, inp[i], wexp[i], oexp[i], ref, w_gate="scaled")
    # each matrix stepped alone gives the same bits
    for i, tr in enumerate(clones):
        _, w1, o1, _ = gpu_step([tr])
        assert torch.equal(o1[0], oexp[i]), shapes[i]
        assert torch.equal(tr[0], trips[i][0]) and torch.equal(tr[2], trips[i][2])


def test_groups_from_a_small_workspace_bitexact():
    shapes = [(256, 512), (512, 256), (384, 384), (128, 640)]
    trips = [case(r, c, 30 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    _, _, o_big, opt = gpu_step(trips, steps=2)
    mn, full = opt.workspace_size()
    _, _, o_small, opt2 = gpu_step(clones, max_workspace=mn, steps=2)
    assert opt2.plan_info()["groups"] > 1
    for a, b in zip(o_big, o_small):
        assert torch.equal(a, b)


@pytest.mark.parametrize("rows,cols,nb", [(256, 1024, 4), (1024, 512, 4),
                                          (300, 600, 3), (128, 2048, 8),
                                          (256, 606, 3), (606, 300, 2)])
def test_blockwise_matches_oracle(rows, cols, nb):
    """Blockwise mode against the oracle's; 202- and 150-column blocks start
    at unaligned addresses (no 16-byte or TMA access to W, G, M there)."""
    trip = case(rows, cols, 40)
    inp, wexp, oexp, _ = gpu_step([trip], mode="blockwise", nb=nb)
    ref = oracle_step(inp[0], mode="blockwise", nb=nb)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref,
                         mode="blockwise", nb=nb, w_gate="scaled")


def test_blockwise_nb1_is_full_bitexact():
    t1 = case(320, 640, 50)
    t2 = [t.clone() for t in t1]
    _, _, o1, _ = gpu_step([t1])
    _, _, o2, _ = gpu_step([t2], mode="blockwise", nb=1)
    assert torch.equal(o1[0], o2[0]) and torch.equal(t1[0], t2[0])


def test_blockwise_block_is_full_on_the_copied_block_bitexact():
    t = case(256, 1024, 51)
    blk = [x[:, 512:768].contiguous() for x in t]
    _, _, o_all, _ = gpu_step([t], mode="blockwise", nb=4)
    _, _, o_blk, _ = gpu_step([blk])
    assert torch.equal(o_all[0][:, 512:768], o_blk[0])


def test_transpose_invariance_bitexact():
    t = case(192, 448, 60)
    tt = [x.t().contiguous() for x in t]
    _, _, o1, _ = gpu_step([t])
    _, _, o2, _ = gpu_step([tt])
    assert torch.equal(o1[0], o2[0].t())


def test_zero_gradient_leaves_weight_unchanged():
    W, G, M = case(160, 288, 70, momentum="zero")
    G.zero_()
    W0 = W.clone()
    _, wexp, oexp, _ = gpu_step([[W, G, M]])
    assert torch.equal(W, W0)
    assert torch.count_nonzero(oexp[0]) == 0
    assert not torch.isnan(wexp[0]).any()


def test_repeat_runs_bitexact():
    t1 = case(300, 700, 80)
    t2 = [x.clone() for x in t1]
    _, _, o1, _ = gpu_step([t1], steps=2)
    _, _, o2, _ = gpu_step([t2], steps=2)
    assert torch.equal(o1[0], o2[0]) and torch.equal(t1[0], t2[0])
    assert torch.equal(t1[2], t2[2])


def test_ns_steps_and_coefficients_are_honoured():
    trip = case(256, 384, 90)
    coeffs = (2.0, -1.5, 0.5)
    inp, wexp, oexp, _ = gpu_step([trip], ns_steps=3, coeffs=coeffs)
    ref = oracle_step(inp[0], ns_steps=3, coeffs=coeffs)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")


def test_output_singular_values_in_band():
    """Normalised singular values >= 1.5e-3 map into p^5's band."""
    trip = case(256, 1024, 95, momentum="zero")
    inp, _, oexp, _ = gpu_step([trip], nesterov=False)
    s_out = np.linalg.svd(to_np(oexp[0]), compute_uv=False)
    assert s_out.min() > 0.6818 - 0.03 and s_out.max() < 1.2024 + 0.03


@pytest.mark.parametrize("fuse_env", [{"MUON_FUSE": "0"},
                                      {"MUON_FUSE_UPDATE": "0"},
                                      {"MUON_FUSE_UPDATE": "1"},
                                      {"MUON_FUSE_STAGES": "0"},
                                      {"MUON_CTA_GROUP": "1"}])
def test_alternative_pipelines_match_oracle(fuse_env, monkeypatch):
    """The unfused pipeline, the update fused into the last GEMM, and the
    single-CTA kernels all meet the same tolerances."""
    for k, v in fuse_env.items():
        monkeypatch.setenv(k, v)
    shapes = [(256, 640), (640, 256), (300, 300), (96, 1000)]
    trips = [case(r, c, 200 + i, w_dtype=torch.float32 if i == 2 else torch.bfloat16)
             for i, (r, c) in enumerate(shapes)]
    inp, wexp, oexp, _ = gpu_step(trips)
    for i, tr in enumerate(trips):
        ref = oracle_step(inp[i])
        check_against_oracle(tr, inp[i], wexp[i], oexp[i], ref, w_gate="scaled")


def test_update_folded_into_gemm_matches_separate_pass_bitexact(monkeypatch):
    """The update folded into the last GEMM (TMA-loaded W blocks) and the
    separate update pass apply the same arithmetic: identical bits."""
    shapes = [(256, 640), (640, 256), (300, 300), (96, 1000), (768, 2048)]
    trips = [case(r, c, 300 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    _, w1, o1, _ = gpu_step(trips)
    monkeypatch.setenv("MUON_FUSE_UPDATE", "0")
    _, w2, o2, _ = gpu_step(clones)
    for i in range(len(shapes)):
        assert torch.equal(trips[i][0], clones[i][0]), shapes[i]
        assert torch.equal(w1[i], w2[i]) and torch.equal(o1[i], o2[i]), shapes[i]


@pytest.mark.parametrize("rows,cols,P", [(256, 1024, 4), (1024, 512, 2),
                                         (384, 1536, 8), (768, 2048, 4),
                                         (200, 640, 2)])
def test_distributed_mode_matches_oracle(rows, cols, P):
    """Distributed mode (P slices of the long side; the partial first
    products summed in slice order) against the oracle's distributed mode."""
    trip = case(rows, cols, 600 + P)
    inp, wexp, oexp, _ = gpu_step([trip], mode="distributed", nb=P)
    ref = oracle_step(inp[0], mode="distributed", nb=P)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")


def test_distributed_one_slice_is_full_mode_bitexact():
    t1 = case(512, 1024, 610)
    t2 = [t.clone() for t in t1]
    _, w1, o1, _ = gpu_step([t1])
    _, w2, o2, _ = gpu_step([t2], mode="distributed", nb=1)
    assert torch.equal(o1[0], o2[0]) and torch.equal(t1[0], t2[0])


def test_distributed_mode_reproducible_and_standalone_bitexact():
    """The slice sum has a fixed order: repeated runs and a matrix stepped
    alone or in a group give the same bits, over two steps (the slot
    counters carry across launches and steps)."""
    shapes = [(512, 2048), (2048, 512), (768, 1024)]
    trips = [case(r, c, 620 + i) for i, (r, c) in enumerate(shapes)]
    again = [[t.clone() for t in tr] for tr in trips]
    alone = [t.clone() for t in trips[1]]
    _, _, o1, _ = gpu_step(trips, mode="distributed", nb=4, steps=2)
    _, _, o2, _ = gpu_step(again, mode="distributed", nb=4, steps=2)
    _, _, o3, _ = gpu_step([alone], mode="distributed", nb=4, steps=2)
    for i in range(len(shapes)):
        assert torch.equal(o1[i], o2[i]), shapes[i]
        assert torch.equal(trips[i][0], again[i][0]), shapes[i]
    assert torch.equal(o1[1], o3[0]) and torch.equal(trips[1][0], alone[0])


@pytest.mark.parametrize("mode,nb,shapes", [
    ("full", 1, [(256, 640), (640, 256), (300, 300)]),
    ("blockwise", 4, [(256, 640), (640, 256), (300, 300)]),
    ("distributed", 2, [(256, 640), (640, 256), (384, 512)])])
def test_step_with_host_buffers_matches_device_step_bitexact(mode, nb, shapes):
    """muon_step_host: gradients in from pinned host memory, weights back out,
    gives the same bits as copying G in and W out around muon_step, in each
    mode."""
    trips = [case(r, c, 700 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    g_host = [torch.randn(r, c, generator=torch.Generator().manual_seed(710 + i)
                          ).to(torch.bfloat16).pin_memory() for i, (r, c) in enumerate(shapes)]
    w_host = [torch.empty(r, c, dtype=torch.bfloat16).pin_memory() for r, c in shapes]
    md = mode_code(mode)
    opt = Muon(trips)
    opt.step_host(g_host, w_host, mode=md, nb=nb)
    opt.sync()
    ref = Muon(clones)
    for (W, G, M), g in zip(clones, g_host):
        G.copy_(g)
    ref.step(mode=md, nb=nb)
    ref.sync()
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(w_host[i], clones[i][0].cpu()), shapes[i]
        assert torch.equal(trips[i][0], clones[i][0]) and torch.equal(trips[i][2], clones[i][2])


def test_layerwise_single_rank_is_the_grouped_step_bitexact():
    """With one rank the layer-wise optimizer owns every matrix: its step is
    libmuon's grouped step (same bits, momentum kept by the optimizer)."""
    from newton_schulz_06_gb300.layerwise import LayerwiseMuon
    shapes = [(256, 640), (640, 256), (300, 300), (96, 1000)]
    trips = [case(r, c, 800 + i, momentum="zero") for i, (r, c) in enumerate(shapes)]
    W2 = [t[0].clone() for t in trips]
    G2 = [t[1].clone() for t in trips]
    opt = Muon(trips)
    lw = LayerwiseMuon(W2, G2)
    assert lw.world == 1 and lw.owned == list(range(len(shapes)))
    for _ in range(2):
        opt.step()
        lw.step()
    opt.sync()
    lw.sync()
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(trips[i][0], W2[i]), shapes[i]
        assert torch.equal(trips[i][2], lw.momentum[i]), shapes[i]


@pytest.mark.parametrize("ns_steps", [1, 2, 5, 64])
def test_chained_launch_bitexact(ns_steps, monkeypatch):
    """One launch holding every product of the step but the last X update
    (tiles waiting on row-block counters) computes every tile as the
    separate launches do: identical bits, over two steps (the counters carry
    across launches and steps), up to the largest iteration count the ABI
    accepts (64: counter targets of 16 x 64 rounds)."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")     # small shapes chain too
    shapes = [(512, 768), (768, 2048), (300, 300), (2048, 640), (96, 1000)]
    trips = [case(r, c, 900 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    _, w1, o1, opt = gpu_step(trips, ns_steps=ns_steps, steps=2)
    assert opt.plan_info()["chained_groups"] == 1
    monkeypatch.setenv("MUON_FUSE_STAGES", "0")
    _, w2, o2, opt2 = gpu_step(clones, ns_steps=ns_steps, steps=2)
    assert opt2.plan_info()["chained_groups"] == 0
    for i in range(len(shapes)):
        assert torch.equal(o1[i], o2[i]), shapes[i]
        assert torch.equal(trips[i][0], clones[i][0]), shapes[i]


@pytest.mark.parametrize("rows,cols,ns_steps", [(200, 200, 1), (200, 200, 3),
                                                (256, 1024, 2), (1000, 300, 5)])
def test_chained_launch_small_matrix_matches_oracle(rows, cols, ns_steps, monkeypatch):
    """A chain over a few tiles leaves most CTA pairs idle and gives some
    pairs only X-update tiles (which they skip in the last iteration): same
    bits as separate launches, within tolerance of the oracle."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")     # small shapes chain too
    trip = case(rows, cols, 970)
    clone = [t.clone() for t in trip]
    inp, wexp, oexp, opt = gpu_step([trip], ns_steps=ns_steps)
    assert opt.plan_info()["chained_groups"] == 1
    ref = oracle_step(inp[0], ns_steps=ns_steps)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")
    monkeypatch.setenv("MUON_FUSE_STAGES", "0")
    _, _, o2, _ = gpu_step([clone], ns_steps=ns_steps)
    assert torch.equal(oexp[0], o2[0])
    assert torch.equal(trip[0], clone[0])


@pytest.mark.parametrize("ns_steps", [1, 2, 5])
def test_chained_last_update_bitexact(ns_steps, monkeypatch):
    """With no validation exports registered the chained launch also runs the
    last X update, the weight update folded in: the weights come out
    bit-identical to the last X update run alone and to one launch per
    product, over two steps (plain and transposed units, one pair holding a
    few tiles)."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")     # small shapes chain too
    shapes = [(512, 768), (768, 2048), (300, 300), (2048, 640), (96, 1000)]
    runs = []
    for env in ({}, {"MUON_CHAIN_LAST": "0"}, {"MUON_FUSE_STAGES": "0"}):
        for k in ("MUON_CHAIN_LAST", "MUON_FUSE_STAGES"):
            monkeypatch.delenv(k, raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        trips = [case(r, c, 990 + i) for i, (r, c) in enumerate(shapes)]
        _, _, _, opt = gpu_step(trips, ns_steps=ns_steps, steps=2, exports=False)
        runs.append([t[0].clone() for t in trips])
        if not env:
            assert opt.plan_info()["chained_groups"] == 1
    for i in range(len(shapes)):
        assert torch.equal(runs[0][i], runs[1][i]), shapes[i]
        assert torch.equal(runs[0][i], runs[2][i]), shapes[i]


@pytest.mark.parametrize("chain_max", ["8", "0"])
def test_update_without_exports_matches_exported_bitexact(chain_max, monkeypatch):
    """The weight update folded into the last X update has an export-writing
    form (validated against the oracle elsewhere) and the production forms
    (8-element pieces; inside the chained launch when the group chains):
    identical weights, plain and transposed units."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")     # small shapes chain too
    monkeypatch.setenv("MUON_CHAIN_MAX_TILES", chain_max)
    shapes = [(768, 1024), (1024, 384), (300, 700)]
    a = [case(r, c, 1000 + i) for i, (r, c) in enumerate(shapes)]
    b = [[t.clone() for t in tr] for tr in a]
    _, _, _, opt = gpu_step(a, steps=2, exports=True)
    gpu_step(b, steps=2, exports=False)
    assert opt.plan_info()["chained_groups"] == (1 if chain_max == "8" else 0)
    for i in range(len(shapes)):
        assert torch.equal(a[i][0], b[i][0]), shapes[i]


def test_chained_last_update_single_small_matrix_bitexact(monkeypatch):
    """A chain over three tiles (some pairs hold only X-update tiles, which
    now also run in the last iteration) gives the same weights as separate
    launches."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")     # small shapes chain too
    out = []
    for env in ({}, {"MUON_FUSE_STAGES": "0"}):
        monkeypatch.delenv("MUON_FUSE_STAGES", raising=False)
        for k, v in env.items():
            monkeypatch.setenv(k, v)
        trip = case(200, 456, 995)
        gpu_step([trip], ns_steps=3, steps=2, exports=False)
        out.append(trip[0].clone())
    assert torch.equal(out[0], out[1])


@pytest.mark.parametrize("rows,cols,mode,nb", [(6144, 1536, "full", 1),
                                               (2048, 4096, "blockwise", 2)])
def test_chained_default_sizes_match_oracle(rows, cols, mode, nb, monkeypatch):
    """Steps that chain under the default bounds (at least one X-update tile
    per CTA pair): a tall matrix (transposed unit) and two column blocks.
    Within tolerance of the oracle, and the same bits as one launch per
    product."""
    trip = case(rows, cols, 1010)
    clone = [t.clone() for t in trip]
    inp, wexp, oexp, opt = gpu_step([trip], mode=mode, nb=nb)
    assert opt.plan_info(mode_code(mode), nb)["chained_groups"] == 1
    ref = oracle_step(inp[0], mode=mode, nb=nb)
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, mode=mode, nb=nb)
    monkeypatch.setenv("MUON_FUSE_STAGES", "0")
    _, _, o2, _ = gpu_step([clone], mode=mode, nb=nb)
    assert torch.equal(oexp[0], o2[0])
    assert torch.equal(trip[0], clone[0])


def test_chained_groups_from_a_small_workspace_bitexact(monkeypatch):
    """A workspace that holds one matrix at a time: every group runs its own
    chained launch (own counter block and rounds), over two steps, with the
    same bits as one launch per product."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")
    shapes = [(1024, 2048), (768, 1536), (1536, 768), (512, 2048)]
    a = [case(r, c, 1030 + i) for i, (r, c) in enumerate(shapes)]
    b = [[t.clone() for t in tr] for tr in a]
    probe = Muon(a)
    mn, _ = probe.workspace_size()
    probe.close()
    _, _, o1, opt = gpu_step(a, steps=2, max_workspace=mn)
    info = opt.plan_info()
    assert info["groups"] > 1 and info["chained_groups"] == info["groups"], info
    monkeypatch.setenv("MUON_FUSE_STAGES", "0")
    _, _, o2, _ = gpu_step(b, steps=2, max_workspace=mn)
    for i in range(len(shapes)):
        assert torch.equal(o1[i], o2[i]), shapes[i]
        assert torch.equal(a[i][0], b[i][0]), shapes[i]


def test_chained_fp32_weights_match_oracle(monkeypatch):
    """fp32 weights (no TMA-folded update): the chain stops before the last X
    update and the separate update pass writes W; within tolerance of the
    oracle and the same bits as one launch per product."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")
    trip = case(768, 1536, 1040, w_dtype=torch.float32, g_dtype=torch.float32)
    clone = [t.clone() for t in trip]
    inp, wexp, oexp, opt = gpu_step([trip])
    assert opt.plan_info()["chained_groups"] == 1
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], oracle_step(inp[0]))
    monkeypatch.setenv("MUON_FUSE_STAGES", "0")
    _, _, o2, _ = gpu_step([clone])
    assert torch.equal(oexp[0], o2[0])
    assert torch.equal(trip[0], clone[0])


@pytest.mark.parametrize("shapes", [[(1024, 5120)], [(256, 768), (768, 256), (300, 300)]])
def test_step_captured_in_cuda_graph_replays_bitexact(shapes):
    """A step captured into a CUDA graph (after one plain step has built the
    plan) and replayed gives the same bits as plain steps: one group that
    chains (the last CTA of every chained launch zeroes its tile counters,
    so replays carry no stale counts) and one that runs a launch per product.
    Plain steps after the replays stay in agreement too."""
    trips = [case(r, c, 960 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    s = torch.cuda.Stream()
    a = Muon(trips, stream=s)
    b = Muon(clones, stream=s)
    with torch.cuda.stream(s):
        a.step()
        b.step()
    a.sync()
    b.sync()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        a.step()
    for _ in range(3):
        g.replay()
        with torch.cuda.stream(s):
            b.step()
    with torch.cuda.stream(s):
        a.step()
        b.step()
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        assert torch.equal(trips[i][0], clones[i][0]), shapes[i]
        assert torch.equal(trips[i][2], clones[i][2]), shapes[i]
    a.close()
    b.close()


def test_capture_before_the_plan_exists_is_refused():
    """The plan's first build uploads tables from host memory, which a
    graph must not capture: muon_step refuses while capturing."""
    trip = case(256, 512, 970)
    s = torch.cuda.Stream()
    opt = Muon([trip], stream=s)
    opt.ensure_workspace(mode_code("full"), 1)
    g = torch.cuda.CUDAGraph()
    with warnings.catch_warnings():
        warnings.simplefilter("ignore")        # the refused capture is empty
        with pytest.raises(Exception):
            with torch.cuda.graph(g, stream=s):
                opt.step()
    torch.cuda.synchronize()
    opt.close()


@pytest.mark.parametrize("mode,nb", [("full", 1), ("blockwise", 4)])
def test_momentum_pass_tma_and_plain_loads_bitexact(mode, nb, monkeypatch):
    """The momentum pass fed by TMA (groups whose momenta and gradients suit
    it) and the pass with plain loads give identical bits: the same element
    map, arithmetic and summation order.  Plain and transposed units, ragged
    edges, fp32 gradients, two steps (momentum carried)."""
    shapes = [(256, 1024), (1024, 256), (320, 640), (64, 2048)]
    a = [case(r, c, 1100 + i, g_dtype=torch.float32 if i == 2 else torch.bfloat16)
         for i, (r, c) in enumerate(shapes)]
    if mode == "full":
        a.append(case(300, 300, 1105))
    b = [[t.clone() for t in tr] for tr in a]
    monkeypatch.setenv("MUON_EW_TMA", "2")
    _, w1, o1, opt = gpu_step(a, steps=2, mode=mode, nb=nb)
    monkeypatch.setenv("MUON_EW_TMA", "0")
    _, w2, o2, _ = gpu_step(b, steps=2, mode=mode, nb=nb)
    for i in range(len(a)):
        assert torch.equal(o1[i], o2[i]), i
        assert torch.equal(a[i][0], b[i][0]) and torch.equal(a[i][2], b[i][2]), i


def test_pipelined_host_step_matches_device_step_bitexact():
    """muon_step_host over a set large enough to be cut into several groups
    (gradients of one group copied in while another computes, weights of a
    finished group copied out while the next computes): two steps give the
    same bits as copying G in and W out around muon_step."""
    shapes = [(2048, 4096)] * 6 + [(4096, 2048)] * 3 + [(768, 2048)] * 4
    trips = [case(r, c, 1200 + i) for i, (r, c) in enumerate(shapes)]
    clones = [[t.clone() for t in tr] for tr in trips]
    opt = Muon(trips)
    ref = Muon(clones)
    for step in range(2):
        g_host = [torch.randn(r, c, generator=torch.Generator().manual_seed(1300 + 17 * step + i)
                              ).to(torch.bfloat16).pin_memory()
                  for i, (r, c) in enumerate(shapes)]
        w_host = [torch.empty(r, c, dtype=torch.bfloat16).pin_memory() for r, c in shapes]
        opt.step_host(g_host, w_host)
        opt.sync()
        for (W, G, M), g in zip(clones, g_host):
            G.copy_(g)
        ref.step()
        ref.sync()
        torch.cuda.synchronize()
        # the pipelined plan (three groups here, each of which chains) is not
        # the single group that muon_step plans for the same set
        assert opt.last_launch_count() != ref.last_launch_count()
        for i in range(len(shapes)):
            assert torch.equal(w_host[i], clones[i][0].cpu()), (step, shapes[i])
            assert torch.equal(trips[i][0], clones[i][0]), (step, shapes[i])
            assert torch.equal(trips[i][2], clones[i][2]), (step, shapes[i])
    opt.close()
    ref.close()


@pytest.mark.parametrize("pad,offset,chained", [(64, 0, False), (40, 3, False),
                                                (64, 0, True), (40, 3, True)])
def test_padded_and_offset_layouts_bitexact(pad, offset, chained, monkeypatch):
    """W, G and M as column views of wider buffers (leading dimension
    cols + pad, first column `offset`): the same bits as contiguous tensors,
    and nothing written outside the views (the padding keeps its sentinel).
    offset 3 leaves every row start unaligned, which rules out the TMA and
    16-byte paths; pad 64 keeps them.  Separate launches over a mixed group,
    and a chained launch over one matrix."""
    shapes = [(256, 640), (640, 256), (300, 300), (768, 2048)]
    if chained:
        monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")
        shapes = [(1024, 2048)]
    ref = [case(r, c, 1400 + i) for i, (r, c) in enumerate(shapes)]
    bigs, views = [], []
    for (W, G, M) in ref:
        r, c = W.shape
        trip_big, trip_view = [], []
        for t in (W, G, M):
            big = torch.full((r, c + pad), 7.0, dtype=t.dtype, device=DEV)
            v = big[:, offset:offset + c]
            v.copy_(t)
            trip_big.append(big)
            trip_view.append(v)
        bigs.append(trip_big)
        views.append(trip_view)
    for _ in range(2):
        gpu_step(ref, exports=False)
        *_, opt = gpu_step(views, exports=False)
        assert opt.plan_info()["chained_groups"] == (1 if chained else 0)
    torch.cuda.synchronize()
    for i in range(len(shapes)):
        for k in (0, 2):                               # W and M
            assert torch.equal(views[i][k], ref[i][k]), (shapes[i], k)
        c = shapes[i][1]
        for big in bigs[i]:
            keep = torch.ones(big.shape[1], dtype=torch.bool, device=DEV)
            keep[offset:offset + c] = False
            assert bool((big[:, keep] == 7.0).all()), shapes[i]
