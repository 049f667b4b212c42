"""Parity at the workloads' full sizes, in the launch configuration the
benchmark times (every matrix of the workload in one grouped step).

The oracle checks a seeded sample of matrices (teacher-forced for multi-step
runs: it starts from the GPU's state before the checked step).  Every other
matrix is covered by properties that hold at any size:
  * its O has the Frobenius norm of p^5's band: the squared singular values
    of O lie in [0.6818^2, 1.2024^2] once the input's normalised singular
    values exceed 1.5e-3, so ||O||_F^2 / m lies in [0.46, 1.45] (a missed
    tile, a wrong block offset or a stale buffer falls outside);
  * the stored bf16 weight is the RNE rounding of the exported fp32 weight;
  * sampled matrices stepped alone give bit-identical O (grouping does not
    change results).
"""
import os

import numpy as np
import pytest
import torch

from gpu_helpers import check_against_oracle, oracle_step, to_np
from newton_schulz_06_gb300 import Muon, mode_code
from newton_schulz_06_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
LR, BETA = float(np.float32(0.02)), float(np.float32(0.95))


def band_ok(O, mode="full", nb=1):
    """||O||_F^2 / m of each unit within p^5's band (computed on the GPU)."""
    r, c = O.shape
    blocks = [O] if mode == "full" else list(O.split(c // nb, dim=1))
    out = []
    for B in blocks:
        m = min(B.shape)
        q = (B.float().pow(2).sum() / m).item()
        out.append(0.46 <= q <= 1.45)
    return all(out)


def run_workload(wl, sample, *, steps=1, exports_for=None, max_ws=None):
    """Runs `steps` grouped steps (fresh gradients from step 2 on).  Returns
    the tensors, host copies and device clones of the sampled matrices taken
    just before the last step, the exports and the handle."""
    Ws, Gs, Ms = I.make_state(wl, DEV)
    trips = list(zip(Ws, Gs, Ms))
    opt = Muon(trips)
    md = mode_code(wl.mode)
    opt.ensure_workspace(md, wl.nb, max_ws)
    idx = range(len(trips)) if exports_for is None else exports_for
    wexp = [None] * len(trips)
    oexp = [None] * len(trips)
    for i in idx:
        wexp[i] = torch.empty(Ws[i].shape, device=DEV, dtype=torch.float32)
        oexp[i] = torch.empty(Ws[i].shape, device=DEV, dtype=torch.bfloat16)
    opt.set_exports(wexp, oexp)
    host = before = None
    for k in range(steps):
        if k > 0:
            for i, G in enumerate(Gs):
                I.fill_grad(G, wl, i, k)
        if k == steps - 1:
            torch.cuda.synchronize()
            host = {i: (to_np(Ws[i]), to_np(Gs[i]), to_np(Ms[i])) for i in sample}
            before = [tuple(t.clone() for t in trips[i]) for i in sample]
        opt.step(lr=LR, beta=BETA, nesterov=True, ns_steps=5, mode=md, nb=wl.nb)
    opt.sync()
    torch.cuda.synchronize()
    return trips, host, before, wexp, oexp, opt


def check_sample(wl, trips, host, wexp, oexp, sample):
    errs = {}
    for i in sample:
        ref = oracle_step(host[i], lr=LR, beta=BETA, mode=wl.mode, nb=wl.nb)
        errs[i] = check_against_oracle(trips[i], host[i], wexp[i], oexp[i], ref,
                                       mode=wl.mode, nb=wl.nb)
    return errs


def check_standalone(wl, trips_before, oexp, sample):
    """Sampled matrices stepped alone give the same bits as in the group."""
    for i, (W, G, M) in zip(sample, trips_before):
        _, _, o1, opt = _alone(W, G, M, wl)
        assert torch.equal(o1, oexp[i]), i
        opt.close()


def _alone(W, G, M, wl):
    opt = Muon([(W, G, M)])
    md = mode_code(wl.mode)
    opt.ensure_workspace(md, wl.nb)
    o = torch.empty(W.shape, device=DEV, dtype=torch.bfloat16)
    opt.set_exports(None, [o])
    opt.step(lr=LR, beta=BETA, nesterov=True, ns_steps=5, mode=md, nb=wl.nb)
    opt.sync()
    return W, M, o, opt


def test_square_4096_three_steps_teacher_forced():
    wl = I.workload("square_4096_bf16")
    trips, host, before, wexp, oexp, _ = run_workload(wl, [0], steps=3)
    errs = check_sample(wl, trips, host, wexp, oexp, [0])
    print("4096^2 step 3", errs)
    check_standalone(wl, before, oexp, [0])


def test_square_4096_distributed4_teacher_forced():
    """Distributed mode over 4 slices at the benchmark's size, two steps."""
    wl = I.workload("square_4096_bf16_distributed4")
    trips, host, before, wexp, oexp, _ = run_workload(wl, [0], steps=2)
    errs = check_sample(wl, trips, host, wexp, oexp, [0])
    print("4096^2 distributed4 step 2", errs)
    check_standalone(wl, before, oexp, [0])


def test_qwen3_block_grouped():
    wl = I.workload("qwen3_30b_a3b_block")
    gen = np.random.default_rng(2026)
    experts = sorted(4 + gen.choice(384, size=4, replace=False))
    sample = [0, 1, 3] + [int(e) for e in experts]
    trips, host, before, wexp, oexp, _ = run_workload(wl, sample)
    errs = check_sample(wl, trips, host, wexp, oexp, sample)
    print("qwen3 block", {wl.shapes[i]: round(e["O"], 4) for i, e in errs.items()})
    for i, (W, G, M) in enumerate(trips):
        assert band_ok(oexp[i]), (i, wl.shapes[i])
        assert torch.equal(W, wexp[i].to(torch.bfloat16)), i
    check_standalone(wl, before, oexp, sample)


@pytest.mark.parametrize("name", ["kimi_k2_layer_full", "kimi_k2_layer_blockwise4"])
def test_kimi_k2_layer(name):
    wl = I.workload(name)
    # q_a, q_b (tall), kv_a (m = 576), kv_b (tall), one expert gate and down
    sample = [0, 1, 2, 3, 5, 7]
    trips, host, before, wexp, oexp, _ = run_workload(wl, sample)
    errs = check_sample(wl, trips, host, wexp, oexp, sample)
    print(name, {wl.shapes[i]: round(e["O"], 4) for i, e in errs.items()})
    for i, (W, G, M) in enumerate(trips):
        assert band_ok(oexp[i], wl.mode, wl.nb), (i, wl.shapes[i])
        assert torch.equal(W, wexp[i].to(torch.bfloat16)), i
    check_standalone(wl, before[:3], oexp, sample[:3])


def test_qwen3_48_layers_ten_steps():
    """18,624 matrices (240 GB of W, G, M) in groups; momentum carried over
    10 steps with fresh gradients; the oracle checks step 10 of a sample
    (teacher-forced)."""
    wl = I.workload("qwen3_30b_a3b_48_layers")
    need = wl.n_elements * (2 + 2 + 4) + (24 << 30)
    import gc
    gc.collect()
    torch.cuda.empty_cache()      # earlier tests' cached blocks count as used
    free, _ = torch.cuda.mem_get_info()
    if free < need:
        pytest.skip(f"needs {need / 2**30:.0f} GiB free, {free / 2**30:.0f} GiB free")
    gen = np.random.default_rng(48)
    sample = [0, 1, 3, 4, 6] + [int(x) for x in gen.choice(wl.n_matrices, 4,
                                                            replace=False)]
    trips, host, before, wexp, oexp, opt = run_workload(
        wl, sample, steps=10, exports_for=sample, max_ws=16 << 30)
    assert opt.plan_info()["groups"] > 1
    errs = check_sample(wl, trips, host, wexp, oexp, sample)
    print("48 layers step 10", {i: round(e["O"], 4) for i, e in errs.items()})
    opt.close()
    del trips, wexp, oexp, opt
    torch.cuda.empty_cache()


# bf16 storage of a weight: relF(RNE(w), w) <= 2^-8 for any w (half an ulp,
# relative); with relF(w32, W_ref) <= 1e-3 the stored weight is within
# 2^-8 * (1 + 1e-3) + 1e-3 of the float64 weight (triangle inequality)
BF16_STORED_W_TOL = 2.0 ** -8 * (1 + 1e-3) + 1e-3


@pytest.mark.parametrize("name", ["square_4096_bf16", "tall_6144x1536_bf16"])
def test_export_free_chain_at_full_size(name):
    """The configuration the benchmark times: no validation exports, so the
    chained launch also runs the last X update with the weight update folded
    in (three launches per step).  Over three steps with fresh gradients its
    W and M are bit-identical to the same steps with exports registered
    (where the chain stops before the last X update and the export-writing
    update launch stores W, the form gated against the oracle), and the
    stored bf16 W of step 3 is within the bf16-storage bound of the float64
    oracle (teacher-forced from the state before step 3)."""
    if name == "square_4096_bf16":
        wl = I.workload(name)
        Wa, Ga, Ma = (t[0] for t in I.make_state(wl, DEV))

        def grad(G, k):
            I.fill_grad(G, wl, 0, k)
    else:
        Wa, Ga, Ma = I.random_case(6144, 1536, 1111, device=DEV)

        def grad(G, k):
            g = torch.Generator(device=DEV)
            g.manual_seed(I.seed_for("tall", k))
            G.copy_(torch.randn(G.shape, generator=g, device=DEV))
    Wb, Gb, Mb = Wa.clone(), Ga.clone(), Ma.clone()
    opt_a, opt_b = Muon([(Wa, Ga, Ma)]), Muon([(Wb, Gb, Mb)])
    for o in (opt_a, opt_b):
        o.ensure_workspace(mode_code("full"), 1)
        assert o.plan_info()["chained_groups"] == 1
    wexp = torch.empty(Wa.shape, device=DEV, dtype=torch.float32)
    oexp = torch.empty(Wa.shape, device=DEV, dtype=torch.bfloat16)
    opt_a.set_exports([wexp], [oexp])
    host = None
    for k in range(3):
        if k > 0:
            grad(Ga, k)
            Gb.copy_(Ga)
        if k == 2:
            torch.cuda.synchronize()
            host = (to_np(Wb), to_np(Gb), to_np(Mb))
        opt_a.step(lr=LR, beta=BETA, nesterov=True, ns_steps=5)
        opt_b.step(lr=LR, beta=BETA, nesterov=True, ns_steps=5)
        # exports: momentum, norm, chain, last X update; none: the chain holds it
        assert opt_a.last_launch_count() == 4 and opt_b.last_launch_count() == 3
        opt_a.sync()
        opt_b.sync()
        torch.cuda.synchronize()
        assert torch.equal(Wa, Wb), (name, k)
        assert torch.equal(Ma, Mb), (name, k)
    ref = oracle_step(host, lr=LR, beta=BETA)
    errs = check_against_oracle((Wa, Ga, Ma), host, wexp, oexp, ref)
    w_rel = float(np.linalg.norm(to_np(Wb) - ref["W"]) / np.linalg.norm(ref["W"]))
    print(name, "step 3", errs, "stored bf16 W vs float64:", w_rel)
    assert w_rel <= BF16_STORED_W_TOL, w_rel
    opt_a.close()
    opt_b.close()
