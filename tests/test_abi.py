"""The C ABI without a GPU: the library loads, exports every declared entry
point, validates arguments, and its host planner counts tiles and FLOPs the
way an independent enumeration does."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from newton_schulz_06_gb300 import build as b
    b.build()
    from newton_schulz_06_gb300 import _lib
    return _lib


def declared_entry_points():
    text = open(os.path.join(ROOT, "include", "muon.h")).read()
    return sorted(set(re.findall(r"MUON_API\s+[\w\s\*]*?\b(muon_\w+)\s*\(", text)))


def test_header_declares_the_binding_list(L):
    assert declared_entry_points() == sorted(L.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    lib = L.lib()
    for name in declared_entry_points():
        assert hasattr(lib, name), name


def test_elf_dynamic_symbols(L):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", L.LIB_PATH],
                         capture_output=True, text=True).stdout
    syms = set(re.findall(r"\bT (muon_\w+)", out))
    assert set(declared_entry_points()) <= syms
    # nothing but the C ABI is exported from the library's own code
    assert all(s.startswith("muon_") for s in syms)


def _planner(shapes, **kw):
    from newton_schulz_06_gb300 import HostPlanner
    return HostPlanner(shapes, **kw)


def _syrk_tiles(m, pair):
    if pair:
        T2 = -(-m // 256)
        return sum(1 for ti in range(T2) for tj in range(T2) if tj >= ti)
    T = -(-m // 128)
    return sum(1 for ti in range(T) for tj in range(-(-T // 2))
               if any(2 * tj + h < T and 2 * tj + h >= ti for h in (0, 1)))


@pytest.mark.parametrize("pair", [True, False])
@pytest.mark.parametrize("shape", [(4096, 4096), (768, 2048), (2048, 768),
                                   (576, 7168), (100, 37), (8, 16)])
def test_plan_tile_counts(L, shape, pair, monkeypatch):
    monkeypatch.setenv("MUON_CTA_GROUP", "2" if pair else "1")
    p = _planner([shape])
    info = p.plan_info()
    m, n = min(shape), max(shape)
    rows = 256 if pair else 128
    assert info["units"] == 1 and info["groups"] == 1
    assert info["syrk_tiles"] == _syrk_tiles(m, pair)
    assert info["gemm_tiles"] == (-(-m // rows)) * (-(-n // 256))
    assert info["ew_tiles"] == (-(-m // 64)) * (-(-n // 64))
    # executed FLOPs: every tile's MACs over the zero-padded K
    kn, km = -(-n // 64) * 64, -(-m // 64) * 64
    if pair:
        ex = 2 * 256 * 256 * (info["syrk_tiles"] * (kn + km) +
                              info["gemm_tiles"] * km)
        assert info["executed_flops"] == ex
    assert info["executed_flops"] >= info["useful_flops"]


def test_useful_flops_match_formula(L):
    from newton_schulz_06_gb300 import flops
    from newton_schulz_06_gb300.inputs import qwen3_30b_a3b_block_shapes
    shapes = qwen3_30b_a3b_block_shapes()
    info = _planner(shapes).plan_info()
    assert info["units"] == 388
    assert 5 * info["useful_flops"] == flops.useful_flops(shapes)
    # executed FLOPs cover the useful ones and stay within the tile waste
    assert info["executed_flops"] >= info["useful_flops"]
    assert info["executed_flops"] < 1.2 * flops.gemm_equiv_flops(shapes) / 5


def test_flop_counts_closed_form():
    from newton_schulz_06_gb300 import flops
    # 4096^2: GEMM-equivalent 6 m^3 per iteration; 2.06 TFLOP for 5 steps
    assert flops.gemm_equiv_flops([(4096, 4096)]) == 5 * 6 * 4096 ** 3
    u = flops.useful_flops([(4096, 4096)])
    assert u == 5 * (2 * 4096 * 4097 * 4096 + 2 * 4096 ** 3)
    assert abs(u / 1e12 - 1.375) < 0.001
    # blockwise: nb blocks of rows x cols/nb
    assert flops.useful_flops([(16384, 512)], mode="blockwise", nb=4) == \
        4 * flops.useful_flops([(16384, 128)])


def test_blockwise_units_and_validation(L):
    from newton_schulz_06_gb300.inputs import kimi_k2_layer_shapes
    shapes = kimi_k2_layer_shapes()
    p = _planner(shapes)
    assert p.plan_info(L.MUON_BLOCKWISE, 4)["units"] == 4 * len(shapes)
    assert p.plan_info(L.MUON_FULL, 4)["units"] == len(shapes)
    with pytest.raises(L.MuonError) as e:
        p.plan_info(L.MUON_BLOCKWISE, 3)
    assert e.value.code == L.MUON_ERR_UNSUPPORTED


def test_workspace_sizes_monotone(L):
    from newton_schulz_06_gb300.inputs import qwen3_30b_a3b_block_shapes
    p = _planner(qwen3_30b_a3b_block_shapes())
    mn, full = p.workspace_size()
    # full holds every unit's X ping-pong: at least 2 * 2 bytes * elements
    elems = sum(r * c for r, c in qwen3_30b_a3b_block_shapes())
    assert full >= 4 * elems and mn < full
    # the largest unit (2048 x 4096) needs its X pair and A, B
    assert mn >= 2 * 2 * 2048 * 4096 + 2 * 2 * 2048 * 2048


def test_register_rejects_bad_params(L):
    import ctypes
    lib = L.lib()
    h = ctypes.c_void_p()
    assert lib.muon_create(ctypes.byref(h), L.MUON_HOST_ONLY, None) == 0
    P = L.MuonParam

    def reg(**kw):
        p = P()
        p.w = p.g = p.m = 0x1000
        p.rows, p.cols = 4, 8
        p.ld_w = p.ld_g = p.ld_m = 8
        p.w_dtype = p.g_dtype = L.MUON_BF16
        for k, v in kw.items():
            setattr(p, k, v)
        arr = (P * 1)(p)
        return lib.muon_register_params(h, 1, arr)

    assert reg() == 0
    assert reg(w=None) == L.MUON_ERR_INVALID_ARG
    assert reg(rows=0) == L.MUON_ERR_INVALID_ARG
    assert reg(ld_g=4) == L.MUON_ERR_INVALID_ARG
    assert reg(w_dtype=7) == L.MUON_ERR_UNSUPPORTED
    assert reg(rows=40000, cols=40000, ld_w=40000, ld_g=40000,
               ld_m=40000) == L.MUON_ERR_UNSUPPORTED
    assert lib.muon_register_params(h, 0, None) == L.MUON_ERR_INVALID_ARG
    assert b"parameters" in lib.muon_last_error(h)
    # a host-only handle plans but never launches
    assert reg() == 0
    assert lib.muon_step(h, 0.02, 0.95, 1, 5, 3.4445, -4.775, 2.0315, 0,
                         1) == L.MUON_ERR_STATE
    # the chained launch's validation switches are an explicit call (no
    # environment variable can turn them on); out-of-range values rejected
    assert lib.muon_debug_set_chain_test(h, 0) == 0
    assert lib.muon_debug_set_chain_test(h, 3) == 0
    assert lib.muon_debug_set_chain_test(h, -1) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_debug_set_chain_test(h, (1 << 20) + 1) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_destroy(h) == 0


def test_distributed_mode_plan_and_validation(L):
    """Distributed mode keeps one unit per matrix, full mode's tiles and
    full mode's workspace (the slices' sum stays in tensor memory); slices
    must be equal multiples of 64 of every long side."""
    shapes = [(4096, 4096), (768, 2048), (2048, 768)]
    p = _planner(shapes)
    full = p.plan_info(L.MUON_FULL, 1)
    dist = p.plan_info(L.MUON_DISTRIBUTED, 4)
    for k in ("units", "syrk_tiles", "gemm_tiles", "useful_flops", "executed_flops"):
        assert dist[k] == full[k], k
    assert p.workspace_size(L.MUON_DISTRIBUTED, 4) == p.workspace_size(L.MUON_FULL, 1)
    assert p.plan_info(L.MUON_DISTRIBUTED, 1)["syrk_tiles"] == full["syrk_tiles"]
    for bad in (3, 64):      # 2048 / 3 is not whole; 2048 / 64 = 32 < 64
        with pytest.raises(L.MuonError) as e:
            p.plan_info(L.MUON_DISTRIBUTED, bad)
        assert e.value.code == L.MUON_ERR_UNSUPPORTED
    with pytest.raises(L.MuonError) as e:
        p.plan_info(L.MUON_DISTRIBUTED, 0)
    assert e.value.code == L.MUON_ERR_INVALID_ARG


def test_distributed_ranks_slice_plan_and_validation(L):
    """A rank's slice (muon_dist_configure) takes the whole matrix's
    orientation: a 4096 x 2048 column slice of a 4096 x 8192 weight keeps
    m = 4096 (its own shape would be transposed to m = 2048), so its plan
    holds 4096^2 products.  Configuration and phases are checked before any
    CUDA call; a host-only handle runs no phase, and a slice never runs
    muon_step."""
    lib = L.lib()
    own = _planner([(4096, 2048)])
    sl = _planner([(4096, 2048)])
    assert lib.muon_dist_configure(sl._h, 0, 2.0) == 0
    t_own = own.plan_info(L.MUON_FULL, 1)["syrk_tiles"]
    t_sl = sl.plan_info(L.MUON_FULL, 1)["syrk_tiles"]
    assert t_own == 8 * 9 // 2 and t_sl == 16 * 17 // 2, (t_own, t_sl)
    assert sl.workspace_size()[1] > own.workspace_size()[1]
    # the same slice as a block of a tall weight's rows: transposed, m = 2048
    assert lib.muon_dist_configure(sl._h, 1, 2.0) == 0
    assert sl.plan_info(L.MUON_FULL, 1)["syrk_tiles"] == t_own
    assert lib.muon_dist_configure(sl._h, 0, 0.5) == L.MUON_ERR_INVALID_ARG
    assert lib.muon_dist_configure(sl._h, 0, float("nan")) == L.MUON_ERR_INVALID_ARG
    with pytest.raises(L.MuonError) as e:                  # slices run in full mode
        sl.plan_info(L.MUON_BLOCKWISE, 2)
    assert e.value.code == L.MUON_ERR_UNSUPPORTED
    buf = ctypes.c_void_p(0x1000)
    assert lib.muon_dist_momentum(sl._h, 0.95, 1, buf) == L.MUON_ERR_STATE
    assert lib.muon_dist_gram(sl._h, buf, 4096, 0, -1) == L.MUON_ERR_STATE
    assert lib.muon_dist_update(sl._h, buf, 4096, 1, 0, buf, 0.02, 1.0, 1.0, 1.0) == \
        L.MUON_ERR_STATE
    assert lib.muon_step(sl._h, 0.02, 0.95, 1, 5, 3.4, -4.7, 2.0, L.MUON_FULL, 1) == \
        L.MUON_ERR_STATE
    two = _planner([(256, 512), (256, 512)])
    assert lib.muon_dist_configure(two._h, 0, 1.0) == 0
    with pytest.raises(L.MuonError) as e:                  # one slice per handle
        two.plan_info(L.MUON_FULL, 1)
    assert e.value.code == L.MUON_ERR_UNSUPPORTED
    assert lib.muon_dist_configure(None, 0, 1.0) == L.MUON_ERR_INVALID_ARG


def test_chained_launch_only_for_few_large_matrices(L):
    """One chained launch per step is planned where a group has at least one
    and at most 8 X-update tiles per CTA pair (76 pairs), in full and
    blockwise mode; distributed mode, small steps and large groups keep one
    launch per product."""
    from newton_schulz_06_gb300.inputs import qwen3_30b_a3b_block_shapes
    sq = _planner([(4096, 4096)])
    assert sq.plan_info(L.MUON_FULL, 1)["chained_groups"] == 1
    assert sq.plan_info(L.MUON_BLOCKWISE, 4)["chained_groups"] == 1
    assert sq.plan_info(L.MUON_DISTRIBUTED, 4)["chained_groups"] == 0
    # 76 pairs x 8 = 608 X-update tiles: 24 x 24 tiles of 256 chain, 25 x 25 not
    assert _planner([(6144, 6144)]).plan_info()["chained_groups"] == 1
    assert _planner([(6400, 6400)]).plan_info()["chained_groups"] == 0
    assert _planner(qwen3_30b_a3b_block_shapes()).plan_info()["chained_groups"] == 0
    # below one wave: 2048^2 has 8 x 8 X-update tiles, 2048 x 8192 has 8 x 32
    assert _planner([(2048, 2048)]).plan_info()["chained_groups"] == 0
    assert _planner([(2048, 8192)]).plan_info()["chained_groups"] == 1
    assert _planner([(256, 512)]).plan_info()["chained_groups"] == 0


@pytest.mark.parametrize("shapes,mode,nb", [
    ([(4096, 4096)], "full", 1),
    ([(6144, 1536), (300, 300), (96, 1000)], "full", 1),
    ([(2048, 4096)], "blockwise", 2),
    ([(512, 768), (768, 2048), (2048, 640), (256, 4096), (1000, 1000)], "full", 1),
    ([(256, 512)], "full", 1),
    ([(7168, 2048)] * 6 + [(2048, 7168)] * 6 + [(1536, 7168), (7168, 8192)], "full", 1),
])
def test_chain_schedule_stage_order_and_coverage(L, shapes, mode, nb):
    """The chained launch's per-pair lists (built on the host, whatever the
    size bounds) hold every tile once, in stage order per pair, with
    consistent offsets and last-iteration ends: the properties its waits need
    to end (each wait only on earlier stages)."""
    from newton_schulz_06_gb300 import mode_code
    _planner(shapes).check_chain_schedule(mode_code(mode), nb)
