"""Distributed mode across ranks on the GPU: libmuon's muon_dist_* phases.

With one rank the phases are the whole step, and the bits must be those of
muon_step in full mode: the first product's fp32 partial, rounded to bf16
after scaling, is what the full step's epilogue stores.  With P slices of one
matrix on one GPU ("virtual ranks": one handle per slice, the group's sums
done on the host in slice order, no kernel waiting on another handle's) the
bits must be those of the one-GPU distributed mode with P slices, which sums
the same fp32 partials in the same order in tensor memory and scales after
the sum.  Both are also gated against the float64 oracle ("Advancing
Emerging Optimizers for Accelerated LLM Training", section "Distributed
mode")."""
import math

import numpy as np
import pytest
import torch

from gpu_helpers import oracle_step, relF, to_np
from newton_schulz_06_gb300 import Muon, mode_code
from newton_schulz_06_gb300.distributed import DistributedMuon, SliceEngine, band_ranges, \
    slice_range
from newton_schulz_06_gb300.inputs import random_case

pytestmark = pytest.mark.gpu

DEV = "cuda:0"
COEFFS = (3.4445, -4.7750, 2.0315)
KW = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5, coeffs=COEFFS)


def case(rows, cols, seed, **kw):
    return list(random_case(rows, cols, seed, device=DEV, **kw))


@pytest.mark.parametrize("shape,bands,w_dtype", [((768, 2048), 1, torch.bfloat16),
                                                 ((2048, 768), 2, torch.bfloat16),
                                                 ((300, 300), 1, torch.bfloat16),
                                                 ((1024, 4096), 3, torch.bfloat16),
                                                 ((640, 1536), 2, torch.float32)])
def test_one_rank_is_the_full_step_bitexact(shape, bands, w_dtype):
    """Two steps (momentum carried) through the phases on one rank against
    muon_step on copies: identical W and M."""
    W, G, M = case(*shape, 5100 + shape[0], w_dtype=w_dtype)
    W2, G2, M2 = W.clone(), G.clone(), M.clone()
    opt = DistributedMuon(W, G, M, full_shape=shape)
    ref = Muon([(W2, G2, M2)])
    for _ in range(2):
        opt.step(bands=bands, **KW)
        ref.step(**KW)
    opt.sync()
    ref.sync()
    torch.cuda.synchronize()
    assert torch.equal(W, W2), shape
    assert torch.equal(M, M2), shape
    opt.engine.close()
    ref.close()


def _virtual_ranks(W, G, M, world, bands, steps=1):
    """P slice handles on one GPU; the group's sums on the host, in order."""
    rows, cols = W.shape
    tall = rows > cols
    scale = math.sqrt(max(1.0, rows / cols))
    m = min(rows, cols)
    engines, views = [], []
    for r in range(world):
        lo, hi = slice_range(rows if tall else cols, world, r)
        # each rank's slice in its own memory, as on its own GPU
        sl = (slice(lo, hi), slice(None)) if tall else (slice(None), slice(lo, hi))
        tw, tg, tm = W[sl].contiguous(), G[sl].contiguous(), M[sl].contiguous()
        engines.append(SliceEngine(tw, tg, tm, transposed=tall, shape_scale=scale))
        views.append((sl, tw, tg, tm))
    As = [e.new_matrix(m) for e in engines]
    total = torch.zeros(m, m, dtype=torch.float32, device=DEV)
    for _ in range(steps):
        ss = [e.momentum(0.95, True) for e in engines]
        sumsq = ss[0].clone()
        for x in ss[1:]:
            sumsq += x
        for s in range(5):
            for e, A in zip(engines, As):
                for band in band_ranges(m, bands):
                    e.gram(A, band)
            total.copy_(As[0])
            for A in As[1:]:
                total += A
            for e in engines:
                e.update(total, first=s == 0, last=s == 4, sumsq_total=sumsq, lr=0.02,
                         coeffs=COEFFS)
    for e in engines:
        e.sync()
    torch.cuda.synchronize()
    Wn, Mn = W.clone(), M.clone()
    for sl, tw, tg, tm in views:
        Wn[sl] = tw
        Mn[sl] = tm
    for e in engines:
        e.close()
    return Wn, Mn


@pytest.mark.parametrize("shape,world,bands", [((768, 2048), 2, 1), ((2048, 768), 4, 2),
                                               ((512, 4096), 4, 1), ((1536, 640), 2, 3)])
def test_virtual_ranks_are_the_one_gpu_distributed_mode_bitexact(shape, world, bands):
    """P slices, each on its own handle, summed on the host in slice order:
    the bits of muon_step in distributed mode with P slices, and within the
    oracle's tolerance of its distributed mode."""
    # fp32 weights, so that W's change carries no storage rounding
    W, G, M = case(*shape, 5200 + world, w_dtype=torch.float32)
    host = (to_np(W), to_np(G), to_np(M))
    W2, G2, M2 = W.clone(), G.clone(), M.clone()
    Wn, Mn = _virtual_ranks(W, G, M, world, bands)
    ref = Muon([(W2, G2, M2)])
    ref.step(mode=mode_code("distributed"), nb=world, **KW)
    ref.sync()
    torch.cuda.synchronize()
    assert torch.equal(Wn, W2), shape
    assert torch.equal(Mn, M2), shape
    ref.close()
    o = oracle_step(host, lr=0.02, beta=0.95, mode="distributed", nb=world)
    dW = to_np(Wn).astype(np.float64) - host[0].astype(np.float64)
    want = o["W"] - host[0].astype(np.float64)
    # the update's direction within the NS-output tolerance (3e-2)
    assert relF(dW, want) <= 3e-2, relF(dW, want)


def test_a_slice_handle_refuses_muon_step():
    """A handle configured as a rank's slice steps only through the phases
    (its norm and products need the group's sums)."""
    W, G, M = case(256, 512, 5310)
    eng = SliceEngine(W, G, M, transposed=False, shape_scale=1.0)
    with pytest.raises(Exception):
        eng._opt.step(**KW)
    eng.close()


def test_phases_out_of_order_are_refused():
    W, G, M = case(256, 512, 5300)
    eng = SliceEngine(W, G, M, transposed=False, shape_scale=1.0)
    A = eng.new_matrix(256)
    with pytest.raises(Exception):
        eng.gram(A, (0, 1))                    # before the momentum phase
    eng.momentum(0.95, True)
    with pytest.raises(Exception):
        eng.update(A, first=True, last=False, sumsq_total=eng._sumsq, lr=0.02,
                   coeffs=COEFFS)              # before this iteration's gram
    with pytest.raises(Exception):
        eng.gram(A, (0, 2))                    # past the last row block
    eng.sync()
    eng.close()
