"""Parity at the edges of what libmuon accepts: degenerate shapes (a single
row, a single column, a 1 x 1 weight) and the largest sizes (the short side
at its 32768 limit, the long side at its 2^20 limit).

A 32768 x 32768 step is far beyond what the float64 oracle can run whole, so
that case uses a gradient and momentum that are zero outside 32 diagonal
1024 x 1024 blocks.  Then U is block diagonal, and so are A = X X^T,
B = b A + c A A and every iterate: the exact step orthogonalises each
diagonal block on its own, every block scaled by the norm of the whole U
("Advancing Emerging Optimizers for Accelerated LLM Training", section
"Distributed mode": the three products of each iteration, after the
Frobenius normalisation).  On the GPU every product still runs over the full
32768-wide operands, so a wrong tile offset, a 32-bit index or a stale
buffer shows as a nonzero off the diagonal blocks or as a wrong block.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (COEFFS, O_TOL, W_TOL, check_against_oracle, f32, gpu_step,
                         oracle_step, relF, to_np)
from newton_schulz_06_gb300 import Muon
from newton_schulz_06_gb300 import inputs as I

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.mark.parametrize("rows,cols", [(1, 1), (1, 64), (64, 1), (2, 3), (3, 2),
                                       (1, 4096), (4096, 1)])
def test_degenerate_shapes_match_oracle(rows, cols):
    """One row or one column: X X^T is 1 x 1 and the step normalises the
    vector and applies p^5 to its single singular value."""
    trip = list(I.random_case(rows, cols, 77, device=DEV))
    inp, wexp, oexp, opt = gpu_step([trip])
    ref = oracle_step(inp[0])
    errs = check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref, w_gate="scaled")
    print((rows, cols), errs)
    opt.close()


@pytest.mark.parametrize("rows,cols", [(64, 1 << 20), (1 << 20, 64)])
def test_longest_side_matches_oracle(rows, cols):
    """The long side at its limit (2^20): 16384 k-blocks in the first
    product's single tile.  The tall form's shape scale is 128, so its weight
    moves by about 13% in one step and the weight gate scales with that move
    (the O gate is the fixed 3e-2)."""
    trip = list(I.random_case(rows, cols, 78, device=DEV))
    inp, wexp, oexp, opt = gpu_step([trip])
    ref = oracle_step(inp[0])
    errs = check_against_oracle(trip, inp[0], wexp[0], oexp[0], ref,
                                w_gate="fixed" if rows < cols else "scaled")
    print((rows, cols), errs)
    opt.close()


def _off_block_nonzeros(T, bs, k):
    """Nonzeros of block row k of T outside its diagonal block."""
    R = T[k * bs:(k + 1) * bs]
    return int(R.count_nonzero()) - int(R[:, k * bs:(k + 1) * bs].count_nonzero())


def test_largest_short_side_block_diagonal():
    m, bs = 32768, 1024
    nblk = m // bs
    lr, beta = f32(0.02), f32(0.95)
    torch.cuda.empty_cache()      # earlier tests' cached blocks count as used
    free, _ = torch.cuda.mem_get_info()
    if free < (40 << 30):
        pytest.skip(f"needs 40 GiB free, {free / 2**30:.0f} GiB free")
    W = I.make_weight((m, m), torch.bfloat16, DEV, "limits", m)
    G = torch.zeros((m, m), dtype=torch.bfloat16, device=DEV)
    M = torch.zeros((m, m), dtype=torch.float32, device=DEV)
    for k in range(nblk):
        _, g, mom = I.random_case(bs, bs, 900 + k, device=DEV)
        s = slice(k * bs, (k + 1) * bs)
        G[s, s] = g
        M[s, s] = mom
    torch.cuda.synchronize()
    Gd = [to_np(G[k * bs:(k + 1) * bs, k * bs:(k + 1) * bs]) for k in range(nblk)]
    Md = [to_np(M[k * bs:(k + 1) * bs, k * bs:(k + 1) * bs]) for k in range(nblk)]
    sample = [0, 1, 17, nblk - 1]
    Wd = {k: to_np(W[k * bs:(k + 1) * bs, k * bs:(k + 1) * bs]) for k in sample}
    W0 = W.clone()

    opt = Muon([(W, G, M)])
    opt.ensure_workspace(0, 1)
    wexp = torch.empty((m, m), dtype=torch.float32, device=DEV)
    oexp = torch.empty((m, m), dtype=torch.bfloat16, device=DEV)
    opt.set_exports([wexp], [oexp])
    opt.step(lr=lr, beta=beta, nesterov=True, ns_steps=5, coeffs=COEFFS)
    opt.sync()
    torch.cuda.synchronize()

    # nothing outside the diagonal blocks: O and M stay zero, W unchanged
    for k in range(nblk):
        assert _off_block_nonzeros(oexp, bs, k) == 0, k
        assert _off_block_nonzeros(M, bs, k) == 0, k
        R = (W[k * bs:(k + 1) * bs] != W0[k * bs:(k + 1) * bs])
        moved = int(R.count_nonzero()) - int(R[:, k * bs:(k + 1) * bs].count_nonzero())
        assert moved == 0, k
    assert torch.equal(W, wexp.to(torch.bfloat16)), "stored W != RNE(fp32)"
    del W0, R

    # the oracle on the blocks: momentum of every block, one norm over all
    # of them (the norm of the block-diagonal U), then each sampled block's
    # own iteration and update
    a, b, c = COEFFS
    mom = [oracle.momentum_update(Md[k], Gd[k], beta, True) for k in range(nblk)]
    X0 = oracle.frobenius_normalise(np.concatenate([u for _, u in mom]), 1e-7)
    errs = {}
    for k in sample:
        s = slice(k * bs, (k + 1) * bs)
        O_ref = oracle.newton_schulz(X0[k * bs:(k + 1) * bs], 5, a, b, c)
        W_ref = Wd[k] - lr * oracle.shape_scale(m, m) * O_ref
        eo = relF(to_np(oexp[s, s]), O_ref)
        ew = relF(to_np(wexp[s, s]), W_ref)
        M_ref = mom[k][0]
        dm = np.abs(to_np(M[s, s]) - M_ref)
        assert np.all(dm <= 1.2e-7 * (np.abs(M_ref) + np.abs(Gd[k])) + 1e-30), k
        errs[k] = (round(eo, 5), round(ew, 7))
        assert eo <= O_TOL and ew <= W_TOL, (k, eo, ew)
    print("32768^2 block-diagonal", errs)
    opt.close()


def test_many_tiny_matrices_in_one_group():
    """5000 matrices of 1 to 96 rows and columns, every one its own unit in
    one grouped step (tables of thousands of units, tiles that are mostly
    edge): a sample against the oracle, and a sample stepped alone gives the
    same bits as inside the group."""
    gen = np.random.default_rng(5000)
    shapes = [tuple(int(x) for x in gen.integers(1, 97, size=2)) for _ in range(5000)]
    trips = [list(I.random_case(r, c, 3000 + i, device=DEV)) for i, (r, c) in enumerate(shapes)]
    sample = sorted(int(i) for i in gen.choice(len(shapes), 12, replace=False))
    clones = {i: [t.clone() for t in trips[i]] for i in sample}
    inp, wexp, oexp, opt = gpu_step(trips)
    assert opt.plan_info()["units"] == len(shapes)
    for i in sample:
        ref = oracle_step(inp[i])
        check_against_oracle(trips[i], inp[i], wexp[i], oexp[i], ref, w_gate="scaled")
        _, _, o1, opt1 = gpu_step([clones[i]])
        assert torch.equal(o1[0], oexp[i]), shapes[i]
        assert torch.equal(clones[i][0], trips[i][0]), shapes[i]
        opt1.close()
    opt.close()
