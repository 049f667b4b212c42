"""Distributed mode across ranks: the phases and the group's sums, as gloo
ranks on the CPU.

Each rank holds its slice of one matrix; DistributedMuon sums the slices'
sums of squares and, per iteration, the partial products' upper tiles band by
band.  The phases run on a GPU in libmuon; here a float64 stand-in engine runs
them with the oracle's arithmetic, so the test checks the orchestration: the
slicing, which sums happen when, that the banded exchange of upper tiles
rebuilds the whole product, the first-iteration norm and the last-iteration
update.  The result must match the oracle's distributed mode ("Advancing
Emerging Optimizers for Accelerated LLM Training", section "Distributed
mode") and its full mode, which the mathematics makes equal."""
import math
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from newton_schulz_06_gb300.distributed import band_ranges, slice_range

COEFFS = (3.4445, -4.7750, 2.0315)


class OracleSlice:
    """The muon_dist_* phases in float64 numpy on one rank's slice."""

    def __init__(self, W, G, M, *, transposed, shape_scale, eps=1e-7):
        self.W, self.G, self.M = (np.array(x, dtype=np.float64) for x in (W, G, M))
        self.transposed, self.scale, self.eps = transposed, shape_scale, eps

    def new_matrix(self, m):
        return torch.zeros(m, m, dtype=torch.float64)

    def momentum(self, beta, nesterov):
        self.M, U = oracle.momentum_update(self.M, self.G, beta, nesterov)
        self.X = U.T if self.transposed else U
        return torch.tensor([float(np.sum(self.X * self.X))], dtype=torch.float64)

    def gram(self, A, band):
        P = self.X @ self.X.T                    # this rank's partial product
        m = P.shape[0]
        for ti in range(*band):                  # upper tiles of these row blocks
            r0, r1 = ti * 256, min(ti * 256 + 256, m)
            A[r0:r1, r0:] = torch.from_numpy(P[r0:r1, r0:].copy())

    def update(self, A, *, first, last, sumsq_total, lr, coeffs):
        a, b, c = coeffs
        m = A.shape[0]
        # the stored upper tiles, whole on the diagonal tiles, mirrored below
        T = (m + 255) // 256
        S = np.zeros((m, m))
        An = A.numpy()
        for ti in range(T):
            for tj in range(ti, T):
                r, cc = slice(ti * 256, min(ti * 256 + 256, m)), slice(tj * 256, min(tj * 256 + 256, m))
                S[r, cc] = An[r, cc]
                if ti != tj:
                    S[cc, r] = An[r, cc].T
        if first:
            inv = 1.0 / (math.sqrt(float(sumsq_total[0])) + self.eps)
            S = S * inv * inv
            self.X = self.X * inv
        B = b * S + c * (S @ S)
        self.X = a * self.X + B @ self.X
        if last:
            O = self.X.T if self.transposed else self.X
            self.W = self.W - lr * self.scale * O

    def sync(self):
        pass


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case(shape, seed):
    g = np.random.default_rng(seed)
    W = 0.02 * g.standard_normal(shape)
    G = g.standard_normal(shape)
    M = g.standard_normal(shape)
    return W, G, M


def _worker(rank, world, port, q, shape, bands, seed):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from newton_schulz_06_gb300.distributed import DistributedMuon
    dist.init_process_group("gloo", rank=rank, world_size=world)
    W, G, M = _case(shape, seed)
    rows, cols = shape
    tall = rows > cols
    lo, hi = slice_range(rows if tall else cols, world, rank)
    sl = (slice(lo, hi), slice(None)) if tall else (slice(None), slice(lo, hi))
    scale = math.sqrt(max(1.0, rows / cols))
    eng = OracleSlice(W[sl], G[sl], M[sl], transposed=tall, shape_scale=scale)
    opt = DistributedMuon(W[sl], G[sl], M[sl], full_shape=shape, engine=eng)
    opt.step(lr=0.02, beta=0.95, nesterov=True, ns_steps=5, coeffs=COEFFS, bands=bands)
    q.put((rank, lo, hi, eng.W, eng.M))
    dist.destroy_process_group()


@pytest.mark.parametrize("shape,world,bands", [((96, 2048), 2, 1), ((640, 1536), 4, 2),
                                               ((1536, 520), 2, 3), ((2048, 300), 4, 1)])
def test_distributed_ranks_match_oracle(shape, world, bands):
    seed = 4100 + world + bands
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, shape, bands, seed))
             for r in range(world)]
    for p in procs:
        p.start()
    got = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    W, G, M = _case(shape, seed)
    rows, cols = shape
    tall = rows > cols
    Wn = np.empty(shape)
    Mn = np.empty(shape)
    for rank, lo, hi, w, m in got:
        if tall:
            Wn[lo:hi, :], Mn[lo:hi, :] = w, m
        else:
            Wn[:, lo:hi], Mn[:, lo:hi] = w, m
    a, b, c = COEFFS
    kw = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5, a=a, b=b, c=c)
    ref_d = oracle.muon_step_matrix(W, G, M, shards=world, **kw)
    ref_f = oracle.muon_step_matrix(W, G, M, **kw)
    assert np.allclose(Mn, ref_d["M"], rtol=0, atol=0)
    dW = Wn - W
    for ref in (ref_d, ref_f):
        err = np.linalg.norm(dW - (ref["W"] - W)) / np.linalg.norm(ref["W"] - W)
        assert err < 1e-12, err


def test_band_ranges_cover_the_row_blocks():
    for m in (1, 256, 257, 768, 4096, 5000):
        T = (m + 255) // 256
        for bands in (1, 2, 3, 8, 100):
            r = band_ranges(m, bands)
            assert r[0][0] == 0 and r[-1][1] == T
            assert all(x[1] == y[0] for x, y in zip(r, r[1:]))
            assert all(x[0] < x[1] for x in r)


def test_slice_range_rejects_uneven_slices():
    assert slice_range(2048, 4, 1) == (512, 1024)
    with pytest.raises(ValueError):
        slice_range(1000, 3, 0)
