"""Distributed mode across ranks: one matrix's iterate split along its long
side over the ranks of a tensor-parallel group, one GPU each.

"Advancing Emerging Optimizers for Accelerated LLM Training", section
"Distributed mode": each rank forms the partial product of its slice of X,
the partials are summed across the group (the all-reduce after the first
matrix product), and every rank then computes B from the sum and updates its
own slice.  Section "SYRK and fused all-reduce": only the symmetric
product's upper tiles need to travel, and they can travel as they finish.
Here the partial product is produced band by band (256-row blocks of A);
each band's upper part is summed across the group as soon as it is queued,
while the next band is still being computed.

Slices: W (rows x cols) is tall when rows > cols, and its iterate is then
W^T, so a rank holds a block of W's rows; otherwise a block of W's columns.
The slices are equal and contiguous (``slice_range``), and every rank keeps
its own slice of the momentum.

Only marshalling and collectives live here: every step of the update runs in
libmuon's ``muon_dist_*`` phases through :class:`SliceEngine`.
"""
from __future__ import annotations

import ctypes
import math
from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import check, lib
from .muon import DEFAULT_COEFFS, Muon


def slice_range(n: int, world: int, rank: int) -> Tuple[int, int]:
    """The [lo, hi) range of the long side that `rank` of `world` holds."""
    if world < 1 or n % world != 0:
        raise ValueError(f"{world} ranks must divide the long side {n}")
    w = n // world
    return rank * w, (rank + 1) * w


def band_ranges(m: int, bands: int) -> List[Tuple[int, int]]:
    """`bands` nearly equal ranges of the 256-row blocks of an m x m A."""
    T = (m + 255) // 256
    bands = max(1, min(bands, T))
    edges = [round(i * T / bands) for i in range(bands + 1)]
    return [(edges[i], edges[i + 1]) for i in range(bands)]


class SliceEngine:
    """libmuon's phases on one rank's slice (CUDA tensors W, G, M of the
    slice, in the weight's orientation; row-major)."""

    def __init__(self, W: torch.Tensor, G: torch.Tensor, M: torch.Tensor, *,
                 transposed: bool, shape_scale: float, stream=None):
        self._opt = Muon([(W, G, M)], stream=stream)
        self._h = self._opt._h
        check(lib().muon_dist_configure(self._h, int(bool(transposed)),
                                        float(shape_scale)), self._h)
        self._opt.ensure_workspace(_lib.MUON_FULL, 1)
        self.device = W.device
        self.m = W.shape[1] if transposed else W.shape[0]
        self._sumsq = torch.zeros(1, dtype=torch.float64, device=W.device)

    def new_matrix(self, m: int) -> torch.Tensor:
        return torch.zeros(m, m, dtype=torch.float32, device=self.device)

    def momentum(self, beta: float, nesterov: bool) -> torch.Tensor:
        check(lib().muon_dist_momentum(self._h, float(beta), int(bool(nesterov)),
                                       ctypes.c_void_p(self._sumsq.data_ptr())), self._h)
        return self._sumsq

    def gram(self, A: torch.Tensor, band: Tuple[int, int]) -> None:
        check(lib().muon_dist_gram(self._h, ctypes.c_void_p(A.data_ptr()), A.stride(0),
                                   band[0], band[1]), self._h)

    def update(self, A: torch.Tensor, *, first: bool, last: bool,
               sumsq_total: torch.Tensor, lr: float, coeffs) -> None:
        a, b, c = coeffs
        check(lib().muon_dist_update(self._h, ctypes.c_void_p(A.data_ptr()), A.stride(0),
                                     int(first), int(last),
                                     ctypes.c_void_p(sumsq_total.data_ptr()), float(lr),
                                     a, b, c), self._h)

    def sync(self) -> None:
        self._opt.sync()

    def close(self) -> None:
        self._opt.close()


class DistributedMuon:
    """One rank's part of a distributed-mode Muon step on one matrix.

    ``W``, ``G``, ``M`` are this rank's slices; ``full_shape`` is the whole
    weight's (rows, cols).  ``group`` is the tensor-parallel process group
    (None: the default group if one is initialised, else a single rank).
    ``engine`` runs the phases; the default is libmuon's :class:`SliceEngine`
    on the current CUDA stream.
    """

    def __init__(self, W, G, M, *, full_shape: Sequence[int], group=None, engine=None):
        rows, cols = (int(x) for x in full_shape)
        self.transposed = rows > cols
        self.shape_scale = math.sqrt(max(1.0, rows / cols))
        self.m = min(rows, cols)
        import torch.distributed as dist
        self._dist = dist if dist.is_available() and dist.is_initialized() else None
        self.group = group
        self.world = self._dist.get_world_size(group) if self._dist else 1
        slice_shape = (rows // self.world, cols) if self.transposed else (rows, cols // self.world)
        if tuple(W.shape) != slice_shape:
            raise ValueError(f"slice {tuple(W.shape)}, expected {slice_shape} "
                             f"of {rows} x {cols} over {self.world} ranks")
        self.engine = engine if engine is not None else SliceEngine(
            W, G, M, transposed=self.transposed, shape_scale=self.shape_scale)
        self.A = self.engine.new_matrix(self.m)

    def _sum(self, t: torch.Tensor, async_op: bool = False):
        if self.world == 1:
            return None
        return self._dist.all_reduce(t, group=self.group, async_op=async_op)

    def step(self, lr: float = 0.02, beta: float = 0.95, nesterov: bool = True,
             ns_steps: int = 5, coeffs=DEFAULT_COEFFS, bands: int = 1) -> None:
        """The rank's step; returns once its work and the group's sums are
        queued (libmuon's stream; wait with sync())."""
        sumsq = self.engine.momentum(beta, nesterov)
        self._sum(sumsq)
        ranges = band_ranges(self.m, bands)
        for s in range(ns_steps):
            pending = []
            for b0, b1 in ranges:
                self.engine.gram(self.A, (b0, b1))
                if self.world > 1:
                    # this band's upper part: its rows, from its first column
                    r0, r1 = b0 * 256, min(b1 * 256, self.m)
                    view = self.A[r0:r1, r0:]
                    buf = view.contiguous()
                    pending.append((self._sum(buf, async_op=True), view, buf))
            for work, view, buf in pending:
                work.wait()
                if buf.data_ptr() != view.data_ptr():
                    view.copy_(buf)
            self.engine.update(self.A, first=s == 0, last=s == ns_steps - 1,
                               sumsq_total=sumsq, lr=lr, coeffs=coeffs)

    def sync(self) -> None:
        self.engine.sync()
