"""Layer-wise distributed Muon over data-parallel ranks.

"Advancing Emerging Optimizers for Accelerated LLM Training", section
"Layer-wise distributed optimizer": Muon needs a layer's whole gradient, so
instead of sharding every tensor element-wise, whole layers are assigned to
data-parallel ranks.  Each rank runs the complete step (momentum,
orthogonalisation, update) for the matrices it owns, keeps momentum only for
them, and the ranks then exchange the updated weights so that every rank
holds all of them (section "Load balancing": today layers are distributed
round-robin, and the optimizer cost differs between attention and MLP
matrices; the same page names gathering the parameters later, overlapped
with compute, as future work).

Here ownership is a longest-processing-time partition by the step's FLOPs
(costliest matrix first, to the least-loaded rank), the same cost model the
single-GPU planner uses for tiles.  The exchange is a variable-size
all-gather (the pages' all_gatherv of the updated parameters): each rank
packs its owned weights' bytes into one buffer of exactly that size, every
owner broadcasts its buffer to the group (one broadcast per rank that owns
anything, each of its own size, none padded), and every rank unpacks the
others' segments.  It can be left pending (``async_gather=True``) so the
caller overlaps it with other work and waits before the weights are read.

Only marshalling and collectives live here: every step of the update runs in
libmuon through :class:`~newton_schulz_06_gb300.muon.Muon`.
"""
from __future__ import annotations

import heapq
from typing import Callable, List, Optional, Sequence

import torch

from . import flops
from .muon import Muon, mode_code


def lpt_partition(costs: Sequence[int], world: int) -> List[int]:
    """Owner rank of each item: costliest first (ties: lower index) to the
    least-loaded rank (ties: lower rank).  Deterministic, so every rank
    computes the same partition independently."""
    if world < 1:
        raise ValueError("world must be >= 1")
    order = sorted(range(len(costs)), key=lambda i: (-costs[i], i))
    loads = [(0, r) for r in range(world)]
    heapq.heapify(loads)
    owner = [0] * len(costs)
    for i in order:
        load, r = heapq.heappop(loads)
        owner[i] = r
        heapq.heappush(loads, (load + int(costs[i]), r))
    return owner


def matrix_costs(shapes, mode: str = "full", nb: int = 1) -> List[int]:
    """The step's useful FLOPs of each matrix (all its units)."""
    return [flops.useful_flops([s], mode=mode, nb=nb) for s in shapes]


class _Pending:
    """A weight exchange in flight; wait() completes it and unpacks."""

    def __init__(self, works, finish: Callable[[], None]):
        self._works = list(works)
        self._finish = finish
        self._done = False

    def wait(self) -> None:
        if not self._done:
            for w in self._works:
                w.wait()
            self._works = []
            self._done = True
            self._finish()


class LayerwiseMuon:
    """One rank's part of a layer-wise distributed Muon step.

    ``weights`` and ``grads`` list every matrix of the model on this rank
    (the gradients already averaged over the data-parallel group).  The rank
    keeps fp32 momentum only for the matrices it owns.  ``engine`` builds the
    local stepper from the owned (W, G, M) triples; the default is libmuon's
    :class:`Muon`.  ``group`` is the data-parallel process group (None: the
    default group if one is initialised, else a single rank).
    """

    def __init__(self, weights: Sequence[torch.Tensor], grads: Sequence[torch.Tensor],
                 group=None, *, mode: str = "full", nb: int = 1,
                 engine: Optional[Callable] = None):
        if len(weights) != len(grads) or not weights:
            raise ValueError("need matching, non-empty weight and gradient lists")
        if not all(w.is_contiguous() for w in weights):
            raise ValueError("weights must be contiguous (they are exchanged as bytes)")
        import torch.distributed as dist
        self._dist = dist if dist.is_available() and dist.is_initialized() else None
        self.group = group
        self.world = self._dist.get_world_size(group) if self._dist else 1
        self.rank = self._dist.get_rank(group) if self._dist else 0
        self.weights = list(weights)
        self.grads = list(grads)
        self.mode, self.nb = mode, nb
        shapes = [tuple(w.shape) for w in self.weights]
        self.owner = lpt_partition(matrix_costs(shapes, mode, nb), self.world)
        self.owned = [i for i, o in enumerate(self.owner) if o == self.rank]
        self.momentum = {i: torch.zeros(self.weights[i].shape, dtype=torch.float32,
                                        device=self.weights[i].device)
                         for i in self.owned}
        triples = [(self.weights[i], self.grads[i], self.momentum[i]) for i in self.owned]
        make = engine if engine is not None else Muon
        self.engine = make(triples) if triples else None
        # exchange layout: every rank's owned weights, packed as bytes
        self._nbytes = [w.numel() * w.element_size() for w in self.weights]
        self._per_rank = [[i for i, o in enumerate(self.owner) if o == r]
                          for r in range(self.world)]
        self._rank_bytes = [sum(self._nbytes[i] for i in ids) for ids in self._per_rank]
        # bytes one exchange moves into every rank: the sum of the owners'
        # packed weights (an equal-size all-gather would move world x max)
        self.exchange_bytes = sum(self._rank_bytes)

    def step(self, *, async_gather: bool = False, **kw):
        """The owned matrices' step, then the weight exchange.  Returns None
        once the weights are exchanged, or (async_gather) a handle whose
        wait() must be called before any weight is read."""
        if self.engine is not None:
            self.engine.step(mode=mode_code(self.mode), nb=self.nb, **kw)
        if self.world == 1:
            return None
        pending = self._exchange()
        if async_gather:
            return pending
        pending.wait()
        return None

    def _exchange(self) -> _Pending:
        dev = self.weights[0].device
        bufs, works = {}, []
        for r in range(self.world):
            if self._rank_bytes[r] == 0:
                continue                       # owns nothing: nothing to send
            buf = torch.empty(self._rank_bytes[r], dtype=torch.uint8, device=dev)
            if r == self.rank:
                off = 0
                for i in self._per_rank[r]:
                    buf[off:off + self._nbytes[i]].copy_(
                        self.weights[i].contiguous().view(-1).view(torch.uint8))
                    off += self._nbytes[i]
            src = r if self.group is None else self._dist.get_global_rank(self.group, r)
            works.append(self._dist.broadcast(buf, src=src, group=self.group, async_op=True))
            bufs[r] = buf

        def finish():
            for r, buf in bufs.items():
                if r == self.rank:
                    continue
                o = 0
                for i in self._per_rank[r]:
                    w = self.weights[i]
                    w.view(-1).view(torch.uint8).copy_(buf[o:o + self._nbytes[i]])
                    o += self._nbytes[i]

        return _Pending(works, finish)

    def sync(self) -> None:
        if self.engine is not None:
            self.engine.sync()
