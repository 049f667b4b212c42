"""Layer-wise distributed Muon: the partition and the weight exchange, as
two gloo ranks on the CPU.  The local step is libmuon on a GPU; here a
stand-in engine applies a fixed update to the owned matrices, so the test
checks ownership, momentum placement and that after the exchange every rank
holds every matrix exactly as its owner updated it."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp

from newton_schulz_06_gb300.layerwise import lpt_partition, matrix_costs


def test_lpt_partition_hand_example_and_invariants():
    # costs 5,4,3,3,2 on two ranks: 5->r0, 4->r1, 3->r1 (4<5), 3->r0 (5<7),
    # 2->r1 (7<8)
    assert lpt_partition([5, 4, 3, 3, 2], 2) == [0, 1, 1, 0, 1]
    assert lpt_partition([7], 4) == [0]
    g = torch.Generator().manual_seed(3)
    costs = [int(x) for x in torch.randint(1, 1000, (57,), generator=g)]
    for world in (1, 2, 3, 8):
        own = lpt_partition(costs, world)
        assert own == lpt_partition(costs, world)           # deterministic
        loads = [sum(c for c, o in zip(costs, own) if o == r) for r in range(world)]
        assert sum(loads) == sum(costs)
        assert max(loads) - min(loads) <= max(costs)        # LPT's bound
    shapes = [(4096, 2048), (768, 2048), (2048, 768), (512, 2048)]
    c = matrix_costs(shapes)
    assert c[1] == c[2] and c[0] > c[1] > c[3]              # orientation-free


class _StandIn:
    """Local stepper for the CPU test: W <- W - 0.125 * G, M <- M + G."""

    def __init__(self, triples):
        self.triples = triples

    def step(self, **kw):
        for W, G, M in self.triples:
            W.sub_(0.125 * G)
            M.add_(G)

    def sync(self):
        pass


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q, async_gather):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import torch.distributed as dist
    from newton_schulz_06_gb300.layerwise import LayerwiseMuon
    dist.init_process_group("gloo", rank=rank, world_size=world)
    # shapes of very different sizes, so the ranks own very different bytes
    shapes = [(64, 32), (16, 48), (40, 40), (8, 8), (96, 16), (24, 72), (33, 5),
              (256, 128), (4, 4)]
    g = torch.Generator().manual_seed(11)
    W0 = [torch.randn(s, generator=g).to(torch.bfloat16) for s in shapes]
    G = [torch.randn(s, generator=g).to(torch.bfloat16) for s in shapes]
    W = [w.clone() for w in W0]
    opt = LayerwiseMuon(W, G, engine=_StandIn)
    h = opt.step(async_gather=async_gather)
    if async_gather:
        h.wait()
    want = [w0 - 0.125 * g0 for w0, g0 in zip(W0, G)]
    ok = all(torch.equal(w, x) for w, x in zip(W, want))
    # the exchange moves the weights' bytes once, with no padding
    ok = ok and opt.exchange_bytes == sum(w.numel() * w.element_size() for w in W)
    q.put((rank, opt.owned, sorted(opt.momentum), ok,
           [float(w.float().sum()) for w in W]))
    dist.destroy_process_group()


@pytest.mark.parametrize("world,async_gather", [(2, False), (2, True), (3, False)])
def test_gloo_ranks_exchange_updated_weights(world, async_gather):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q, async_gather))
             for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    owned = [o[1] for o in out]
    assert all(o[3] for o in out)            # every matrix as its owner updated it
    assert sorted(sum(owned, [])) == list(range(9))
    assert sum(len(o) for o in owned) == len(set(sum(owned, [])))   # disjoint
    assert all(o[2] == o[1] for o in out)    # momentum only for owned matrices
    assert all(o[4] == out[0][4] for o in out)   # every rank holds the same weights
