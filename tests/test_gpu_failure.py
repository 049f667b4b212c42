"""Failure detection on the GPU without a fault: a bounded wait that nothing
satisfies runs out after a short limit, records the timeout in a device
error word, and leaves the CUDA context usable for ordinary work."""
import ctypes

import pytest
import torch

from gpu_helpers import check_against_oracle, gpu_step, oracle_step
from newton_schulz_06_gb300 import Muon, _lib
from newton_schulz_06_gb300.inputs import random_case

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def test_bounded_wait_runs_out_and_context_survives():
    W, G, M = random_case(128, 256, 3, device=DEV)
    opt = Muon([(W, G, M)])
    err = torch.zeros(1, dtype=torch.int32, device=DEV)
    rc = _lib.lib().muon_debug_wait_timeout(opt._h, ctypes.c_void_p(err.data_ptr()), 200)
    assert rc == _lib.MUON_ERR_TIMEOUT, _lib.lib().muon_last_error(opt._h)
    assert int(err.item()) == 1          # the device's timeout code
    opt.close()
    # the context still runs the real kernels correctly
    trip = list(random_case(192, 320, 4, device=DEV))
    inp, wexp, oexp, _ = gpu_step([trip])
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], oracle_step(inp[0]),
                         w_gate="scaled")


def test_chained_launch_wait_runs_out_and_context_survives(monkeypatch):
    """A chained launch whose second products wait for counter rounds that
    never come (the skew of muon_debug_set_chain_test): the watcher's and the
    other bounded waits run out after the limit, the step reports
    MUON_ERR_TIMEOUT at sync, and a new handle steps correctly on the same
    context."""
    monkeypatch.setenv("MUON_CHAIN_MIN_TILES", "0")
    monkeypatch.setenv("MUON_WAIT_LIMIT_MS", "300")
    W, G, M = random_case(512, 1024, 5, device=DEV)
    opt = Muon([(W, G, M)])
    opt.set_chain_test(skew_rounds=1000)
    opt.ensure_workspace(_lib.MUON_FULL, 1)
    assert opt.plan_info()["chained_groups"] == 1
    opt.step()
    with pytest.raises(_lib.MuonError) as ei:
        opt.sync()
    assert ei.value.code == _lib.MUON_ERR_TIMEOUT
    opt.close()
    trip = list(random_case(512, 1024, 6, device=DEV))
    inp, wexp, oexp, opt2 = gpu_step([trip])
    assert opt2.plan_info()["chained_groups"] == 1
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], oracle_step(inp[0]))
