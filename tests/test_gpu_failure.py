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
    check_against_oracle(trip, inp[0], wexp[0], oexp[0], oracle_step(inp[0]))
