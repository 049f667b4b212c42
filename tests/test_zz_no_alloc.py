"""muon_step_noalloc against muon_step, through the C ABI, on the GPU.

muon_step_noalloc serves callers that cannot call cudaMalloc or hand the
library a workspace (a plugin whose host owns device memory through a pool it
does not expose, a process whose caching allocator has reserved the GPU, a hot
loop that cannot afford cudaMalloc's device synchronisation); its scratch is a
fixed array inside the library.  Here two calls in a row must give the same
weights and momenta as two calls of the workspace-based muon_step on copies
of the same inputs, within the tolerances of the parity tests.  The file is
named to run last; it passes on its own in a fresh process as well.
"""
import ctypes

import numpy as np
import pytest
import torch

from newton_schulz_06_gb300 import Muon, _lib
from newton_schulz_06_gb300.inputs import random_case
from newton_schulz_06_gb300.muon import _param

pytestmark = pytest.mark.gpu

COEFFS = tuple(float(np.float32(x)) for x in (3.4445, -4.7750, 2.0315))
LR, BETA = float(np.float32(0.02)), float(np.float32(0.95))


def relF(a, b):
    a = a.double().cpu()
    b = b.double().cpu()
    return (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item()


def noalloc_step(W, G, M):
    p = _param(W, G, M)
    buf = ctypes.create_string_buffer(512)
    rc = _lib.lib().muon_step_noalloc(
        ctypes.byref(p), LR, BETA, 1, 5, *COEFFS,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream), buf, 512)
    return rc, buf.value.decode()


@pytest.mark.parametrize("rows,cols", [(256, 640), (700, 300), (1024, 4096)])
def test_noalloc_matches_workspace_step_two_calls(rows, cols):
    W, G, M = random_case(rows, cols, 123, device="cuda:0")
    W2, G2, M2 = W.clone(), G.clone(), M.clone()
    opt = Muon([(W2, G2, M2)])
    for call in range(2):
        rc, msg = noalloc_step(W, G, M)
        assert rc == 0, msg
        opt.step(lr=LR, beta=BETA, nesterov=True, ns_steps=5, coeffs=COEFFS)
        opt.sync()
        torch.cuda.synchronize()
        assert relF(W, W2) <= 1e-3, (call, relF(W, W2))
        assert relF(M, M2) <= 1e-6, (call, relF(M, M2))
        # same planner, kernels and tile order as muon_step: the same bits
        assert torch.equal(W, W2), (rows, cols, call)
        assert torch.equal(M, M2), (rows, cols, call)
        # the next call gets a fresh gradient on both sides
        G.copy_(G.flip(0))
        G2.copy_(G)
    opt.close()


def test_noalloc_rejects_a_matrix_beyond_its_scratch():
    W, G, M = random_case(2048, 2048, 5, device="cuda:0")
    W0, M0 = W.clone(), M.clone()
    rc, msg = noalloc_step(W, G, M)
    torch.cuda.synchronize()
    assert rc == _lib.MUON_ERR_UNSUPPORTED
    assert "33554432" in msg and "workspace" in msg
    assert torch.equal(W, W0) and torch.equal(M, M0)
