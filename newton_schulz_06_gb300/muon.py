"""Python face of libmuon: register torch tensors, own the workspace, step.

PyTorch supplies device memory and the stream; every step of the optimizer
runs in libmuon's kernels.  Nothing here computes.

    from newton_schulz_06_gb300 import Muon
    opt = Muon([(W, G, M), ...])          # device tensors, row-major 2-D
    opt.step(lr=0.02, beta=0.95)           # queued on the current stream
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import torch

from . import _lib
from ._lib import check, lib

DEFAULT_COEFFS = (3.4445, -4.7750, 2.0315)

_DT = {torch.float32: _lib.MUON_F32, torch.bfloat16: _lib.MUON_BF16}


def _param(W: torch.Tensor, G: torch.Tensor, M: torch.Tensor) -> _lib.MuonParam:
    for name, t in (("W", W), ("G", G), ("M", M)):
        if t.dim() != 2:
            raise ValueError(f"{name} must be 2-D, got {tuple(t.shape)}")
        if t.stride(1) != 1:
            raise ValueError(f"{name} must be row-major (stride(1) == 1)")
    if W.shape != G.shape or W.shape != M.shape:
        raise ValueError(f"shape mismatch {W.shape} {G.shape} {M.shape}")
    if W.dtype not in _DT or G.dtype not in _DT:
        raise ValueError("W and G must be float32 or bfloat16")
    if M.dtype != torch.float32:
        raise ValueError("M (momentum) must be float32")
    p = _lib.MuonParam()
    p.w, p.g, p.m = W.data_ptr(), G.data_ptr(), M.data_ptr()
    p.rows, p.cols = W.shape
    p.ld_w, p.ld_g, p.ld_m = W.stride(0), G.stride(0), M.stride(0)
    p.w_dtype, p.g_dtype = _DT[W.dtype], _DT[G.dtype]
    return p



def mode_code(name: str) -> int:
    """The C ABI's mode constant for "full", "blockwise" or "distributed"."""
    return {"full": _lib.MUON_FULL, "blockwise": _lib.MUON_BLOCKWISE,
            "distributed": _lib.MUON_DISTRIBUTED}[name]

class Muon:
    """One libmuon handle over a fixed list of (W, G, M) device tensors."""

    def __init__(self, params: Sequence[Tuple[torch.Tensor, torch.Tensor,
                                              torch.Tensor]],
                 device: Optional[int] = None, stream=None):
        if not params:
            raise ValueError("need at least one parameter")
        dev = params[0][0].device
        if dev.type != "cuda":
            raise ValueError("libmuon runs on CUDA tensors only")
        self.device = dev.index if device is None else device
        self._tensors = [tuple(t) for t in params]   # keep alive
        self._h = ctypes.c_void_p()
        s = stream if stream is not None else torch.cuda.current_stream(self.device)
        check(lib().muon_create(ctypes.byref(self._h), self.device,
                                ctypes.c_void_p(s.cuda_stream)))
        arr = (_lib.MuonParam * len(params))(*[_param(*p) for p in params])
        check(lib().muon_register_params(self._h, len(params), arr), self._h)
        self._ws = None
        self._ws_key = None
        self._exports = None

    # -- workspace -------------------------------------------------------
    def workspace_size(self, mode: int = _lib.MUON_FULL, nb: int = 1):
        mn, full = ctypes.c_size_t(), ctypes.c_size_t()
        check(lib().muon_workspace_size(self._h, mode, nb, ctypes.byref(mn),
                                        ctypes.byref(full)), self._h)
        return mn.value, full.value

    def set_workspace(self, nbytes: int):
        """Allocates (through torch) and hands over a workspace of nbytes."""
        buf = torch.empty(nbytes + 1024, dtype=torch.uint8,
                          device=f"cuda:{self.device}")
        base = buf.data_ptr()
        off = (-base) % 1024
        check(lib().muon_set_workspace(self._h, ctypes.c_void_p(base + off),
                                       nbytes), self._h)
        self._ws = buf
        return nbytes

    def ensure_workspace(self, mode: int, nb: int,
                         max_bytes: Optional[int] = None):
        mn, full = self.workspace_size(mode, nb)
        want = full if max_bytes is None else max(mn, min(full, max_bytes))
        key = (mode, nb, want)
        if self._ws is None or self._ws_key != key:
            self._ws = None
            self.set_workspace(want)
            self._ws_key = key
        return want

    # -- stepping --------------------------------------------------------
    def step(self, lr: float = 0.02, beta: float = 0.95, nesterov: bool = True,
             ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
             mode: int = _lib.MUON_FULL, nb: int = 1,
             max_workspace: Optional[int] = None):
        if self._ws is None:
            self.ensure_workspace(mode, nb, max_workspace)
        a, b, c = coeffs
        check(lib().muon_step(self._h, lr, beta, int(bool(nesterov)),
                              ns_steps, a, b, c, mode, nb), self._h)

    def step_host(self, g_host, w_host, lr: float = 0.02, beta: float = 0.95,
                  nesterov: bool = True, ns_steps: int = 5, coeffs=DEFAULT_COEFFS,
                  mode: int = _lib.MUON_FULL, nb: int = 1,
                  max_workspace: Optional[int] = None):
        """One step with gradients from, and weights back to, host memory
        (contiguous CPU tensors, ideally pinned; w_host entries may be None).
        The tensors must stay alive and unchanged until sync()."""
        if self._ws is None:
            self.ensure_workspace(mode, nb, max_workspace)
        n = len(self._tensors)
        if len(g_host) != n or len(w_host) != n:
            raise ValueError(f"need {n} gradient and weight host tensors")
        gp = (ctypes.c_void_p * n)(*[g.data_ptr() for g in g_host])
        wp = (ctypes.c_void_p * n)(*[None if w is None else w.data_ptr() for w in w_host])
        a, b, c = coeffs
        check(lib().muon_step_host(self._h, n, gp, wp, lr, beta, int(bool(nesterov)),
                                   ns_steps, a, b, c, mode, nb), self._h)

    def sync(self):
        check(lib().muon_sync(self._h), self._h)

    def set_stream(self, stream):
        check(lib().muon_set_stream(self._h, ctypes.c_void_p(stream.cuda_stream)),
              self._h)

    # -- measurement / validation ----------------------------------------
    def set_profiling(self, on: bool):
        check(lib().muon_set_profiling(self._h, int(bool(on))), self._h)

    def stage_times(self):
        ms = (ctypes.c_float * _lib.MUON_N_STAGES)()
        n = (ctypes.c_int * _lib.MUON_N_STAGES)()
        check(lib().muon_stage_times(self._h, ms, n, _lib.MUON_N_STAGES),
              self._h)
        return {k: (ms[i], n[i]) for i, k in enumerate(_lib.STAGE_NAMES)}

    def last_launch_count(self) -> int:
        return lib().muon_last_launch_count(self._h)

    def set_exports(self, w_f32: Optional[List[torch.Tensor]],
                    o_bf16: Optional[List[torch.Tensor]]):
        n = len(self._tensors)
        if w_f32 is None and o_bf16 is None:
            check(lib().muon_debug_set_exports(self._h, 0, None, None), self._h)
            self._exports = None
            return
        wp = (ctypes.c_void_p * n)(*[t.data_ptr() if t is not None else None
                                     for t in (w_f32 or [None] * n)])
        op = (ctypes.c_void_p * n)(*[t.data_ptr() if t is not None else None
                                     for t in (o_bf16 or [None] * n)])
        check(lib().muon_debug_set_exports(self._h, n, wp, op), self._h)
        self._exports = (w_f32, o_bf16)

    def plan_info(self, mode: int = _lib.MUON_FULL, nb: int = 1) -> dict:
        info = _lib.MuonPlanInfo()
        check(lib().muon_get_plan_info(self._h, mode, nb, ctypes.byref(info)),
              self._h)
        return {k: getattr(info, k) for k, _ in info._fields_}

    def set_chain_test(self, skew_rounds: int = 0):
        """Validation of the chained launch: waits that run out (skew rounds
        that never come); 0 = normal operation."""
        check(lib().muon_debug_set_chain_test(self._h, int(skew_rounds)), self._h)

    def close(self):
        if self._h:
            lib().muon_destroy(self._h)
            self._h = ctypes.c_void_p()
        self._ws = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class HostPlanner:
    """A host-only libmuon handle: plan statistics and workspace sizes for
    a list of shapes, with no CUDA call (usable without a GPU)."""

    def __init__(self, shapes, w_dtype=_lib.MUON_BF16, g_dtype=_lib.MUON_BF16):
        self._h = ctypes.c_void_p()
        check(lib().muon_create(ctypes.byref(self._h), _lib.MUON_HOST_ONLY,
                                None))
        arr = (_lib.MuonParam * len(shapes))()
        for i, (r, c) in enumerate(shapes):
            p = arr[i]
            p.w = p.g = p.m = 0x1000   # never dereferenced by a host handle
            p.rows, p.cols = r, c
            p.ld_w = p.ld_g = p.ld_m = c
            p.w_dtype, p.g_dtype = w_dtype, g_dtype
        self.rc = lib().muon_register_params(self._h, len(shapes), arr)
        check(self.rc, self._h)

    def workspace_size(self, mode=_lib.MUON_FULL, nb=1):
        mn, full = ctypes.c_size_t(), ctypes.c_size_t()
        check(lib().muon_workspace_size(self._h, mode, nb, ctypes.byref(mn),
                                        ctypes.byref(full)), self._h)
        return mn.value, full.value

    def plan_info(self, mode=_lib.MUON_FULL, nb=1) -> dict:
        info = _lib.MuonPlanInfo()
        check(lib().muon_get_plan_info(self._h, mode, nb, ctypes.byref(info)),
              self._h)
        return {k: getattr(info, k) for k, _ in info._fields_}

    def check_chain_schedule(self, mode=_lib.MUON_FULL, nb=1) -> None:
        """Raises if a chained launch's per-pair tile lists for these shapes
        would break the properties its waits rely on."""
        check(lib().muon_debug_check_chain_schedule(self._h, mode, nb), self._h)

    def close(self):
        if self._h:
            lib().muon_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
