"""Seeded synthetic workloads: shapes and random inputs, nothing else.

This module is shared by the tests (which feed the same tensors to the CUDA
library and to the float64 oracle) and by the benchmark.  It holds no part of
the optimizer's arithmetic: only matrix shapes, dtypes and the random
distributions of weights, gradients and initial momenta.

Shapes follow the model families the pages name (Kimi K2 and Qwen3-30B-A3B,
"Advancing Emerging Optimizers for Accelerated LLM Training", section
"Muon training performance on NVIDIA GB300 NVL72"); their sizes are those of
the public model architectures.  All data are synthetic: no dataset or
trained weight is used.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import List, Optional, Tuple

import torch

# Coefficients of the quintic Newton-Schulz polynomial used throughout.
NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_STEPS = 5
# Hyper-parameters of the single-matrix workload; reused by the others.
LR = 0.02
BETA = 0.95
NESTEROV = True
WEIGHT_STD = 0.02


@dataclasses.dataclass
class Workload:
    name: str
    shapes: List[Tuple[int, int]]
    w_dtype: torch.dtype
    g_dtype: torch.dtype
    grad: str                # "normal" | "log_scale_step" | "log_sigma"
    grad_std: float = 1.0
    init_momentum: str = "zero"   # "zero" | "normal"
    steps: int = 1
    mode: str = "full"
    nb: int = 1

    @property
    def n_matrices(self) -> int:
        return len(self.shapes)

    @property
    def n_elements(self) -> int:
        return sum(r * c for r, c in self.shapes)


def qwen3_30b_a3b_block_shapes() -> List[Tuple[int, int]]:
    """One Qwen3-30B-A3B MoE block (hidden 2048): q, k, v, o projections and
    128 experts with gate, up and down projections (388 matrices)."""
    shapes = [(4096, 2048), (512, 2048), (512, 2048), (2048, 4096)]
    for _ in range(128):
        shapes += [(768, 2048), (768, 2048), (2048, 768)]
    return shapes


def kimi_k2_layer_shapes(n_experts: int = 48) -> List[Tuple[int, int]]:
    """A Kimi-K2 MoE layer (hidden 7168): the MLA projections q_a, q_b,
    kv_a, kv_b, o and ``n_experts`` experts with gate, up and down."""
    shapes = [(1536, 7168), (12288, 1536), (576, 7168), (16384, 512),
              (7168, 8192)]
    for _ in range(n_experts):
        shapes += [(2048, 7168), (2048, 7168), (7168, 2048)]
    return shapes


def workload(name: str) -> Workload:
    """The named synthetic workloads."""
    if name == "single_256x512_f32":
        return Workload(name, [(256, 512)], torch.float32, torch.float32,
                        grad="normal", init_momentum="normal")
    if name == "square_4096_bf16":
        return Workload(name, [(4096, 4096)], torch.bfloat16, torch.bfloat16,
                        grad="log_scale_step", steps=20)
    if name == "qwen3_30b_a3b_block":
        return Workload(name, qwen3_30b_a3b_block_shapes(), torch.bfloat16,
                        torch.bfloat16, grad="log_sigma")
    if name == "qwen3_30b_a3b_48_layers":
        return Workload(name, qwen3_30b_a3b_block_shapes() * 48,
                        torch.bfloat16, torch.bfloat16, grad="log_sigma",
                        steps=10)
    if name == "kimi_k2_layer_full":
        return Workload(name, kimi_k2_layer_shapes(), torch.bfloat16,
                        torch.bfloat16, grad="normal", grad_std=1e-2)
    if name == "kimi_k2_layer_blockwise4":
        return Workload(name, kimi_k2_layer_shapes(), torch.bfloat16,
                        torch.bfloat16, grad="normal", grad_std=1e-2,
                        mode="blockwise", nb=4)
    if name == "square_4096_f32":
        # fp32 weights and gradients at the square size: the update runs as
        # its own pass (measurement of that pass's HBM rate)
        return Workload(name, [(4096, 4096)], torch.float32, torch.float32,
                        grad="log_scale_step", steps=20)
    if name == "square_4096_bf16_distributed4":
        return Workload(name, [(4096, 4096)], torch.bfloat16, torch.bfloat16,
                        grad="log_scale_step", mode="distributed", nb=4)
    if name == "qwen3_30b_a3b_block_distributed4":
        return Workload(name, qwen3_30b_a3b_block_shapes(), torch.bfloat16,
                        torch.bfloat16, grad="log_sigma", mode="distributed",
                        nb=4)
    raise KeyError(name)


WORKLOADS = ["single_256x512_f32", "square_4096_bf16", "qwen3_30b_a3b_block",
             "qwen3_30b_a3b_48_layers", "kimi_k2_layer_full",
             "kimi_k2_layer_blockwise4", "square_4096_bf16_distributed4",
             "qwen3_30b_a3b_block_distributed4", "square_4096_f32"]


def seed_for(*parts) -> int:
    """A stable 63-bit seed from any tuple of names and integers."""
    h = hashlib.sha256("/".join(str(p) for p in parts).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _gen(device, *parts) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed_for(*parts))
    return g


def make_weight(shape, dtype, device, *seed_parts) -> torch.Tensor:
    g = _gen(device, "W", *seed_parts)
    return (torch.randn(shape, generator=g, device=device,
                        dtype=torch.float32) * WEIGHT_STD).to(dtype)


def make_momentum(shape, kind, device, *seed_parts) -> torch.Tensor:
    if kind == "zero":
        return torch.zeros(shape, device=device, dtype=torch.float32)
    g = _gen(device, "M", *seed_parts)
    return torch.randn(shape, generator=g, device=device, dtype=torch.float32)


def grad_scale(wl: Workload, idx: int, step: int) -> float:
    """The scalar standard deviation of matrix ``idx``'s gradient at ``step``."""
    if wl.grad == "normal":
        return wl.grad_std
    gen = torch.Generator().manual_seed(seed_for("S", wl.name, idx, step))
    u = torch.rand((), generator=gen, dtype=torch.float64).item()
    if wl.grad == "log_scale_step":        # 10 ** U(-3, 0), fresh every step
        return 10.0 ** (-3.0 + 3.0 * u)
    if wl.grad == "log_sigma":             # 10 ** U(-4, -1), fixed per matrix
        gen = torch.Generator().manual_seed(seed_for("S", wl.name, idx))
        u = torch.rand((), generator=gen, dtype=torch.float64).item()
        return 10.0 ** (-4.0 + 3.0 * u)
    raise ValueError(wl.grad)


def fill_grad(out: torch.Tensor, wl: Workload, idx: int, step: int) -> None:
    """Write matrix ``idx``'s gradient for ``step`` into ``out`` in place."""
    g = _gen(out.device, "G", wl.name, idx, step)
    tmp = torch.randn(out.shape, generator=g, device=out.device,
                      dtype=torch.float32)
    tmp.mul_(grad_scale(wl, idx, step))
    out.copy_(tmp)


def make_state(wl: Workload, device, shapes: Optional[List] = None):
    """Weights, zero/normal momenta and first-step gradients for a workload.

    Returns (W list, G list, M list).  ``shapes`` may restrict the set (used
    by tests that take a sample of a large workload); default all."""
    shapes = wl.shapes if shapes is None else shapes
    Ws, Gs, Ms = [], [], []
    for i, (r, c) in enumerate(shapes):
        Ws.append(make_weight((r, c), wl.w_dtype, device, wl.name, i))
        Ms.append(make_momentum((r, c), wl.init_momentum, device, wl.name, i))
        G = torch.empty((r, c), device=device, dtype=wl.g_dtype)
        fill_grad(G, wl, i, 0)
        Gs.append(G)
    return Ws, Gs, Ms


def random_case(rows, cols, seed, *, w_dtype=torch.bfloat16,
                g_dtype=torch.bfloat16, grad_std=1.0, momentum="normal",
                device="cpu"):
    """One seeded (W, G, M) triple of any shape for parity tests."""
    W = make_weight((rows, cols), w_dtype, device, "case", rows, cols, seed)
    M = make_momentum((rows, cols), momentum, device, "case", rows, cols, seed)
    g = _gen(device, "Gcase", rows, cols, seed)
    G = (torch.randn((rows, cols), generator=g, device=device,
                     dtype=torch.float32) * grad_std).to(g_dtype)
    return W, G, M
