"""FLOP accounting of the orthogonalisation, counted two ways.

For a unit oriented m x n (m = short side), one Newton-Schulz iteration
takes three products (section "Distributed mode" of "Advancing Emerging
Optimizers for Accelerated LLM Training"): X X^T (m x m, K = n), A A
(m x m, K = m) and B X (m x n, K = m).
  * GEMM-equivalent: every product counted as a full GEMM,
        2 m^2 n + 2 m^3 + 2 m^2 n = 4 m^2 n + 2 m^3 per iteration;
  * useful: the two symmetric products counted on their upper triangle
    including the diagonal (section "SYRK and fused all-reduce": close to
    half the FLOPs are saved), m (m+1) n + m (m+1) m + 2 m^2 n.
"""
from __future__ import annotations


def unit_shapes(rows, cols, mode="full", nb=1):
    """(m, n) of each unit a rows x cols matrix contributes."""
    if mode == "blockwise":
        cols = cols // nb
        k = nb
    else:
        k = 1
    return [(min(rows, cols), max(rows, cols))] * k


def gemm_equiv_flops(shapes, ns_steps=5, mode="full", nb=1) -> int:
    tot = 0
    for r, c in shapes:
        for m, n in unit_shapes(r, c, mode, nb):
            tot += 4 * m * m * n + 2 * m ** 3
    return tot * ns_steps


def useful_flops(shapes, ns_steps=5, mode="full", nb=1) -> int:
    tot = 0
    for r, c in shapes:
        for m, n in unit_shapes(r, c, mode, nb):
            tot += m * (m + 1) * n + m * (m + 1) * m + 2 * m * m * n
    return tot * ns_steps
