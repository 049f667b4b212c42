"""Plain float64 CPU oracle of one Muon optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only the test-suite, the smoke check of the package entry file and the CPU
baseline leg of the benchmark script run it.  It shares no code, tables or
constants with the CUDA library; every quantity it needs arrives as an
argument.

What it computes, and where it comes from (pages are cited by title and
section; see the design notes for the readings taken where they are silent):

* "Advancing Emerging Optimizers for Accelerated LLM Training" (NVIDIA
  developer blog, reproduced as a Chinese translation, section
  "Distributed Newton-Schulz" / "Duplicated mode"): each layer keeps a full
  momentum-buffer matrix, the momentum is orthogonalised by Newton-Schulz
  iterations ("usually five"), and the weights are updated with the
  orthogonalised momentum.
* Same page, "Distributed mode": every Newton-Schulz iteration consists of
  three matrix products.  The three products are taken in their standard
  quintic form  A = X X^T,  B = b A + c A A,  X <- a X + B X  with one fixed
  coefficient triple (a, b, c) for every iteration.
* Same page, "Blockwise mode": orthogonalisation and update use only a block
  of the momentum / weight; here the block is one of nb equal contiguous
  column blocks and is treated exactly like a matrix of its own.
* Same page, "Distributed mode": the iteration's work is spread over the
  ranks of a tensor-parallel group, with one all-reduce after the first of
  the three products of every iteration.  Reading: each rank holds an equal
  contiguous slice of the iterate's long side (X = [X_0 ... X_{P-1}]), so
  A = sum_p X_p X_p^T is the reduced sum of per-rank partial products, B is
  formed from the reduced A, and X_p <- a X_p + B X_p is local.  The norm of
  the whole matrix is the square root of the summed per-rank squares.

Readings where the pages are silent (stated once, used everywhere):
  momentum      M <- beta*M + G ; Nesterov U = G + beta*M_new, else U = M_new
  orientation   if rows > cols the iteration runs on U^T (short side first)
                and the result is transposed back
  normalisation X0 = U / (||U||_F + eps)
  shape scale   max(1, rows/cols) ** 0.5 of the (block) shape
  update        W <- W - lr * scale * O

Every step is plain float64 numpy; matrix products use numpy's ``@``.  There
is no blocking, fusion or reordering beyond the algorithm as stated.
Parity of the end-to-end step against a number printed on the pages is
unpinned (the pages print no worked example); each part is pinned in
tests/test_oracle.py by closed forms, brute force and invariants instead.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "momentum_update",
    "frobenius_normalise",
    "newton_schulz",
    "shape_scale",
    "muon_step_matrix",
    "muon_step",
    "column_blocks",
    "shard_ranges",
    "newton_schulz_distributed",
]


def momentum_update(M, G, beta, nesterov):
    """Heavy-ball momentum on the full momentum-buffer matrix.

    Returns (M_new, U): the new buffer and the matrix handed to the
    orthogonalisation ("momentum buffer matrix", page "Advancing Emerging
    Optimizers ...", section "Distributed Newton-Schulz").
    """
    M = np.asarray(M, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    M_new = beta * M + G
    U = G + beta * M_new if nesterov else M_new
    return M_new, U


def frobenius_normalise(U, eps):
    """X0 = U / (||U||_F + eps); the Frobenius norm summed in float64."""
    U = np.asarray(U, dtype=np.float64)
    s = np.sqrt(np.sum(U * U))
    return U / (s + eps)


def newton_schulz(X, steps, a, b, c):
    """``steps`` quintic Newton-Schulz iterations, three products each.

    X is m x n with m <= n (the caller orients it).  Each iteration takes the
    three products in order (section "Distributed mode": three matrix
    multiplications per iteration): A = X X^T, B = b A + c A A,
    X <- a X + B X.
    """
    X = np.array(X, dtype=np.float64, copy=True)
    for _ in range(steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X


def shard_ranges(n, shards):
    """Column ranges of the P equal contiguous slices of the long side."""
    if shards <= 0 or n % shards != 0:
        raise ValueError(f"{shards} shards must divide n={n}")
    w = n // shards
    return [(p * w, (p + 1) * w) for p in range(shards)]


def newton_schulz_distributed(X, steps, a, b, c, shards):
    """The iteration as the ranks of a P-way tensor-parallel group run it
    (section "Distributed mode"): per iteration every rank forms the partial
    product of its slice, the partials are summed (the all-reduce after the
    first product), then B and the slice update follow from the sum.
    """
    X = np.array(X, dtype=np.float64, copy=True)
    parts = shard_ranges(X.shape[1], shards)
    for _ in range(steps):
        A = np.zeros((X.shape[0], X.shape[0]))
        for lo, hi in parts:                  # all-reduce of the partials
            A += X[:, lo:hi] @ X[:, lo:hi].T
        B = b * A + c * (A @ A)
        Xn = np.empty_like(X)
        for lo, hi in parts:                  # local to each rank
            Xn[:, lo:hi] = a * X[:, lo:hi] + B @ X[:, lo:hi]
        X = Xn
    return X


def shape_scale(rows, cols):
    """max(1, rows/cols) ** 0.5 for a rows x cols (block of a) weight."""
    return max(1.0, rows / cols) ** 0.5


def muon_step_matrix(W, G, M, *, lr, beta, nesterov, ns_steps, a, b, c,
                     eps=1e-7, shards=0):
    """One Muon step on one weight matrix (or one block treated as one).

    With shards = P > 0 the iteration runs in distributed mode over P slices
    of the iterate's long side.  Returns a dict of float64 arrays: ``W``
    (updated weight), ``M`` (updated momentum) and ``O`` (orthogonalised
    update in the weight's orientation).
    """
    W = np.asarray(W, dtype=np.float64)
    rows, cols = W.shape
    M_new, U = momentum_update(M, G, beta, nesterov)
    tall = rows > cols
    X0 = frobenius_normalise(U.T if tall else U, eps)
    if shards:
        X = newton_schulz_distributed(X0, ns_steps, a, b, c, shards)
    else:
        X = newton_schulz(X0, ns_steps, a, b, c)
    O = X.T if tall else X
    W_new = W - lr * shape_scale(rows, cols) * O
    return {"W": W_new, "M": M_new, "O": O}


def column_blocks(cols, nb):
    """Column ranges of the nb equal contiguous blocks ("Blockwise mode")."""
    if nb <= 0 or cols % nb != 0:
        raise ValueError(f"nb={nb} must divide cols={cols}")
    w = cols // nb
    return [(j * w, (j + 1) * w) for j in range(nb)]


def muon_step(W, G, M, *, lr, beta, nesterov, ns_steps, a, b, c,
              mode="full", nb=1, eps=1e-7):
    """One Muon step in full, blockwise or distributed mode.

    Blockwise mode splits the columns into nb equal blocks and runs the whole
    step on each block as an independent matrix: its own norm, its own
    iteration and its own shape scale (section "Blockwise mode").
    Distributed mode runs the full step with the iteration spread over nb
    tensor-parallel slices of the iterate's long side (section "Distributed
    mode").
    """
    W = np.asarray(W, dtype=np.float64)
    G = np.asarray(G, dtype=np.float64)
    M = np.asarray(M, dtype=np.float64)
    kw = dict(lr=lr, beta=beta, nesterov=nesterov, ns_steps=ns_steps,
              a=a, b=b, c=c, eps=eps)
    if mode == "full":
        return muon_step_matrix(W, G, M, **kw)
    if mode == "distributed":
        return muon_step_matrix(W, G, M, shards=nb, **kw)
    if mode != "blockwise":
        raise ValueError(f"unknown mode {mode!r}")
    out = {"W": np.empty_like(W), "M": np.empty_like(M), "O": np.empty_like(W)}
    for lo, hi in column_blocks(W.shape[1], nb):
        r = muon_step_matrix(W[:, lo:hi], G[:, lo:hi], M[:, lo:hi], **kw)
        for k in out:
            out[k][:, lo:hi] = r[k]
    return out
