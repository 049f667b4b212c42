"""Pins of the float64 oracle against facts that do not come from the oracle.

The pages print no worked example of the step ("Advancing Emerging Optimizers
for Accelerated LLM Training" and its summaries give only end-to-end training
throughput), so the oracle is pinned by mathematics:

* closed form: one quintic iteration maps every singular value x of X to
  p(x) = a x + b x^3 + c x^5 and keeps the singular vectors, so the whole
  orthogonalisation is U diag(p∘p∘p∘p∘p(s / (||s|| + eps))) V^T.  The scalar
  polynomial here is iterated on numbers, not on matrices, and the singular
  vectors come from LAPACK's SVD;
* brute force: the three products of one iteration with pure-Python loops;
* the band that p∘…∘p maps [x*, 1] into, found on a dense grid;
* the geometric-series closed form of repeated momentum updates;
* invariants (transpose, blockwise nb=1, zero gradient);
* mutation checks: plausible mistakes planted in a copy of the oracle are
  each rejected by one of the pins above.
"""
import numpy as np
import pytest

import oracle
from oracle import muon_ref

A_, B_, C_ = 3.4445, -4.7750, 2.0315
EPS = 1e-7


def p_iter(x, steps, a=A_, b=B_, c=C_):
    x = np.asarray(x, dtype=np.float64)
    for _ in range(steps):
        x = a * x + b * x ** 3 + c * x ** 5
    return x


def svd_matrix(rows, cols, s, seed):
    rng = np.random.default_rng(seed)
    m = min(rows, cols)
    U, _ = np.linalg.qr(rng.standard_normal((rows, m)))
    V, _ = np.linalg.qr(rng.standard_normal((cols, m)))
    return U, V, (U * s) @ V.T


def closed_form_O(U, V, s, steps=5, eps=EPS):
    x = s / (np.sqrt(np.sum(s * s)) + eps)
    return (U * p_iter(x, steps)) @ V.T


def run(W, G, M, **kw):
    base = dict(lr=0.02, beta=0.95, nesterov=True, ns_steps=5, a=A_, b=B_,
                c=C_)
    base.update(kw)
    return oracle.muon_step(W, G, M, **base)


@pytest.mark.parametrize("rows,cols", [(8, 16), (16, 8), (12, 12), (48, 80),
                                       (96, 40)])
def test_closed_form_svd_constructed(rows, cols):
    m = min(rows, cols)
    s = np.geomspace(1e-3, 1.0, m)[::-1]
    U, V, G = svd_matrix(rows, cols, s, seed=rows * 131 + cols)
    out = run(np.zeros((rows, cols)), G, np.zeros((rows, cols)),
              nesterov=False, beta=0.9)
    expect = closed_form_O(U, V, s)
    assert np.max(np.abs(out["O"] - expect)) < 1e-12
    # M starts at zero and no Nesterov term: the buffer is the gradient.
    assert np.array_equal(out["M"], G)


@pytest.mark.parametrize("rows,cols", [(32, 64), (64, 32), (40, 40)])
def test_closed_form_from_lapack_svd_of_gaussian(rows, cols):
    """Any input: the result equals p^5 applied to LAPACK's singular values."""
    rng = np.random.default_rng(7 + rows)
    G = rng.standard_normal((rows, cols))
    out = run(np.zeros((rows, cols)), G, np.zeros((rows, cols)),
              nesterov=False)
    U, s, Vt = np.linalg.svd(G, full_matrices=False)
    expect = (U * p_iter(s / (np.linalg.norm(s) + EPS), 5)) @ Vt
    assert np.max(np.abs(out["O"] - expect)) < 1e-11


def test_eps_enters_the_normalisation():
    """At a norm of 1e-7 the eps term halves the normalised singular values."""
    s = np.array([6e-8, 8e-8, 0.0, 0.0])          # ||s|| = 1e-7
    U, V, G = svd_matrix(4, 8, s, seed=3)
    out = run(np.zeros((4, 8)), G, np.zeros((4, 8)), nesterov=False)
    x = np.array([0.3, 0.4, 0.0, 0.0])             # s / (1e-7 + 1e-7)
    expect = (U * p_iter(x, 5)) @ V.T
    assert np.max(np.abs(out["O"] - expect)) < 1e-12


def test_ns_steps_count():
    s = np.array([1.0, 0.5, 0.25, 0.1])
    U, V, G = svd_matrix(4, 9, s, seed=11)
    for steps in (1, 2, 3, 7):
        out = run(np.zeros((4, 9)), G, np.zeros((4, 9)), nesterov=False,
                  ns_steps=steps)
        assert np.allclose(out["O"], closed_form_O(U, V, s, steps),
                           atol=1e-12, rtol=0)


def _loops_ns(X, steps, a, b, c):
    """Pure-Python triple-loop products; no numpy matrix routine."""
    m, n = len(X), len(X[0])
    X = [list(map(float, row)) for row in X]
    for _ in range(steps):
        A = [[sum(X[i][k] * X[j][k] for k in range(n)) for j in range(m)]
             for i in range(m)]
        AA = [[sum(A[i][k] * A[k][j] for k in range(m)) for j in range(m)]
              for i in range(m)]
        Bm = [[b * A[i][j] + c * AA[i][j] for j in range(m)] for i in range(m)]
        BX = [[sum(Bm[i][k] * X[k][j] for k in range(m)) for j in range(n)]
              for i in range(m)]
        X = [[a * X[i][j] + BX[i][j] for j in range(n)] for i in range(m)]
    return np.array(X)


@pytest.mark.parametrize("m,n", [(8, 16), (8, 8), (5, 13)])
def test_products_against_triple_loops(m, n):
    rng = np.random.default_rng(m * 100 + n)
    X = rng.standard_normal((m, n))
    X /= np.linalg.norm(X)
    got = oracle.newton_schulz(X, 5, A_, B_, C_)
    want = _loops_ns(X.tolist(), 5, A_, B_, C_)
    assert np.max(np.abs(got - want)) < 1e-12


def _band(lo, steps=5):
    x = np.linspace(lo, 1.0, 400001)
    y = p_iter(x, steps)
    return y.min(), y.max()


@pytest.mark.parametrize("rows,cols", [(64, 256), (256, 96), (128, 128)])
def test_output_singular_values_in_band(rows, cols):
    rng = np.random.default_rng(rows + 3 * cols)
    G = rng.standard_normal((rows, cols))
    out = run(np.zeros((rows, cols)), G, np.zeros((rows, cols)),
              nesterov=False)
    s_in = np.linalg.svd(G, compute_uv=False)
    x_in = s_in / np.linalg.norm(s_in)
    s_out = np.linalg.svd(out["O"], compute_uv=False)
    lo, hi = _band(1.5e-3)
    # singular values of the input at or above x* land in the band
    keep = np.sort(x_in)[::-1] >= 1.5e-3
    assert np.all(s_out[keep] >= lo - 1e-9) and np.all(s_out[keep] <= hi + 1e-9)
    assert 0.67 < lo < 0.69 and 1.15 < _band(5e-3)[1] < 1.16


def test_momentum_geometric_series():
    """t updates with a constant gradient from zero: M_t = G (1-b^t)/(1-b)."""
    rng = np.random.default_rng(5)
    G = rng.standard_normal((3, 4))
    beta = 0.9
    M = np.zeros_like(G)
    for t in range(1, 6):
        M, U = muon_ref.momentum_update(M, G, beta, nesterov=True)
        geo = (1 - beta ** t) / (1 - beta)
        assert np.allclose(M, geo * G, rtol=1e-14, atol=0)
        assert np.allclose(U, (1 + beta * geo) * G, rtol=1e-14, atol=0)
        _, U2 = muon_ref.momentum_update(M / beta - G / beta, G, beta, False)
        assert np.allclose(U2, M, rtol=1e-13, atol=1e-13)


def test_momentum_worked_example():
    """Exact binary arithmetic by hand: beta=1/2, M=1, G=2 -> M'=5/2,
    Nesterov U = 2 + 5/4 = 13/4; without Nesterov U = M'."""
    M, U = muon_ref.momentum_update(np.array([[1.0]]), np.array([[2.0]]),
                                    0.5, nesterov=True)
    assert M[0, 0] == 2.5 and U[0, 0] == 3.25
    M, U = muon_ref.momentum_update(np.array([[1.0]]), np.array([[2.0]]),
                                    0.5, nesterov=False)
    assert M[0, 0] == 2.5 and U[0, 0] == 2.5


@pytest.mark.parametrize("rows,cols", [(48, 16), (16, 48), (24, 24)])
def test_weight_update_shape_scale(rows, cols):
    m = min(rows, cols)
    s = np.linspace(1.0, 0.05, m)
    U, V, G = svd_matrix(rows, cols, s, seed=rows + cols)
    rng = np.random.default_rng(1)
    W = rng.standard_normal((rows, cols))
    out = run(W, G, np.zeros((rows, cols)), nesterov=False, lr=0.1)
    scale = np.sqrt(rows / cols) if rows > cols else 1.0
    expect = W - 0.1 * scale * closed_form_O(U, V, s)
    assert np.max(np.abs(out["W"] - expect)) < 1e-12


def test_blockwise_closed_form():
    rows, cols, nb = 24, 64, 4
    w = cols // nb
    G = np.zeros((rows, cols))
    O = np.zeros((rows, cols))
    for j in range(nb):
        # 24 x 16 blocks are tall: scale sqrt(24/16) and short side 16
        s = np.geomspace(0.02, 1.0, w) * (j + 1) * 10.0 ** (-j)
        U, V, Gj = svd_matrix(rows, w, s, seed=40 + j)
        G[:, j * w:(j + 1) * w] = Gj
        O[:, j * w:(j + 1) * w] = closed_form_O(U, V, s)
    out = run(np.zeros((rows, cols)), G, np.zeros((rows, cols)),
              nesterov=False, mode="blockwise", nb=nb, lr=1.0)
    assert np.max(np.abs(out["O"] - O)) < 1e-12
    assert np.max(np.abs(out["W"] + np.sqrt(rows / w) * O)) < 1e-12


def test_blockwise_nb1_is_full():
    rng = np.random.default_rng(9)
    W, G, M = (rng.standard_normal((20, 30)) for _ in range(3))
    a = run(W, G, M, mode="blockwise", nb=1)
    b = run(W, G, M)
    for k in ("W", "M", "O"):
        assert np.array_equal(a[k], b[k])


def test_blockwise_rejects_nondividing_nb():
    z = np.zeros((4, 10))
    with pytest.raises(ValueError):
        run(z, z, z, mode="blockwise", nb=3)


def test_transpose_invariance():
    rng = np.random.default_rng(2)
    G = rng.standard_normal((24, 40))
    M = rng.standard_normal((24, 40))
    a = run(np.zeros((24, 40)), G, M)
    b = run(np.zeros((40, 24)), G.T, M.T)
    assert np.array_equal(a["O"], b["O"].T)


def test_zero_gradient_gives_zero_update():
    z = np.zeros((16, 32))
    W = np.arange(512, dtype=np.float64).reshape(16, 32)
    out = run(W, z, z)
    assert np.all(out["O"] == 0) and np.array_equal(out["W"], W)
    assert not np.any(np.isnan(out["O"]))


# --------------------------------------------------------------------------
# Mutation checks: a mistake planted in a copy of the oracle must be caught.

def _mutant_ns(kind):
    def ns(X, steps, a, b, c):
        X = np.array(X, dtype=np.float64, copy=True)
        for _ in range(steps):
            A = X @ X.T
            if kind == "drop_c":
                B = b * A
            elif kind == "sign_b":
                B = -b * A + c * (A @ A)
            elif kind == "no_square":
                B = b * A + c * A
            else:
                B = b * A + c * (A @ A)
            X = (X if kind == "drop_a" else a * X) + B @ X
        return X
    return ns


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("kind", ["drop_c", "sign_b", "no_square", "drop_a"])
def test_pins_reject_planted_ns_mistakes(kind, monkeypatch):
    monkeypatch.setattr(muon_ref, "newton_schulz", _mutant_ns(kind))
    s = np.geomspace(1e-2, 1.0, 8)[::-1]
    U, V, G = svd_matrix(8, 16, s, seed=1)
    out = muon_ref.muon_step(np.zeros((8, 16)), G, np.zeros((8, 16)), lr=0.1,
                             beta=0.9, nesterov=False, ns_steps=5, a=A_,
                             b=B_, c=C_)
    assert not np.max(np.abs(out["O"] - closed_form_O(U, V, s))) <= 1e-3


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
def test_pins_reject_planted_normalisation_mistake(monkeypatch):
    monkeypatch.setattr(muon_ref, "frobenius_normalise",
                        lambda U, eps: U / (np.abs(U).max() + eps))
    s = np.geomspace(1e-2, 1.0, 8)[::-1]
    U, V, G = svd_matrix(8, 16, s, seed=1)
    out = muon_ref.muon_step(np.zeros((8, 16)), G, np.zeros((8, 16)), lr=0.1,
                             beta=0.9, nesterov=False, ns_steps=5, a=A_,
                             b=B_, c=C_)
    assert not np.max(np.abs(out["O"] - closed_form_O(U, V, s))) <= 1e-3


def test_pins_reject_planted_scale_and_orientation_mistakes(monkeypatch):
    s = np.linspace(1.0, 0.1, 8)
    U, V, G = svd_matrix(32, 8, s, seed=4)
    expect = -0.1 * 2.0 * closed_form_O(U, V, s)
    monkeypatch.setattr(muon_ref, "shape_scale",
                        lambda r, c: max(1.0, c / r) ** 0.5)
    out = muon_ref.muon_step(np.zeros((32, 8)), G, np.zeros((32, 8)), lr=0.1,
                             beta=0.9, nesterov=False, ns_steps=5, a=A_,
                             b=B_, c=C_)
    assert not np.max(np.abs(out["W"] - expect)) <= 1e-3


# --------------------------------------------------------------------------
# Distributed mode: the iteration over P tensor-parallel slices of the
# iterate's long side, with the partial first products summed.

@pytest.mark.parametrize("rows,cols,P", [(8, 16, 2), (16, 8, 4), (12, 24, 3),
                                         (40, 96, 8)])
def test_distributed_closed_form(rows, cols, P):
    """The slices' summed partials give the same iteration: the closed form
    U p^5(s/||s||) V^T of an SVD-constructed input."""
    s = np.geomspace(1.0, 0.05, min(rows, cols))
    U, V, G = svd_matrix(rows, cols, s, seed=rows + 7 * cols + P)
    out = run(np.zeros((rows, cols)), G, np.zeros((rows, cols)), nesterov=False,
              beta=0.0, mode="distributed", nb=P)
    assert np.max(np.abs(out["O"] - closed_form_O(U, V, s))) < 1e-9


@pytest.mark.parametrize("m,n,P", [(6, 12, 3), (4, 8, 2), (5, 10, 5)])
def test_distributed_products_against_triple_loops(m, n, P):
    rng = np.random.default_rng(m * 31 + n)
    X = rng.standard_normal((m, n))
    X /= np.linalg.norm(X)
    got = oracle.newton_schulz_distributed(X, 5, A_, B_, C_, P)
    want = _loops_ns(X.tolist(), 5, A_, B_, C_)
    assert np.max(np.abs(got - want)) < 1e-12


def test_distributed_one_slice_is_full_and_slices_must_divide():
    rng = np.random.default_rng(3)
    W, G, M = (rng.standard_normal((24, 40)) for _ in range(3))
    a = run(W, G, M, mode="distributed", nb=1)
    b = run(W, G, M)
    for k in ("W", "M", "O"):
        assert np.array_equal(a[k], b[k])
    with pytest.raises(ValueError):
        run(W, G, M, mode="distributed", nb=3)      # 3 does not divide 40


def _mutant_distributed(kind):
    def ns(X, steps, a, b, c, shards):
        X = np.array(X, dtype=np.float64, copy=True)
        n = X.shape[1]
        w = n // shards
        for _ in range(steps):
            if kind == "short_side":          # slices of the rows instead
                h = X.shape[0] // shards
                A = np.zeros((X.shape[0], X.shape[0]))
                for p in range(shards):
                    r = slice(p * h, (p + 1) * h)
                    A[r, r] += X[r] @ X[r].T
            else:
                parts = range(shards - 1) if kind == "drop_slice" else range(shards)
                if kind == "no_reduce":
                    parts = range(1)
                A = sum(X[:, p * w:(p + 1) * w] @ X[:, p * w:(p + 1) * w].T
                        for p in parts)
            B = b * A + c * (A @ A)
            X = a * X + B @ X
        return X
    return ns


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("kind", ["drop_slice", "no_reduce", "short_side"])
def test_pins_reject_planted_distributed_mistakes(kind, monkeypatch):
    monkeypatch.setattr(muon_ref, "newton_schulz_distributed",
                        _mutant_distributed(kind))
    s = np.geomspace(1.0, 0.05, 8)
    U, V, G = svd_matrix(8, 16, s, seed=11)
    out = muon_ref.muon_step(np.zeros((8, 16)), G, np.zeros((8, 16)), lr=0.1,
                             beta=0.0, nesterov=False, ns_steps=5, a=A_,
                             b=B_, c=C_, mode="distributed", nb=4)
    assert not np.max(np.abs(out["O"] - closed_form_O(U, V, s))) <= 1e-3
