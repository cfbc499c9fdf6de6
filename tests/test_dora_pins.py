"""Pins of the oracle's DoRA forward and backward (column-norm magnitude/direction split).

Against closed forms, invariants of the definition and finite differences, not
against a second copy of the same formulas."""
import numpy as np
import pytest

from oracle import lora_oracle as O


def problem(seed, m=24, k=20, n=18, r=4):
    rng = np.random.default_rng(seed)
    X = rng.standard_normal((m, k))
    W = rng.standard_normal((k, n)) / np.sqrt(k)
    A = rng.uniform(-1, 1, (k, r)) / np.sqrt(k)
    B = rng.standard_normal((r, n)) * 0.3
    mag = rng.uniform(0.5, 2.0, n)
    dY = rng.standard_normal((m, n))
    return X, W, A, B, mag, dY


def test_identity_at_initialisation():
    # DoRA starts from mag = ||W||_col and B = 0: the layer is X W exactly
    X, W, A, B, _, _ = problem(0)
    B0 = np.zeros_like(B)
    mag = np.linalg.norm(W, axis=0)
    Y, _, _, g, _ = O.dora_forward(X, W, A, B0, mag, 2.0, 0.0, 1)
    np.testing.assert_allclose(g, np.ones_like(g), rtol=1e-14)
    np.testing.assert_allclose(Y, X @ W, rtol=1e-12, atol=1e-12)


def test_merged_weight_has_the_magnitudes_as_column_norms():
    X, W, A, B, mag, _ = problem(1)
    alpha = 1.5
    Y, _, _, g, _ = O.dora_forward(X, W, A, B, mag, alpha, 0.0, 3)
    W_merged = g * (W + alpha * A @ B)                       # p = 0: Y = X W'
    np.testing.assert_allclose(Y, X @ W_merged, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(np.linalg.norm(W_merged, axis=0), mag, rtol=1e-12)


def test_each_output_column_only_keeps_its_direction():
    # scaling column j of W and of B by c_j > 0 scales column j of W + alpha A B by c_j: Y must not change;
    # a norm taken over the wrong axis would mix the columns and fail this
    X, W, A, B, mag, _ = problem(2)
    c = np.random.default_rng(5).uniform(0.2, 5.0, W.shape[1])
    Y1 = O.dora_forward(X, W, A, B, mag, 2.0, 0.0, 7)[0]
    Y2 = O.dora_forward(X, W * c, A, B * c, mag, 2.0, 0.0, 7)[0]
    np.testing.assert_allclose(Y1, Y2, rtol=1e-11, atol=1e-12)


def test_factored_norm_identity():
    # "Scaling DoRA": ||W + s BA||^2 = ||W||^2 + 2 s <W, BA> + s^2 ||BA||^2 with the cross term from
    # U = W^T A and the last term from the Gram matrix G = A^T A (this layer's orientation)
    _, W, A, B, _, _ = problem(3, k=64, n=40, r=8)
    s = 2.0
    U = W.T @ A
    G = A.T @ A
    factored = (W * W).sum(0) + 2 * s * (B.T * U).sum(1) + s * s * ((B.T @ G) * B.T).sum(1)
    np.testing.assert_allclose(np.sqrt(factored), O.dora_column_norms(W, A, B, s), rtol=1e-12)


def test_dmag_is_the_exact_derivative():
    # Y is linear in mag, so central differences are exact up to rounding
    X, W, A, B, mag, dY = problem(4)
    alpha, p, seed = 2.0, 0.25, 11
    _, _, _, dmag = O.dora_backward(dY, X, W, A, B, mag, alpha, p, seed)
    h = 1e-3
    for j in range(mag.size):
        e = np.zeros_like(mag)
        e[j] = h
        fp = (dY * O.dora_forward(X, W, A, B, mag + e, alpha, p, seed)[0]).sum()
        fm = (dY * O.dora_forward(X, W, A, B, mag - e, alpha, p, seed)[0]).sum()
        assert abs((fp - fm) / (2 * h) - dmag[j]) < 1e-9 * max(1.0, abs(dmag[j]))


@pytest.mark.parametrize("which", ["X", "A", "B"])
def test_gradients_with_the_norm_held_constant(which):
    # with g frozen at its value, L = sum(dY * g * Z) is linear in X and in A, B separately -> exact FD
    X, W, A, B, mag, dY = problem(5)
    alpha, p, seed = 2.0, 0.2, 13
    dX, dA, dB, _ = O.dora_backward(dY, X, W, A, B, mag, alpha, p, seed)
    g = mag / O.dora_column_norms(W, A, B, alpha)

    def loss(X_, A_, B_):
        Z = O.lora_forward(X_, W, A_, B_, alpha, p, seed)[0]
        return (dY * g * Z).sum()

    base = {"X": X, "A": A, "B": B}
    grad = {"X": dX, "A": dA, "B": dB}[which]
    rng = np.random.default_rng(9)
    h = 1e-3
    for _ in range(20):
        idx = tuple(rng.integers(0, s) for s in base[which].shape)
        args_p = {key: v.copy() for key, v in base.items()}
        args_m = {key: v.copy() for key, v in base.items()}
        args_p[which][idx] += h
        args_m[which][idx] -= h
        fd = (loss(args_p["X"], args_p["A"], args_p["B"]) - loss(args_m["X"], args_m["A"], args_m["B"])) / (2 * h)
        assert abs(fd - grad[idx]) < 1e-8 * max(1.0, abs(grad[idx]))


def test_backward_reduces_to_lora_when_g_is_one():
    # mag equal to the column norms of the adapted weight gives g = 1: plain LoRA gradients, and
    # dmag_j = sum_t dY Z / norm_j
    X, W, A, B, _, dY = problem(6)
    alpha, p, seed = 2.0, 0.1, 17
    mag = O.dora_column_norms(W, A, B, alpha)
    dX, dA, dB, dmag = O.dora_backward(dY, X, W, A, B, mag, alpha, p, seed)
    lX, lA, lB, _ = O.lora_backward(dY, X, W, A, B, alpha, p, seed)
    np.testing.assert_allclose(dX, lX, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dA, lA, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dB, lB, rtol=1e-12, atol=1e-12)
