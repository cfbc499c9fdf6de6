"""Pins for the fp64 oracle: each test ties it to something other than itself.

- the Philox rounds against numpy's own Philox-4x64 bit generator (a library
  routine) and the key increments against their closed forms;
- the keep mask against binomial statistics and independence;
- the forward against brute-force loops in the special cases that reduce to
  a plain product (alpha = 0, p = 0 merged weight W + alpha A B);
- the gradients against central finite differences (exact here: Y is linear
  in each of X, A and B once the mask is fixed);
- the multi-adapter routing against per-row brute force.

A last group plants mistakes in the oracle and checks that these pins fail.
"""
import math

import numpy as np
import pytest

from oracle import lora_oracle as O


# ---------------------------------------------------------------------------
# helpers (independent of the oracle's arithmetic)
# ---------------------------------------------------------------------------

def brute_matmul(a, b):
    """Triple loop over Python floats: a textbook product for tiny shapes."""
    m, k = a.shape
    k2, n = b.shape
    assert k == k2
    out = np.zeros((m, n))
    for i in range(m):
        for j in range(n):
            s = 0.0
            for t in range(k):
                s += float(a[i, t]) * float(b[t, j])
            out[i, j] = s
    return out


def rand(rng, *shape, scale=1.0):
    return rng.standard_normal(shape) * scale


def small_problem(seed=0, m=6, k=16, n=8, r=3):
    rng = np.random.default_rng(seed)
    return dict(X=rand(rng, m, k), W=rand(rng, k, n, scale=0.25), A=rand(rng, k, r, scale=0.3),
                B=rand(rng, r, n, scale=0.3), dY=rand(rng, m, n))


# ---------------------------------------------------------------------------
# Philox
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("counter,key", [((0, 0, 0, 0), (0, 0)), ((5, 7, 0, 0), (11, 13)),
                                         ((2**64 - 2, 3, 9, 2**63), (2**64 - 1, 12345)),
                                         ((123456789, 987654321, 55, 66), (0xDEADBEEF, 0xFEEDFACE))])
def test_philox_rounds_match_numpy_philox4x64(counter, key):
    """numpy's Philox bit generator is Philox-4x64-10; it advances the counter by one before each block."""
    bg = np.random.Philox(counter=np.array(counter, dtype=np.uint64), key=np.array(key, dtype=np.uint64))
    ref = [int(v) for v in bg.random_raw(4)]
    c = list(counter)
    c[0] = (c[0] + 1) % 2**64
    if c[0] == 0:
        c[1] = (c[1] + 1) % 2**64
    assert list(O.philox4_scalar(c, key, width=64)) == ref


def test_philox_weyl_increments_closed_form():
    """Key increments: floor(2^w (sqrt5-1)/2) and floor(2^w (sqrt3-1))."""
    for w in (32, 64):
        phi_frac = (math.isqrt(5 << (2 * w)) - (1 << w)) // 2
        sqrt3_m1 = math.isqrt(3 << (2 * w)) - (1 << w)
        assert O.PHILOX[w]["W0"] == phi_frac
        assert O.PHILOX[w]["W1"] == sqrt3_m1


def test_philox_vectorised_equals_scalar():
    rng = np.random.default_rng(1)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
    for key in [(0, 0), (0xFFFFFFFF, 1), (123, 456789)]:
        vec = O.philox4x32(ctr[:, 0], ctr[:, 1], ctr[:, 2], ctr[:, 3], *key)
        for i in range(ctr.shape[0]):
            assert tuple(int(v[i]) for v in vec) == O.philox4_scalar(ctr[i], key, width=32)


def test_philox_is_a_bijection_on_small_domain():
    """Distinct counters under one key give distinct outputs (a Philox round is invertible)."""
    c0 = np.arange(4096, dtype=np.uint32)
    out = O.philox4x32(c0, 7, 0, 0, 99, 100)
    packed = {tuple(int(v[i]) for v in out) for i in range(c0.size)}
    assert len(packed) == c0.size


# ---------------------------------------------------------------------------
# dropout mask
# ---------------------------------------------------------------------------

def test_threshold_values():
    assert O.dropout_threshold(0.0) == 0
    assert O.dropout_threshold(0.1) == 6554
    assert O.dropout_threshold(0.5) == 32768
    assert O.dropout_threshold(0.05) == 3277
    for bad in (1.0, 1.5, -0.1):
        with pytest.raises(ValueError):
            O.dropout_threshold(bad)


def test_p0_keeps_everything():
    D = O.keep_mask(1234, np.arange(64), 256, O.dropout_threshold(0.0))
    assert D.all()


@pytest.mark.parametrize("p", [0.05, 0.1, 0.3, 0.5, 0.9])
def test_keep_fraction_is_binomial(p):
    T = O.dropout_threshold(p)
    D = O.keep_mask(7, np.arange(512), 1024, T)
    keep = 1.0 - T / 65536.0
    n = D.size
    sigma = math.sqrt(keep * (1 - keep) / n)
    assert abs(D.mean() - keep) < 6 * sigma


def test_mask_decisions_are_uncorrelated():
    """Neighbouring features (same and next 8-group), neighbouring rows and other seeds are independent."""
    T = O.dropout_threshold(0.5)
    D = O.keep_mask(3, np.arange(1024), 512, T).astype(np.float64)
    D2 = O.keep_mask(4, np.arange(1024), 512, T).astype(np.float64)

    def corr(a, b):
        a = a.ravel() - a.mean()
        b = b.ravel() - b.mean()
        return float((a * b).sum() / math.sqrt((a * a).sum() * (b * b).sum()))

    bound = 6.0 / math.sqrt(D[:, :-1].size)
    for lag in range(1, 9):  # lags inside one Philox call and across calls
        assert abs(corr(D[:, :-lag], D[:, lag:])) < bound
    assert abs(corr(D[:-1], D[1:])) < bound
    assert abs(corr(D, D2)) < bound


def test_mask_uses_global_row_index():
    full = O.keep_mask(11, np.arange(300), 64, O.dropout_threshold(0.2))
    part = O.keep_mask(11, [257, 3, 128], 64, O.dropout_threshold(0.2))
    assert (part == full[[257, 3, 128]]).all()


def test_seed_high_word_matters():
    a = O.keep_mask(5, np.arange(32), 64, 32768)
    b = O.keep_mask(5 + (1 << 32), np.arange(32), 64, 32768)
    assert (a != b).any()


def test_mask_bits_packing_roundtrip():
    D = O.keep_mask(2, np.arange(8), 64, O.dropout_threshold(0.3))
    bits = O.pack_mask_bits(D)
    unpacked = ((bits[:, :, None] >> np.arange(8)) & 1).reshape(8, 64).astype(bool)
    assert (unpacked == D).all()


def test_inverted_dropout_is_unbiased_and_has_binomial_variance():
    """Over many seeds: E[S] = X A (the q scale undoes the drop), Var[S] = sum_j X^2 A^2 q^2 keep (1-keep)."""
    rng = np.random.default_rng(5)
    X = rng.standard_normal((4, 32))
    A = rng.standard_normal((32, 2))
    p = 0.3
    keep = 1.0 - O.dropout_threshold(p) / 65536.0
    q = O.dropout_scale(p)
    samples = np.stack([O.lora_forward(X, np.zeros((32, 1)), A, np.zeros((2, 1)), 1.0, p, s)[1]
                        for s in range(3000)])
    mean = samples.mean(axis=0)
    var_theory = (X ** 2) @ (A ** 2) * q * q * keep * (1 - keep)
    mean_theory = X @ A * q * keep
    # standard error of the mean is sqrt(var/N)
    assert np.all(np.abs(mean - mean_theory) < 6 * np.sqrt(var_theory / samples.shape[0]))
    np.testing.assert_allclose(samples.var(axis=0), var_theory, rtol=0.2)
    np.testing.assert_allclose(q * keep, 1.0, atol=1e-4)


# ---------------------------------------------------------------------------
# forward: reductions to a plain product
# ---------------------------------------------------------------------------

def test_alpha_zero_is_the_frozen_layer():
    P = small_problem()
    Y, _, _ = O.lora_forward(P["X"], P["W"], P["A"], P["B"], 0.0, 0.3, 9)
    np.testing.assert_allclose(Y, brute_matmul(P["X"], P["W"]), rtol=1e-12, atol=1e-12)
    dX, dA, dB, _ = O.lora_backward(P["dY"], P["X"], P["W"], P["A"], P["B"], 0.0, 0.3, 9)
    np.testing.assert_allclose(dX, brute_matmul(P["dY"], P["W"].T), rtol=1e-12, atol=1e-12)
    assert not dB.any()
    assert not dA.any()


def test_zero_B_leaves_the_frozen_output():
    P = small_problem(1)
    Y, _, _ = O.lora_forward(P["X"], P["W"], P["A"], np.zeros_like(P["B"]), 2.0, 0.1, 0)
    np.testing.assert_allclose(Y, brute_matmul(P["X"], P["W"]), rtol=1e-12, atol=1e-12)


def test_merged_weight_without_dropout():
    """p = 0: X W + alpha (X A) B = X (W + alpha A B), with A B formed first."""
    P = small_problem(2)
    alpha = 1.75
    merged = P["W"] + alpha * brute_matmul(P["A"], P["B"])
    Y, S, D = O.lora_forward(P["X"], P["W"], P["A"], P["B"], alpha, 0.0, 42)
    assert D.all()
    np.testing.assert_allclose(Y, brute_matmul(P["X"], merged), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(S, brute_matmul(P["X"], P["A"]), rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# backward: finite differences
# ---------------------------------------------------------------------------

def fd_check(forward, backward, P, alpha, p, seed):
    """Central differences of L = sum(dY * Y) w.r.t. every entry of X, A, B (h = 1 is exact: L is linear in each)."""
    def loss(X, A, B):
        Y = forward(X, P["W"], A, B, alpha, p, seed)[0]
        return float((P["dY"] * Y).sum())

    dX, dA, dB = backward(P["dY"], P["X"], P["W"], P["A"], P["B"], alpha, p, seed)[:3]
    for name, grad in (("X", dX), ("A", dA), ("B", dB)):
        base = {k: P[k].copy() for k in ("X", "A", "B")}
        fd = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            plus = {k: v.copy() for k, v in base.items()}
            minus = {k: v.copy() for k, v in base.items()}
            plus[name][idx] += 1.0
            minus[name][idx] -= 1.0
            fd[idx] = (loss(plus["X"], plus["A"], plus["B"]) - loss(minus["X"], minus["A"], minus["B"])) / 2.0
        scale = max(1.0, float(np.abs(fd).max()))
        if not np.allclose(grad, fd, rtol=0, atol=1e-9 * scale):
            return name
    return None


@pytest.mark.parametrize("alpha,p,seed", [(1.5, 0.3, 0), (2.0, 0.0, 1), (0.5, 0.6, 2**40 + 3)])
def test_gradients_match_finite_differences(alpha, p, seed):
    P = small_problem(3, m=5, k=16, n=6, r=3)
    assert fd_check(O.lora_forward, O.lora_backward, P, alpha, p, seed) is None


def test_dS_is_the_gradient_of_S():
    """dS = alpha dY B^T is the derivative of sum(dY * Y) w.r.t. S (Y depends on S through alpha S B)."""
    P = small_problem(4)
    alpha = 1.25
    dS = O.lora_backward(P["dY"], P["X"], P["W"], P["A"], P["B"], alpha, 0.2, 3)[3]
    S0 = np.zeros((P["X"].shape[0], P["A"].shape[1]))
    fd = np.zeros_like(S0)
    for idx in np.ndindex(*S0.shape):
        e = np.zeros_like(S0)
        e[idx] = 1.0
        fd[idx] = float((P["dY"] * (alpha * brute_matmul(e, P["B"]))).sum())
    np.testing.assert_allclose(dS, fd, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------------------
# multi-adapter routing
# ---------------------------------------------------------------------------

def multi_problem(seed=0, m=640, k=32, n=24, ranks=(4, 8, 2, 6)):
    rng = np.random.default_rng(seed)
    adapters = [dict(A=rand(rng, k, r, scale=0.3), B=rand(rng, r, n, scale=0.3), alpha=a, p=p)
                for r, a, p in zip(ranks, (1.0, 2.0, 2.0, 4.0), (0.0, 0.1, 0.3, 0.05))]
    X = rand(rng, m, k)
    W = rand(rng, k, n, scale=0.2)
    dY = rand(rng, m, n)
    # tile 1 uncovered, adapter 2 unused, last segment ends mid-tile at m
    segments = [(0, 128, 1), (256, 256, 0), (512, m - 512, 3)]
    return X, W, dY, adapters, segments


def test_multi_with_one_adapter_equals_single():
    X, W, dY, adapters, _ = multi_problem(1, m=300)
    ad = adapters[2]
    seg = [(0, 300, 0)]
    Ym, Sm, _ = O.multi_lora_forward(X, W, [ad], seg, 77)
    Ys, Ss, _ = O.lora_forward(X, W, ad["A"], ad["B"], ad["alpha"], ad["p"], 77)
    np.testing.assert_array_equal(Ym, Ys)
    np.testing.assert_array_equal(Sm[0], Ss)
    dXm, dAm, dBm, _, _ = O.multi_lora_backward(dY, X, W, [ad], seg, 77)
    dXs, dAs, dBs, _ = O.lora_backward(dY, X, W, ad["A"], ad["B"], ad["alpha"], ad["p"], 77)
    np.testing.assert_array_equal(dXm, dXs)
    np.testing.assert_array_equal(dAm[0], dAs)
    np.testing.assert_array_equal(dBm[0], dBs)


def test_multi_matches_per_row_brute_force():
    """Every row processed alone with its own adapter gives the tile-routed result; gradients sum per adapter."""
    X, W, dY, adapters, segments = multi_problem(2)
    m = X.shape[0]
    seed = 2024
    Y, _, owner = O.multi_lora_forward(X, W, adapters, segments, seed)
    dX, dA, dB, _, _ = O.multi_lora_backward(dY, X, W, adapters, segments, seed)
    expect_owner = np.full(m, -1)
    for s, r, a in segments:
        expect_owner[s:s + r] = a
    assert (owner == expect_owner).all()
    dA_ref = [np.zeros_like(a["A"]) for a in adapters]
    dB_ref = [np.zeros_like(a["B"]) for a in adapters]
    for t in range(m):
        a = expect_owner[t]
        if a < 0:
            np.testing.assert_allclose(Y[t], X[t] @ W, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(dX[t], dY[t] @ W.T, rtol=1e-12, atol=1e-12)
            continue
        ad = adapters[a]
        Yt = O.lora_forward(X[t:t + 1], W, ad["A"], ad["B"], ad["alpha"], ad["p"], seed, rows=[t])[0]
        dXt, dAt, dBt, _ = O.lora_backward(dY[t:t + 1], X[t:t + 1], W, ad["A"], ad["B"], ad["alpha"], ad["p"],
                                           seed, rows=[t])
        np.testing.assert_allclose(Y[t], Yt[0], rtol=1e-11, atol=1e-11)
        np.testing.assert_allclose(dX[t], dXt[0], rtol=1e-11, atol=1e-11)
        dA_ref[a] += dAt
        dB_ref[a] += dBt
    for i in range(len(adapters)):
        np.testing.assert_allclose(dA[i], dA_ref[i], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dB[i], dB_ref[i], rtol=1e-10, atol=1e-10)
    assert not dA[2].any() and not dB[2].any()


def test_multi_backward_on_row_subsets_adds_up():
    """Restricting the packed backward to rows: dX rows agree with the full pass and each dA_i / dB_i
    is the sum of its parts over a partition of the rows (sums over rows, by the definition)."""
    X, W, dY, adapters, segments = multi_problem(3)
    m = X.shape[0]
    seed = 99
    dX, dA, dB, _, _ = O.multi_lora_backward(dY, X, W, adapters, segments, seed)
    rng = np.random.default_rng(5)
    perm = rng.permutation(m)
    parts = [np.sort(perm[: m // 3]), np.sort(perm[m // 3:])]
    dA_sum = [np.zeros_like(a["A"]) for a in adapters]
    dB_sum = [np.zeros_like(a["B"]) for a in adapters]
    for rows in parts:
        dXp, dAp, dBp, _, owner = O.multi_lora_backward(dY[rows], X[rows], W, adapters, segments, seed, rows=rows)
        np.testing.assert_allclose(dXp, dX[rows], rtol=1e-12, atol=1e-12)
        for i in range(len(adapters)):
            dA_sum[i] += dAp[i]
            dB_sum[i] += dBp[i]
    for i in range(len(adapters)):
        np.testing.assert_allclose(dA_sum[i], dA[i], rtol=1e-10, atol=1e-10)
        np.testing.assert_allclose(dB_sum[i], dB[i], rtol=1e-10, atol=1e-10)


def multi_fd_mismatch(backward, seed=5):
    """Central differences of L = sum(dY * Y) through the packed multi-adapter forward, w.r.t. a sample of X
    entries (rows of both adapters and of the uncovered tail) and every entry of each A_i and B_i.  L is linear
    in each of them, so h = 1 is exact.  Returns the first gradient that disagrees with `backward`, or None."""
    rng = np.random.default_rng(seed)
    k, n = 8, 6
    adapters = [dict(A=rand(rng, k, r, scale=0.4), B=rand(rng, r, n, scale=0.4), alpha=a, p=pp)
                for r, a, pp in ((2, 1.5, 0.3), (3, 2.0, 0.0), (2, 0.5, 0.5))]
    m = 128 + 128 + 7
    segments = [(0, 128, 1), (128, 128, 0)]          # rows 256..262 have no adapter; adapter 2 owns no rows
    X, W, dY = rand(rng, m, k), rand(rng, k, n, scale=0.3), rand(rng, m, n)
    seed_mask = 2**36 + 11

    def loss(Xv, ads):
        return float((dY * O.multi_lora_forward(Xv, W, ads, segments, seed_mask)[0]).sum())

    dX, dA, dB = backward(dY, X, W, adapters, segments, seed_mask)[:3]

    def central(bump):
        plus, minus = bump(1.0), bump(-1.0)
        return (loss(*plus) - loss(*minus)) / 2.0

    for t, j in [(0, 0), (5, 7), (127, 3), (128, 1), (200, 6), (255, 2), (256, 4), (262, 0)]:
        def bump(h, t=t, j=j):
            Xh = X.copy()
            Xh[t, j] += h
            return Xh, adapters
        if abs(central(bump) - dX[t, j]) > 1e-9 * max(1.0, abs(dX[t, j])):
            return "dX"
    for i in range(len(adapters)):
        for name, grad in (("A", dA[i]), ("B", dB[i])):
            for idx in np.ndindex(*grad.shape):
                def bump(h, i=i, name=name, idx=idx):
                    ads = [dict(a) for a in adapters]
                    mat = ads[i][name].copy()
                    mat[idx] += h
                    ads[i][name] = mat
                    return X, ads
                if abs(central(bump) - grad[idx]) > 1e-9 * max(1.0, abs(grad[idx])):
                    return f"d{name}{i}"
    return None


def test_multi_gradients_match_finite_differences():
    """The packed backward against central differences of the packed forward itself, independent of the
    single-adapter backward: each dA_i / dB_i collects exactly its own rows, with its own alpha and p."""
    assert multi_fd_mismatch(O.multi_lora_backward) is None


def test_multi_finite_differences_catch_misrouted_gradients():
    """Planted in the oracle's output: adapter 0's one tile counted twice in its dB, or its dA scaled by
    adapter 1's alpha in place of its own.  The finite-difference pin must reject both."""
    def tile_twice_in_dB(*args):
        dX, dA, dB, dS, owner = O.multi_lora_backward(*args)
        dB = [2.0 * dB[0]] + list(dB[1:])
        return dX, dA, dB, dS, owner

    def wrong_alpha(*args):
        dX, dA, dB, dS, owner = O.multi_lora_backward(*args)
        dA = [dA[0] * (2.0 / 1.5)] + list(dA[1:])
        return dX, dA, dB, dS, owner

    assert multi_fd_mismatch(tile_twice_in_dB) is not None
    assert multi_fd_mismatch(wrong_alpha) is not None


def test_tile_table_brute_force():
    segments = [(0, 128, 1), (256, 256, 0), (512, 128, 3)]
    tiles = O.tile_adapters(segments, 700, 4)
    expect = []
    for t in range(-(-700 // 128)):
        row = t * 128
        a = -1
        for s, r, ad in segments:
            if s <= row < s + r:
                a = ad
        expect.append(a)
    assert tiles.tolist() == expect


@pytest.mark.parametrize("segments", [[(64, 128, 0)], [(0, 100, 0), (128, 128, 0)], [(0, 256, 0), (128, 128, 1)],
                                      [(0, 128, 5)], [(0, 1024, 0)]])
def test_routing_rejects_bad_tables(segments):
    with pytest.raises(ValueError):
        O.row_adapters(segments, 512, 2)


# ---------------------------------------------------------------------------
# planted mistakes: the pins above must catch each of these
# ---------------------------------------------------------------------------

def _mutated_backward(kind):
    def backward(dY, X, W, A, B, alpha, p, seed, rows=None):
        if rows is None:
            rows = np.arange(X.shape[0])
        D = O.keep_mask(seed, rows, X.shape[1], O.dropout_threshold(p))
        q = O.dropout_scale(p)
        X_hat = X * D * q
        S = X_hat @ A
        dS = alpha * (dY @ B.T)
        dB = alpha * (S.T @ dY)
        dA = X_hat.T @ dS
        dXb = (D * q) * (dS @ A.T)
        if kind == "dX_without_branch":
            dXb = 0 * dXb
        elif kind == "dB_without_alpha":
            dB = S.T @ dY
        elif kind == "dA_without_mask":
            dA = X.T @ dS
        elif kind == "dX_branch_without_mask":
            dXb = q * (dS @ A.T)
        elif kind == "dS_sign":
            dA = -dA
        return dY @ W.T + dXb, dA, dB, dS
    return backward


@pytest.mark.parametrize("kind", ["dX_without_branch", "dB_without_alpha", "dA_without_mask",
                                  "dX_branch_without_mask", "dS_sign"])
def test_finite_differences_catch_planted_gradient_mistakes(kind):
    P = small_problem(3, m=5, k=16, n=6, r=3)
    assert fd_check(O.lora_forward, _mutated_backward(kind), P, 1.5, 0.3, 0) is not None


def test_merged_weight_catches_transposed_branch():
    """Planting (X A) B -> (X A) B^T-shaped mistakes: using A B^T style contraction changes the result."""
    P = small_problem(2, n=3, r=3)
    alpha = 1.75
    merged = P["W"] + alpha * brute_matmul(P["A"], P["B"])
    wrong = P["X"] @ P["W"] + alpha * (P["X"] @ P["A"]) @ P["B"].T
    assert not np.allclose(wrong, brute_matmul(P["X"], merged))


def test_variance_pin_catches_missing_mask_and_missing_scale():
    rng = np.random.default_rng(5)
    X = rng.standard_normal((4, 32))
    A = rng.standard_normal((32, 2))
    p = 0.3
    keep = 1.0 - O.dropout_threshold(p) / 65536.0
    q = O.dropout_scale(p)
    # no mask applied: zero variance across seeds, far below the binomial variance
    var_theory = (X ** 2) @ (A ** 2) * q * q * keep * (1 - keep)
    assert np.all(var_theory > 0.0)
    # mask without the 1/(1-p) scale: the mean drifts by the factor keep
    no_scale = np.stack([(X * O.keep_mask(s, np.arange(4), 32, O.dropout_threshold(p))) @ A for s in range(3000)])
    assert np.any(np.abs(no_scale.mean(axis=0) - X @ A) > 6 * np.sqrt(var_theory / 3000))
