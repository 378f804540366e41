"""Pins for the float64 oracle against facts fixed by the pages and by the mathematics.

None of these re-type the oracle's own formula: each check uses brute force on
tiny inputs, a closed form, an invariant, or an independent library routine
(LAPACK through NumPy/SciPy) for a step the oracle writes out by hand.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import oracle as O
import workloads as W

RNG = np.random.default_rng(1234)


# ---------------------------------------------------------------- factors

def _brute_factor(x, has_bias, scale):
    """Sum over rows of outer products, element by element, in exact rationals."""
    M, d = len(x), len(x[0])
    n = d + has_bias
    col = lambda r, j: Fraction(x[r][j]) if j < d else Fraction(1)
    s = Fraction(scale) if scale is not None else Fraction(1, M)
    return [[s * sum(col(r, i) * col(r, j) for r in range(M)) for j in range(n)]
            for i in range(n)]


@pytest.mark.parametrize("M,d,has_bias", [(1, 1, 0), (3, 2, 1), (5, 4, 0), (8, 4, 1), (7, 3, 1)])
def test_factor_brute_force(M, d, has_bias):
    x = RNG.integers(-5, 6, size=(M, d)).astype(np.float64) / 4.0
    F = O.factor(x, has_bias)
    ref = _brute_factor(x.tolist(), has_bias, None)
    for i in range(d + has_bias):
        for j in range(d + has_bias):
            assert abs(F[i, j] - float(ref[i][j])) <= 1e-15 * max(1.0, abs(float(ref[i][j])))


def test_factor_custom_scale_and_shape():
    x = RNG.standard_normal((6, 3))
    F = O.factor(x, 1, scale=0.25)
    assert F.shape == (4, 4)
    ref = _brute_factor(x.tolist(), 1, 0.25)
    assert np.allclose(F, np.array(ref, dtype=float), rtol=1e-14, atol=1e-14)


def test_factor_symmetric_psd_and_bias_entries():
    M, d = 200, 37
    a = np.maximum(RNG.standard_normal((M, d)), 0)
    A = O.factor(a, 1)
    assert np.array_equal(A, A.T)                       # symmetric to the last bit
    ev = np.linalg.eigvalsh(A)
    assert ev.min() >= -A.shape[0] * np.finfo(float).eps * np.abs(ev).max()
    assert A[d, d] == 1.0                               # s * M with s = 1/M
    assert np.allclose(A[:d, d], a.mean(axis=0), rtol=1e-14, atol=1e-16)
    assert np.allclose(np.diag(A)[:d], (a * a).mean(axis=0), rtol=1e-13)


def test_factor_upper_triangle_count():
    # Osawa et al. §3.4: an N x N symmetric factor has N(N+1)/2 distinct entries
    A = O.factor(RNG.standard_normal((30, 11)), 1)
    iu = np.triu_indices(12)
    assert len(iu[0]) == 12 * 13 // 2
    rebuilt = np.zeros_like(A)
    rebuilt[iu] = A[iu]
    rebuilt = rebuilt + np.triu(rebuilt, 1).T
    assert np.array_equal(rebuilt, A)


# ---------------------------------------------------------------- EMA

@pytest.mark.parametrize("xi", [0.0, 0.5, 0.95])
def test_ema_constant_input_closed_form(xi):
    C = RNG.standard_normal((5, 5))
    F0 = RNG.standard_normal((5, 5))
    F = F0.copy()
    for t in range(1, 40):
        F = O.ema(F, C, xi)
        closed = C + xi ** t * (F0 - C)
        assert np.allclose(F, closed, rtol=1e-12, atol=1e-12)
    if xi == 0.0:
        assert np.array_equal(O.ema(F0, C, 0.0), C)


def test_ema_zero_start_converges():
    C = O.factor(RNG.standard_normal((50, 6)), 1)
    F = np.zeros_like(C)
    for _ in range(400):
        F = O.ema(F, C, 0.95)
    assert np.allclose(F, C, rtol=1e-8, atol=1e-8)


# ---------------------------------------------------------------- Cholesky / inverse

def test_cholesky_hand_examples():
    L = O.cholesky_lower([[4.0, 2.0], [2.0, 2.0]])
    assert np.array_equal(L, np.array([[2.0, 0.0], [1.0, 1.0]]))
    L = O.cholesky_lower([[9.0, 3.0, 6.0], [3.0, 5.0, 6.0], [6.0, 6.0, 21.0]])
    assert np.allclose(L, [[3, 0, 0], [1, 2, 0], [2, 2, 3.605551275463989]], atol=1e-15)


@pytest.mark.parametrize("n", [1, 7, 64, 200])
def test_cholesky_matches_lapack(n):
    X = RNG.standard_normal((n + 5, n))
    S = X.T @ X / (n + 5) + 0.1 * np.eye(n)
    L = O.cholesky_lower(S)
    assert np.allclose(L, np.linalg.cholesky(S), rtol=1e-12, atol=1e-13)
    assert np.abs(L @ L.T - S).max() <= 1e-13 * np.abs(S).max()
    assert np.array_equal(L, np.tril(L))


def test_cholesky_not_pd_column():
    with pytest.raises(O.NotPositiveDefinite) as e:
        O.cholesky_lower(np.diag([1.0, 2.0, -1.0, 3.0]))
    assert e.value.column == 2
    with pytest.raises(O.NotPositiveDefinite) as e:
        O.cholesky_lower([[1.0, 2.0], [2.0, 1.0]])
    assert e.value.column == 1
    with pytest.raises(O.NotPositiveDefinite) as e:
        O.cholesky_lower([[float("nan")]])
    assert e.value.column == 0


@pytest.mark.parametrize("n", [1, 5, 70])
def test_lower_inverse_vs_solve_triangular(n):
    L = np.tril(RNG.standard_normal((n, n))) + 3 * np.eye(n)
    X = O.lower_inverse(L)
    ref = scipy.linalg.solve_triangular(L, np.eye(n), lower=True)
    assert np.allclose(X, ref, rtol=1e-12, atol=1e-13)
    assert np.allclose(L @ X, np.eye(n), atol=1e-13)


@pytest.mark.parametrize("n", [3, 40, 257])
def test_damped_inverse_vs_lapack(n):
    A = O.factor(np.maximum(RNG.standard_normal((n // 2 + 3, n - 1)), 0), 1)
    gamma = 1e-3
    Ainv = O.damped_inverse(A, gamma)
    Ad = A + math.sqrt(gamma) * np.eye(n)
    ref = np.linalg.inv(Ad)
    assert np.linalg.norm(Ainv - ref) <= 1e-10 * np.linalg.norm(ref)
    assert np.abs(Ad @ Ainv - np.eye(n)).max() <= 1e-10
    assert np.array_equal(Ainv, Ainv.T)


def test_damped_inverse_of_zero_factor():
    n = 9
    Ainv = O.damped_inverse(np.zeros((n, n)), 1e-3)
    assert np.allclose(Ainv, np.eye(n) / math.sqrt(1e-3), rtol=1e-15, atol=0)


# ---------------------------------------------------------------- preconditioning

@pytest.mark.parametrize("o,d,has_bias", [(1, 1, 1), (3, 4, 1), (6, 8, 1), (5, 9, 0), (4, 2, 0)])
def test_precondition_kronecker_identity(o, d, has_bias):
    """vec_r(G P A) = (G kron A^T) vec_r(P): solve with the materialised Kronecker matrix."""
    M, gamma = 12, 1e-2
    a = RNG.standard_normal((M, d))
    g = RNG.standard_normal((M, o)) * 0.1
    A, G = O.factor(a, has_bias), O.factor(g, 0)
    gw = RNG.standard_normal((o, d))
    gb = RNG.standard_normal(o) if has_bias else None
    gh = O.grad_hat(gw, gb)
    P = O.precondition(O.damped_inverse(G, gamma), gh, O.damped_inverse(A, gamma))
    Ad = A + math.sqrt(gamma) * np.eye(d + has_bias)
    Gd = G + math.sqrt(gamma) * np.eye(o)
    K = np.kron(Gd, Ad.T)
    vecP = np.linalg.solve(K, gh.reshape(-1))
    assert np.allclose(P.reshape(-1), vecP, rtol=1e-10, atol=1e-12)


def test_full_path_reduces_to_diag_path_on_diagonal_inputs():
    """Rows +-c_k e_k make a-hat^T a-hat exactly diagonal, ones column included.

    With diagonal factors the full path divides by (g_i+sqrt(gamma))(a_j+sqrt(gamma));
    the diagonal path divides by (g_i a_j + gamma).  Feeding the diagonal path
    g' = g + sqrt(gamma), a' = a + sqrt(gamma), gamma' = 0 must give the same P.
    """
    d, o, gamma = 5, 3, 1e-3
    ca, cg = RNG.uniform(0.5, 2.0, d), RNG.uniform(0.01, 0.1, o)
    a = np.concatenate([np.diag(ca), -np.diag(ca)])             # [2d, d]
    g = np.concatenate([np.diag(cg), -np.diag(cg)])             # [2o, o]
    # pad both to the same row count with zero rows (zero rows add nothing)
    M = 2 * max(d, o)
    a = np.vstack([a, np.zeros((M - len(a), d))])
    g = np.vstack([g, np.zeros((M - len(g), o))])
    A, G = O.factor(a, 1), O.factor(g, 0)
    assert np.count_nonzero(A - np.diag(np.diag(A))) == 0
    assert np.count_nonzero(G - np.diag(np.diag(G))) == 0
    assert np.allclose(np.diag(A), O.diag_factor(a, 1), rtol=1e-15)
    assert np.allclose(np.diag(G), O.diag_factor(g, 0), rtol=1e-15)
    gh = O.grad_hat(RNG.standard_normal((o, d)), RNG.standard_normal(o))
    P_full = O.precondition(O.damped_inverse(G, gamma), gh, O.damped_inverse(A, gamma))
    sg = math.sqrt(gamma)
    P_diag = O.diag_precondition(gh, np.diag(G) + sg, np.diag(A) + sg, 0.0)
    assert np.allclose(P_full, P_diag, rtol=1e-12, atol=0)


# ---------------------------------------------------------------- diagonal step

def test_diag_factor_brute_force():
    x = RNG.integers(-3, 4, size=(6, 4)).astype(float)
    v = O.diag_factor(x, 1)
    for j in range(4):
        assert math.isclose(v[j], sum(float(x[r, j]) ** 2 for r in range(6)) / 6, rel_tol=4e-16)
    assert v[4] == 1.0


def test_diag_step_elementwise_closed_form():
    o, n = 4, 3
    gw = RNG.standard_normal((o, n))
    W = RNG.standard_normal((o, n))
    m = RNG.standard_normal((o, n))
    gs, as_ = RNG.uniform(0, 1, o), RNG.uniform(0, 1, n)
    gamma, eta, mu, lam = 1e-3, 0.1, 0.9, 5e-4
    P = O.diag_precondition(gw, gs, as_, gamma)
    Wn, mn = O.momentum_update(P, W, m, eta, mu, lam)
    for i in range(o):
        for j in range(n):
            p = gw[i, j] / (gs[i] * as_[j] + gamma)
            mm = mu * m[i, j] + (p + lam * W[i, j])
            assert math.isclose(P[i, j], p, rel_tol=1e-15)
            assert math.isclose(mn[i, j], mm, rel_tol=1e-14)
            assert math.isclose(Wn[i, j], W[i, j] - eta * mm, rel_tol=1e-14, abs_tol=1e-15)


def test_update_special_cases():
    o, n = 3, 5
    gw, W = RNG.standard_normal((o, n)), RNG.standard_normal((o, n))
    gs, as_ = RNG.uniform(0.1, 1, o), RNG.uniform(0.1, 1, n)
    P = O.diag_precondition(gw, gs, as_, 1e-3)
    Wn, _ = O.momentum_update(P, W, np.zeros((o, n)), 0.0, 0.9, 5e-4)
    assert np.array_equal(Wn, W)                                    # eta = 0
    Wn, mn = O.momentum_update(P, W, np.zeros((o, n)), 0.1, 0.0, 0.0)
    assert np.allclose(Wn, W - 0.1 * gw / (np.outer(gs, as_) + 1e-3), rtol=1e-14)


# ---------------------------------------------------------------- whole step

def _c1_run(steps=10, invert_every=1, ema_init="zero"):
    cfg = W.get_config("c1")
    hp = cfg.hp
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay,
                       invert_every, ema_init)
    L = cfg.layers[0]
    w0, b0 = W.initial_params(cfg, 0)
    st = O.LayerState("kron", L.d_out, L.d_in, L.has_bias, w0, b0)
    hist = []
    for t in range(1, steps + 1):
        x = W.layer_inputs(cfg, 0, t)
        orc.step_kron(st, x["a"], x["g"], x["grad_w"], x["grad_b"])
        hist.append((st.A.copy(), st.Ainv.copy(), st.W.copy()))
    return cfg, st, hist


def test_refresh_schedule():
    _, _, hist = _c1_run(steps=8, invert_every=3)
    refreshed = [t for t in range(1, 8) if not np.array_equal(hist[t][1], hist[t - 1][1])]
    assert [t + 1 for t in refreshed] == [4, 7]                 # steps 1, 4, 7 refresh


def test_ema_init_first_and_zero():
    cfg = W.get_config("c1")
    x = W.layer_inputs(cfg, 0, 1)
    _, st, _ = _c1_run(steps=1, ema_init="first")
    assert np.allclose(st.A, O.factor(x["a"], 1), rtol=1e-15)
    _, st, _ = _c1_run(steps=1, ema_init="zero")
    assert np.allclose(st.A, 0.05 * O.factor(x["a"], 1), rtol=1e-14)


def test_c1_golden_trajectory():
    """Regression record of the oracle's c1 run (written by tests/golden/make_golden.py)."""
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "c1_oracle_trajectory.npz")
    ref = np.load(path)
    _, st, hist = _c1_run()
    for t in range(10):
        assert np.allclose(hist[t][2], ref["W"][t], rtol=1e-12, atol=1e-15)
    assert np.allclose(st.A, ref["A"], rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- convolution layers

CONV_GEOMS = [  # (B, C, H, W, kh, kw, sh, sw, ph, pw, dh, dw)
    (2, 3, 5, 6, 3, 3, 1, 1, 1, 1, 1, 1),
    (1, 2, 7, 5, 3, 2, 2, 1, 1, 0, 1, 1),
    (2, 1, 9, 8, 3, 3, 2, 2, 2, 1, 2, 2),
    (3, 4, 4, 4, 1, 1, 1, 1, 0, 0, 1, 1),
    (1, 2, 11, 11, 7, 7, 2, 2, 3, 3, 1, 1),
]


@pytest.mark.parametrize("geom", CONV_GEOMS)
def test_im2col_matches_torch_unfold(geom):
    """The patch rows equal torch.nn.functional.unfold's columns (an independent
    library routine), transposed to one row per (image, output position)."""
    torch = pytest.importorskip("torch")
    B, C, H, Wd, kh, kw, sh, sw, ph, pw, dh, dw = geom
    x = RNG.standard_normal((B, C, H, Wd))
    got = O.im2col(x, (kh, kw), (sh, sw), (ph, pw), (dh, dw))
    u = torch.nn.functional.unfold(torch.from_numpy(x), (kh, kw), dilation=(dh, dw),
                                   padding=(ph, pw), stride=(sh, sw))      # [B, C*kh*kw, L]
    ref = u.transpose(1, 2).reshape(-1, C * kh * kw).numpy()
    assert got.shape == ref.shape
    np.testing.assert_array_equal(got, ref)


def test_im2col_brute_force():
    """Every entry by its definition, with explicit bounds checks, on a tiny case."""
    B, C, H, Wd, kh, kw, sh, sw, ph, pw, dh, dw = 2, 2, 5, 4, 3, 2, 2, 1, 1, 1, 1, 2
    x = RNG.integers(-9, 10, size=(B, C, H, Wd)).astype(np.float64)
    Ho = (H + 2 * ph - dh * (kh - 1) - 1) // sh + 1
    Wo = (Wd + 2 * pw - dw * (kw - 1) - 1) // sw + 1
    got = O.im2col(x, (kh, kw), (sh, sw), (ph, pw), (dh, dw))
    assert got.shape == (B * Ho * Wo, C * kh * kw)
    for b in range(B):
        for oh in range(Ho):
            for ow in range(Wo):
                row = (b * Ho + oh) * Wo + ow
                for c in range(C):
                    for i in range(kh):
                        for j in range(kw):
                            y, xx = oh * sh - ph + i * dh, ow * sw - pw + j * dw
                            v = x[b, c, y, xx] if 0 <= y < H and 0 <= xx < Wd else 0.0
                            assert got[row, (c * kh + i) * kw + j] == v


def test_conv_1x1_patches_are_the_pixels():
    """A 1x1 convolution with unit stride and no padding sees each pixel's channel
    vector: its patch rows are the input laid out as output rows."""
    x = RNG.standard_normal((3, 5, 4, 6))
    np.testing.assert_array_equal(O.im2col(x, (1, 1)), O.output_rows(x))


@pytest.mark.parametrize("H,Wd", [(4, 4), (5, 7), (1, 3)])
def test_conv_factor_of_constant_image_closed_form(H, Wd):
    """On an all-ones image with a 3x3, pad-1, stride-1 kernel, taps with row
    offsets i, i' (0..2) both fall inside the image at the output rows oh with
    max(0, 1 - min(i, i')) <= oh <= min(H - 1, H - max(i, i')), and likewise for
    columns; A's entry is that count over H*W, the bias column the single-tap count."""
    C = 2
    x = np.ones((1, C, H, Wd))
    gy = np.zeros((1, 3, H, Wd))
    A, _ = O.conv_factors(x, gy, (3, 3), (1, 1), (1, 1), (1, 1), has_bias=1)
    M = H * Wd
    n = C * 9 + 1
    assert A.shape == (n, n)

    def rows(ext, a, b):
        lo, hi = max(0, 1 - min(a, b)), min(ext - 1, ext - max(a, b))
        return max(0, hi - lo + 1)

    for p in range(C * 9):
        i, j = (p % 9) // 3, p % 3
        assert A[p, n - 1] == pytest.approx(rows(H, i, i) * rows(Wd, j, j) / M, rel=1e-15)
        for q in range(C * 9):
            i2, j2 = (q % 9) // 3, q % 3
            want = rows(H, i, i2) * rows(Wd, j, j2) / M
            assert A[p, q] == pytest.approx(want, rel=1e-15, abs=1e-300)
    assert A[n - 1, n - 1] == 1.0


def test_conv_G_is_channel_covariance_over_positions():
    """G sums g g^T over every (image, position): the same as contracting the
    NCHW output gradient over batch and both spatial axes."""
    gy = RNG.standard_normal((3, 4, 5, 2))
    x = RNG.standard_normal((3, 2, 5, 2))
    _, G = O.conv_factors(x, gy, (1, 1))
    ref = np.einsum("bchw,bdhw->cd", gy, gy) / (3 * 5 * 2)
    np.testing.assert_allclose(G, ref, rtol=1e-14, atol=0)


# ---------------------------------------------------------------- stale-factor schedule

def test_stale_refresh_hand_example():
    """warm-up 3, A every 4, G every 2: steps 1-3 both; then G at 5, 7, 9; A at 7, 11."""
    got = [O.stale_refresh(t, 3, 4, 2) for t in range(1, 12)]
    want = [(True, True)] * 3 + [(False, False), (False, True), (False, False), (True, True),
                                 (False, False), (False, True), (False, False), (True, True)]
    assert got == want


@pytest.mark.parametrize("T,w,ka,kg", [(1000, 500, 20, 5), (37, 0, 7, 3), (10, 10, 3, 3)])
def test_stale_refresh_counts_closed_form(T, w, ka, kg):
    """Refreshes in T steps: w + floor((T - w)/k) for each factor."""
    flags = [O.stale_refresh(t, w, ka, kg) for t in range(1, T + 1)]
    assert sum(f[0] for f in flags) == w + (T - w) // ka
    assert sum(f[1] for f in flags) == w + (T - w) // kg


def _sched_layer(seed, o=5, d=4, bias=1):
    rng = np.random.default_rng(seed)
    w0 = rng.standard_normal((o, d))
    b0 = rng.standard_normal(o)
    return O.LayerState("kron", o, d, bias, w0, b0), rng


def test_schedule_all_true_reduces_to_plain_step():
    """update = refresh = (True, True) every step is the plain step with k = 1."""
    orc = O.KfacOracle(0.9, 1e-2, 0.1, 0.9, 1e-3, invert_every=1)
    s1, rng = _sched_layer(3)
    s2, _ = _sched_layer(3)
    for _ in range(4):
        a, g = rng.standard_normal((20, 4)), rng.standard_normal((20, 5))
        gw, gb = rng.standard_normal((5, 4)), rng.standard_normal(5)
        P1 = orc.step_kron(s1, a, g, gw, gb)
        P2 = orc.step_kron_sched(s2, a, g, gw, gb)
        np.testing.assert_array_equal(P1, P2)
        np.testing.assert_array_equal(s1.W, s2.W)


def test_schedule_skipped_factor_keeps_value_and_inverse():
    """A skipped update leaves the running factor unchanged; a skipped refresh
    leaves the inverse unchanged, so P moves only through dW-hat and G."""
    orc = O.KfacOracle(0.9, 1e-2, 0.1, 0.9, 1e-3)
    st, rng = _sched_layer(5)
    a, g = rng.standard_normal((20, 4)), rng.standard_normal((20, 5))
    gw, gb = rng.standard_normal((5, 4)), rng.standard_normal(5)
    orc.step_kron_sched(st, a, g, gw, gb)
    A1, Ai1, G1 = st.A.copy(), st.Ainv.copy(), st.G.copy()
    a2, g2 = 3 * rng.standard_normal((20, 4)), rng.standard_normal((20, 5))
    P = orc.step_kron_sched(st, a2, g2, gw, gb, update=(False, True), refresh=(False, True))
    np.testing.assert_array_equal(st.A, A1)
    np.testing.assert_array_equal(st.Ainv, Ai1)
    assert not np.array_equal(st.G, G1)
    # P = Ginv dW Ainv with the new G inverse and the old A inverse, by LAPACK
    Gd = st.G + math.sqrt(1e-2) * np.eye(5)
    Ad = A1 + math.sqrt(1e-2) * np.eye(5)
    ref = np.linalg.solve(Gd, np.linalg.solve(Ad.T, O.grad_hat(gw, gb).T).T)
    np.testing.assert_allclose(P, ref, rtol=1e-10, atol=1e-12)


def test_shared_a_uses_the_source_inverse():
    """A layer sharing another's A preconditions with the source's A inverse."""
    orc = O.KfacOracle(0.9, 1e-2, 0.1, 0.9, 1e-3)
    src, rng = _sched_layer(8)
    tied, _ = _sched_layer(9)
    a, g, g2 = (rng.standard_normal((20, 4)), rng.standard_normal((20, 5)),
                rng.standard_normal((20, 5)))
    gw, gb = rng.standard_normal((5, 4)), rng.standard_normal(5)
    orc.step_kron_sched(src, a, g, gw, gb)
    P = orc.step_kron_sched(tied, None, g2, gw, gb, shared_a=src)
    Gd = O.factor(g2, 0) * 0.1 + math.sqrt(1e-2) * np.eye(5)      # zero-start EMA, xi = 0.9
    Ad = O.factor(a, 1) * 0.1 + math.sqrt(1e-2) * np.eye(5)
    ref = np.linalg.solve(Gd, np.linalg.solve(Ad.T, O.grad_hat(gw, gb).T).T)
    np.testing.assert_allclose(P, ref, rtol=1e-10, atol=1e-12)


# ---------------------------------------------------------------- inverse-free update

def _spd(n, seed, cond=50.0):
    rng = np.random.default_rng(seed)
    Q, _ = np.linalg.qr(rng.standard_normal((n, n)))
    return (Q * np.linspace(1.0, cond, n)) @ Q.T * 1e-2


def test_ikfac_init_is_the_exact_inverse_factor():
    F = _spd(7, 1)
    K = O.ikfac_init(F, 1e-2)
    Fd = F + 0.1 * np.eye(7)
    np.testing.assert_allclose(K @ K.T, np.linalg.inv(Fd), rtol=1e-10, atol=1e-12)
    assert np.allclose(np.tril(K, -1), 0.0)          # L^{-T} is upper triangular


def test_ikfac_fixed_point():
    """At K K^T = (F + sqrt(gamma) I)^{-1} the residual vanishes and K stays."""
    F = _spd(9, 2)
    K = O.ikfac_init(F, 1e-2)
    np.testing.assert_allclose(O.ikfac_update(K, F, 1e-2, 0.7), K, rtol=0, atol=1e-12)


def test_ikfac_scalar_closed_form():
    """n = 1: k <- k (1 - (beta/2)(f_d k^2 - 1)), in exact rationals."""
    k, f, gam, beta = Fraction(3, 4), Fraction(5, 2), Fraction(1, 16), Fraction(1, 2)
    fd = f + Fraction(1, 4)                              # sqrt(1/16)
    want = k * (1 - beta / 2 * (fd * k * k - 1))
    got = O.ikfac_update(np.array([[float(k)]]), np.array([[float(f)]]), float(gam), float(beta))
    assert got[0, 0] == pytest.approx(float(want), rel=1e-15)


def test_ikfac_is_first_order_exponential_map():
    """One step equals K expm(-(beta/2) E) up to O(beta^2) (scipy's expm): the
    error falls by about 4x when beta halves."""
    F = _spd(6, 3)
    K0 = O.ikfac_init(_spd(6, 4), 1e-2)                  # the inverse factor of another F
    E = K0.T @ (F + 0.1 * np.eye(6)) @ K0 - np.eye(6)
    errs = []
    for beta in (0.02, 0.01, 0.005):
        exact = K0 @ scipy.linalg.expm(-0.5 * beta * E)
        errs.append(np.linalg.norm(O.ikfac_update(K0, F, 1e-2, beta) - exact))
    assert 3.5 < errs[0] / errs[1] < 4.5 and 3.5 < errs[1] / errs[2] < 4.5


@pytest.mark.parametrize("beta", [0.5, 1.0, 1.5])
def test_ikfac_iteration_converges_to_the_lapack_inverse(beta):
    """Repeated steps with a fixed F drive K K^T to (F + sqrt(gamma) I)^{-1}
    (np.linalg.inv), from the inverse factor of a nearby F."""
    F1 = _spd(8, 5)
    F2 = F1 + 0.2 * _spd(8, 6)
    K = O.ikfac_init(F1, 1e-2)
    for _ in range(60):
        K = O.ikfac_update(K, F2, 1e-2, beta)
    np.testing.assert_allclose(O.ikfac_inverse(K), np.linalg.inv(F2 + 0.1 * np.eye(8)),
                               rtol=1e-9, atol=1e-9)


@pytest.mark.parametrize("geom", CONV_GEOMS)
def test_conv_diag_factors_are_the_diagonals_of_the_conv_factors(geom):
    """Column sums of squares equal the diagonals of the full factors (a second
    route: the matrix product and its diagonal)."""
    B, C, H, Wd, kh, kw, sh, sw, ph, pw, dh, dw = geom
    x = RNG.standard_normal((B, C, H, Wd))
    Ho = O.conv_out_size(H, kh, sh, ph, dh)
    Wo = O.conv_out_size(Wd, kw, sw, pw, dw)
    gy = RNG.standard_normal((B, 5, Ho, Wo))
    gn, an = O.conv_diag_factors(x, gy, (kh, kw), (sh, sw), (ph, pw), (dh, dw), 1)
    A, G = O.conv_factors(x, gy, (kh, kw), (sh, sw), (ph, pw), (dh, dw), 1)
    np.testing.assert_allclose(an, np.diag(A), rtol=1e-13)
    np.testing.assert_allclose(gn, np.diag(G), rtol=1e-13)
    assert an[-1] == pytest.approx(1.0)                # s * M for the ones column


def test_conv_diag_factors_of_constant_image_closed_form():
    """All-ones image, 3x3 kernel, pad 1, stride 1: tap (i, j) sees the image at
    (H - |i-1|)(W - |j-1|) of the H*W positions."""
    H, Wd = 5, 7
    x = np.ones((2, 3, H, Wd))
    gy = np.zeros((2, 4, H, Wd))
    _, an = O.conv_diag_factors(x, gy, (3, 3), (1, 1), (1, 1), (1, 1), 1)
    for c in range(3):
        for i in range(3):
            for j in range(3):
                want = (H - abs(i - 1)) * (Wd - abs(j - 1)) / (H * Wd)
                assert an[(c * 3 + i) * 3 + j] == pytest.approx(want, rel=1e-15)


# ---------------------------------------------------------------- property checks (hypothesis)

def _hyp():
    return pytest.importorskip("hypothesis")


def test_property_im2col_matches_unfold_on_random_geometries():
    hyp = _hyp()
    torch = pytest.importorskip("torch")
    st = hyp.strategies

    @hyp.settings(max_examples=60, deadline=None)
    @hyp.given(B=st.integers(1, 2), C=st.integers(1, 3), H=st.integers(1, 9), Wd=st.integers(1, 9),
               kh=st.integers(1, 4), kw=st.integers(1, 4), sh=st.integers(1, 3), sw=st.integers(1, 3),
               ph=st.integers(0, 2), pw=st.integers(0, 2), dh=st.integers(1, 2), dw=st.integers(1, 2))
    def check(B, C, H, Wd, kh, kw, sh, sw, ph, pw, dh, dw):
        hyp.assume(O.conv_out_size(H, kh, sh, ph, dh) >= 1 and O.conv_out_size(Wd, kw, sw, pw, dw) >= 1)
        x = np.random.default_rng(B * 7 + C).standard_normal((B, C, H, Wd))
        got = O.im2col(x, (kh, kw), (sh, sw), (ph, pw), (dh, dw))
        u = torch.nn.functional.unfold(torch.from_numpy(x), (kh, kw), dilation=(dh, dw),
                                       padding=(ph, pw), stride=(sh, sw))
        np.testing.assert_array_equal(got, u.transpose(1, 2).reshape(-1, C * kh * kw).numpy())

    check()


def test_property_damped_inverse_and_factor_invariants():
    """For random inputs: the factor is symmetric PSD with the bias entries s*M and
    column means; the damped inverse times F + sqrt(gamma) I is the identity."""
    hyp = _hyp()
    st = hyp.strategies

    @hyp.settings(max_examples=40, deadline=None)
    @hyp.given(M=st.integers(1, 40), d=st.integers(1, 12), seed=st.integers(0, 10**6),
               gamma=st.sampled_from([1e-4, 1e-3, 1e-1]))
    def check(M, d, seed, gamma):
        a = np.random.default_rng(seed).standard_normal((M, d))
        F = O.factor(a, 1)
        assert np.array_equal(F, F.T)
        assert np.linalg.eigvalsh(F).min() >= -1e-12 * max(1.0, np.abs(F).max())
        assert F[d, d] == pytest.approx(1.0)
        np.testing.assert_allclose(F[:d, d], a.mean(axis=0), rtol=1e-12, atol=1e-14)
        Fi = O.damped_inverse(F, gamma)
        np.testing.assert_allclose(Fi @ (F + math.sqrt(gamma) * np.eye(d + 1)), np.eye(d + 1),
                                   atol=1e-8 * np.linalg.cond(F + math.sqrt(gamma) * np.eye(d + 1)))

    check()


# ------------------------------------------------- the diagonal step as a whole

def _diag_step_rational(st, g_new, a_new, gw_hat, xi, gamma, eta, mu, lam, first):
    """One diagonal step in exact rationals, in the order the CAFIN page's Kernel
    Fusion Strategy gives: EMA of the diagonal factors first, then the gradient
    divided by the *updated* factors, then weight decay and momentum, then the
    in-place parameter write.  st = (gs, as, W, m) as lists of Fractions."""
    gs, as_, Wt, m = st
    if first:
        gs = list(g_new)
        as_ = list(a_new)
    else:
        gs = [xi * o + (1 - xi) * v for o, v in zip(gs, g_new)]
        as_ = [xi * o + (1 - xi) * v for o, v in zip(as_, a_new)]
    P = [[gw_hat[i][j] / (gs[i] * as_[j] + gamma) for j in range(len(as_))]
         for i in range(len(gs))]
    m = [[mu * m[i][j] + P[i][j] + lam * Wt[i][j] for j in range(len(as_))]
         for i in range(len(gs))]
    Wt = [[Wt[i][j] - eta * m[i][j] for j in range(len(as_))] for i in range(len(gs))]
    return (gs, as_, Wt, m), P


@pytest.mark.parametrize("ema_init", ["zero", "first"])
def test_step_diag_two_steps_exact_rationals(ema_init):
    """KfacOracle.step_diag over two steps of a 2 x (1 + bias) layer against a
    hand-worked case in exact rationals.  All inputs are small rationals, so the
    float64 oracle agrees to a few ulps.  The order of the fused operations is
    pinned too: the two plausible slips (preconditioning with the factors from
    before the EMA; the EMA-first option applied at the wrong step) end far from
    the exact parameters."""
    F = Fraction
    xi, gamma, eta, mu, lam = F(1, 2), F(1, 8), F(1, 4), F(1, 2), F(1, 4)
    W0 = [[F(1), F(2)], [F(3), F(-1)]]                 # [W | b], o = 2, d_in = 1
    steps = [([F(2), F(3)], [F(1), F(4)], [[F(1)], [F(2)]], [F(3), F(-4)]),
             ([F(1), F(1, 2)], [F(2), F(1)], [[F(-1)], [F(1, 2)]], [F(1), F(2)])]
    orc = O.KfacOracle(float(xi), float(gamma), float(eta), float(mu), float(lam), 1,
                       ema_init=ema_init)
    st = O.LayerState("diag", 2, 1, 1, np.array([[1.0], [3.0]]), np.array([2.0, -1.0]))
    exact = ([F(0)] * 2, [F(0)] * 2, W0, [[F(0)] * 2 for _ in range(2)])
    slip_first = exact          # EMA-first applied at step 2 instead of step 1
    for t, (gn, an, gw, gb) in enumerate(steps, start=1):
        gw_hat = [[gw[i][0], gb[i]] for i in range(2)]
        P = orc.step_diag(st, np.array([float(v) for v in gn]), np.array([float(v) for v in an]),
                          np.array([[float(v[0])] for v in gw]), np.array([float(v) for v in gb]))
        first = ema_init == "first" and t == 1
        exact, Pe = _diag_step_rational(exact, gn, an, gw_hat, xi, gamma, eta, mu, lam, first)
        slip_first, _ = _diag_step_rational(slip_first, gn, an, gw_hat, xi, gamma, eta, mu, lam,
                                            ema_init == "first" and t == 2)
        for i in range(2):
            assert st.gs[i] == pytest.approx(float(exact[0][i]), rel=1e-15, abs=0)
            assert st.as_[i] == pytest.approx(float(exact[1][i]), rel=1e-15, abs=0)
            for j in range(2):
                assert P[i, j] == pytest.approx(float(Pe[i][j]), rel=1e-14, abs=0)
                assert st.m[i, j] == pytest.approx(float(exact[3][i][j]), rel=1e-14, abs=1e-15)
                assert st.W[i, j] == pytest.approx(float(exact[2][i][j]), rel=1e-14, abs=1e-15)
    far = lambda A, B: max(abs(float(A[i][j] - B[i][j])) for i in range(2) for j in range(2))
    Wpre = _two_steps_preconditioning_with_old_factors(steps, W0, xi, gamma, eta, mu, lam,
                                                       ema_init == "first")
    assert far(Wpre, exact[2]) > 1e-2
    if ema_init == "first":
        assert far(slip_first[2], exact[2]) > 1e-2


def _two_steps_preconditioning_with_old_factors(steps, W0, xi, gamma, eta, mu, lam, first):
    """The slip 'precondition with the factors from before the EMA', two steps."""
    F = Fraction
    gs, as_, Wt, m = [F(0)] * 2, [F(0)] * 2, [r[:] for r in W0], [[F(0)] * 2 for _ in range(2)]
    for t, (gn, an, gw, gb) in enumerate(steps, start=1):
        gw_hat = [[gw[i][0], gb[i]] for i in range(2)]
        P = [[gw_hat[i][j] / (gs[i] * as_[j] + gamma) for j in range(2)] for i in range(2)]
        if first and t == 1:
            gs, as_ = list(gn), list(an)
        else:
            gs = [xi * o + (1 - xi) * v for o, v in zip(gs, gn)]
            as_ = [xi * o + (1 - xi) * v for o, v in zip(as_, an)]
        m = [[mu * m[i][j] + P[i][j] + lam * Wt[i][j] for j in range(2)] for i in range(2)]
        Wt = [[Wt[i][j] - eta * m[i][j] for j in range(2)] for i in range(2)]
    return Wt
