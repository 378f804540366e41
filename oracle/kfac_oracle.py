"""Float64 CPU oracle of the Kronecker-factored (K-FAC / AdaFisher-style) optimizer step.

TEST INFRASTRUCTURE.  This module exists to check the CUDA path.  Only the
tests, the package's smoke entry and the benchmark's CPU-baseline leg may
import it; the library never does, and it shares no code with the library.

Every quantity is float64.  Inputs arrive already rounded to their storage
type (fp32 or bf16) and are promoted to float64 here.  Where a step has a
plain definition it is written out as that definition, using NumPy matrix
products as the only library primitive; the Cholesky factorisation and the
triangular solves are the textbook column algorithms, written out.

Sources (page title, section):
  * Osawa et al., "Large-Scale Distributed Second-Order Optimization Using
    Kronecker-Factored Approximate Curvature for Deep Convolutional Neural
    Networks", §3.2: the Fisher of a layer is approximated by the Kronecker
    product of a factor built from the layer's input activations (A) and one
    built from its output gradients (G); its inverse is taken through the
    inverses of the two factors.
  * same page, §3.4: the factors are symmetric, so an N x N factor carries
    N(N+1)/2 distinct entries.
  * same page, §5.4: curvature refreshed less often than every step (stale
    factors); BatchNorm Fisher approximated by its diagonal.
  * "CAFIN: CUDA-accelerated Adaptive Fisher Information Matrix Network
    Optimization via GPU-Native Kernel Fusion", Introduction: AdaFisher keeps
    diagonal Kronecker factors as exponential moving averages; Kernel Fusion
    Strategy: the fused step loads gradient and parameter, updates the EMA of
    the diagonal Fisher blocks, preconditions the gradient, adds momentum and
    weight decay, and writes the parameter in place.

Where the pages leave a step open, this module takes the reading below (each
one is also listed, under the same number, in the repository's design notes;
R9 to R17 there concern inputs and tolerances, not this module's arithmetic):
  R1  EMA starts from zero (F_0 = 0); ``ema_init="first"`` gives F_1 = F_new.
  R2  "decay xi" means the old value keeps weight xi: F <- xi F + (1-xi) F_new.
  R3  factor scale s = 1/M, M = number of rows (batch, or B*H*W for conv).
  R4  inverses are refreshed at step 1 and then every k steps; a step uses the
      inverses of the latest refresh at or before it.
  R5  update: u = P + lambda*W ; m <- mu*m + u ; W <- W - eta*m (m_0 = 0).
  R6  damping: sqrt(gamma) added to the diagonal of each factor.
  R7  diagonal step: P_ij = dW_ij / (g_i a_j + gamma), g and a the EMA diagonals.
  R8  a layer with a bias carries it as the last column of W-hat = [W | b] and
      its activations get a ones column: a-hat = [a | 1].
  R18 a convolution's activation rows are its zero-padded input patches, one
      per (image, output position), columns in weight order (c, i, j); its
      output-gradient rows are the channels at the same positions.
  R19 stale factors: a step recomputes and re-inverts every factor during a
      warm-up of w steps, afterwards A every k_A and G every k_G steps counted
      from the end of the warm-up; a factor skipped on a step keeps both its
      running value and its inverse.
  R20 inverse-free update: K (K K^T in place of (F + sqrt(gamma) I)^{-1}) is
      seeded from the Cholesky refresh (K = L^{-T}) and stepped by
      K <- K (I - (beta/2)(K^T (F + sqrt(gamma) I) K - I)), beta in (0, 2);
      the preconditioner uses K K^T.  The page states only that the update is
      inverse-free and subtracts in the matrix-logarithm space; this first-order
      exponential-map step on K's right factor is the plainest such update.

Parity pins for every function live in tests/test_oracle.py.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np


class NotPositiveDefinite(ArithmeticError):
    """Raised by :func:`cholesky_lower` with the 0-based failing column."""

    def __init__(self, column: int):
        super().__init__(f"leading minor {column + 1} is not positive definite")
        self.column = column


def _f64(x) -> np.ndarray:
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# factors (Osawa et al. §3.2; symmetry §3.4)

def augment_ones(a, has_bias: int) -> np.ndarray:
    """a-hat = [a | 1] when the layer has a bias (reading R8), else a."""
    a = _f64(a)
    if not has_bias:
        return a
    return np.concatenate([a, np.ones((a.shape[0], 1))], axis=1)


def factor(x, has_bias: int = 0, scale: Optional[float] = None) -> np.ndarray:
    """New factor s * x-hat^T x-hat for x of shape [M, d] (rows are samples).

    A is built from input activations with has_bias; G from output gradients
    with has_bias = 0.  The result is symmetrised as (F + F^T)/2 so that it is
    symmetric to the last bit.
    """
    xh = augment_ones(x, has_bias)
    M = xh.shape[0]
    s = 1.0 / M if scale is None else float(scale)
    F = s * (xh.T @ xh)
    return 0.5 * (F + F.T)


def ema(old, new, decay: float) -> np.ndarray:
    """Running factor by exponential moving average (reading R2)."""
    return decay * _f64(old) + (1.0 - decay) * _f64(new)


# ---------------------------------------------------------------------------
# convolution layers (Osawa et al. §3.2, §5.1): a 2-D convolution is a linear
# map applied at every output position, so its A factor is built from the input
# patches, one row per (image, output position), and its G factor from the
# output gradient at the same positions; M = B * H_out * W_out.

def conv_out_size(size: int, kernel: int, stride: int, pad: int, dilation: int) -> int:
    """Output extent of a 2-D convolution along one axis."""
    return (size + 2 * pad - dilation * (kernel - 1) - 1) // stride + 1


def im2col(x, kernel, stride=(1, 1), pad=(0, 0), dilation=(1, 1)) -> np.ndarray:
    """Input patches of a 2-D convolution as rows: x [B, C, H, W] -> [B*Ho*Wo, C*kh*kw].

    Row order (b, oh, ow); column order (c, i, j), the order of a weight
    [o, C, kh, kw] flattened to [o, C*kh*kw].  Entry (row, column) is
    x[b, c, oh*sh - ph + i*dh, ow*sw - pw + j*dw], zero outside the image.
    """
    x = _f64(x)
    B, C, H, W = x.shape
    (kh, kw), (sh, sw), (ph, pw), (dh, dw) = kernel, stride, pad, dilation
    Ho = conv_out_size(H, kh, sh, ph, dh)
    Wo = conv_out_size(W, kw, sw, pw, dw)
    xp = np.zeros((B, C, H + 2 * ph, W + 2 * pw))
    xp[:, :, ph:ph + H, pw:pw + W] = x
    cols = np.empty((B, Ho, Wo, C, kh, kw))
    for i in range(kh):
        for j in range(kw):
            win = xp[:, :, i * dh: i * dh + sh * (Ho - 1) + 1: sh,
                     j * dw: j * dw + sw * (Wo - 1) + 1: sw]          # [B, C, Ho, Wo]
            cols[:, :, :, :, i, j] = win.transpose(0, 2, 3, 1)
    return cols.reshape(B * Ho * Wo, C * kh * kw)


def output_rows(gy) -> np.ndarray:
    """Output gradient [B, o, Ho, Wo] as rows [B*Ho*Wo, o], row order (b, oh, ow)."""
    gy = _f64(gy)
    return gy.transpose(0, 2, 3, 1).reshape(-1, gy.shape[1])


def conv_factors(x, gy, kernel, stride=(1, 1), pad=(0, 0), dilation=(1, 1),
                 has_bias: int = 1, scale: Optional[float] = None):
    """New (A, G) of a 2-D convolution from its input x [B, C, H, W] and output
    gradient gy [B, o, Ho, Wo]: A = s * [P 1]^T [P 1] with P = im2col(x),
    G = s * R^T R with R = output_rows(gy), s = 1/(B*Ho*Wo) unless given."""
    P = im2col(x, kernel, stride, pad, dilation)
    R = output_rows(gy)
    if P.shape[0] != R.shape[0]:
        raise ValueError("input patches and output gradient rows differ")
    return factor(P, has_bias, scale), factor(R, 0, scale)


# ---------------------------------------------------------------------------
# damped inverse (Osawa et al. §3.2: inverse through the factor inverses)

def damped(F, damping: float) -> np.ndarray:
    """F + sqrt(gamma) I (reading R6)."""
    F = _f64(F)
    return F + math.sqrt(damping) * np.eye(F.shape[0])


def cholesky_lower(S) -> np.ndarray:
    """Textbook column-by-column Cholesky: S = L L^T with L lower triangular.

    Column j:  L[j,j] = sqrt(S[j,j] - sum_{k<j} L[j,k]^2),
               L[i,j] = (S[i,j] - sum_{k<j} L[i,k] L[j,k]) / L[j,j]   (i > j).
    Raises NotPositiveDefinite(j) when the pivot is not > 0 (or not finite).
    """
    S = _f64(S)
    n = S.shape[0]
    L = np.zeros_like(S)
    for j in range(n):
        d = S[j, j] - L[j, :j] @ L[j, :j]
        if not (d > 0.0 and math.isfinite(d)):
            raise NotPositiveDefinite(j)
        L[j, j] = math.sqrt(d)
        if j + 1 < n:
            L[j + 1:, j] = (S[j + 1:, j] - L[j + 1:, :j] @ L[j, :j]) / L[j, j]
    return L


def lower_inverse(L) -> np.ndarray:
    """X = L^{-1} by forward substitution on the identity, row by row.

    Row i of L X = I gives X[i, :] = (e_i - sum_{k<i} L[i,k] X[k, :]) / L[i,i];
    X is lower triangular, so only columns <= i are formed.
    """
    L = _f64(L)
    n = L.shape[0]
    X = np.zeros_like(L)
    for i in range(n):
        r = -(L[i, :i] @ X[:i, :i + 1])
        r[i] += 1.0
        X[i, :i + 1] = r / L[i, i]
    return X


def spd_inverse_from_cholesky(L) -> np.ndarray:
    """S^{-1} = L^{-T} L^{-1}: forward substitution on I, then the transpose product."""
    X = lower_inverse(L)
    Sinv = X.T @ X
    return 0.5 * (Sinv + Sinv.T)


def damped_inverse(F, damping: float) -> np.ndarray:
    """(F + sqrt(gamma) I)^{-1} via the textbook Cholesky and substitutions."""
    return spd_inverse_from_cholesky(cholesky_lower(damped(F, damping)))


# ---------------------------------------------------------------------------
# inverse-free factor update ("Structured Inverse-Free Natural Gradient" page,
# abstract: an inverse-free K-FAC update by subtraction in the matrix-logarithm
# space instead of an inversion; reading R20 below)

def ikfac_init(F, damping: float) -> np.ndarray:
    """K = L^{-T} for F + sqrt(gamma) I = L L^T, so that K K^T = (F + sqrt(gamma) I)^{-1}
    exactly (the factor left by a Cholesky refresh)."""
    return lower_inverse(cholesky_lower(damped(F, damping))).T


def ikfac_update(K, F, damping: float, beta: float) -> np.ndarray:
    """One inverse-free step on K, where K K^T stands for (F + sqrt(gamma) I)^{-1}:
    with E = K^T (F + sqrt(gamma) I) K - I (zero when K K^T is the exact inverse),
    K <- K (I - (beta/2) E): the first-order form of K exp(-(beta/2) E), a
    subtraction of (beta/2) E in the logarithm of K's right factor."""
    K = _f64(K)
    n = K.shape[0]
    E = K.T @ damped(F, damping) @ K - np.eye(n)
    return K @ (np.eye(n) - 0.5 * beta * E)


def ikfac_inverse(K) -> np.ndarray:
    """The preconditioning inverse K K^T."""
    K = _f64(K)
    return K @ K.T


# ---------------------------------------------------------------------------
# preconditioning and update

def grad_hat(grad_w, grad_b=None) -> np.ndarray:
    """dW-hat = [dW | db] (reading R8)."""
    gw = _f64(grad_w)
    if grad_b is None:
        return gw
    return np.concatenate([gw, _f64(grad_b).reshape(-1, 1)], axis=1)


def precondition(Ginv, gw_hat, Ainv) -> np.ndarray:
    """Natural-gradient direction P = G_d^{-1} . dW-hat . A_d^{-1} (Osawa et al. §3.2)."""
    return _f64(Ginv) @ _f64(gw_hat) @ _f64(Ainv)


def momentum_update(P, W_hat, m, lr, momentum, weight_decay):
    """u = P + lambda W ; m <- mu m + u ; W <- W - eta m  (reading R5).

    Returns (W_new, m_new).  Follows the CAFIN briefing's fused order: apply
    the preconditioner, then momentum and weight decay, then write W.
    """
    u = _f64(P) + weight_decay * _f64(W_hat)
    m_new = momentum * _f64(m) + u
    W_new = _f64(W_hat) - lr * m_new
    return W_new, m_new


# ---------------------------------------------------------------------------
# diagonal path (CAFIN Introduction / Kernel Fusion Strategy; Osawa et al. §5.4 BN)

def diag_factor(x, has_bias: int = 0, scale: Optional[float] = None) -> np.ndarray:
    """diag(s * x-hat^T x-hat): s * sum_r x[r, j]^2 per column (ones column -> s*M)."""
    xh = augment_ones(x, has_bias)
    M = xh.shape[0]
    s = 1.0 / M if scale is None else float(scale)
    return s * np.sum(xh * xh, axis=0)


def conv_diag_factors(x, gy, kernel, stride=(1, 1), pad=(0, 0), dilation=(1, 1),
                      has_bias: int = 1, scale: Optional[float] = None):
    """New diagonal factors of a 2-D convolution (reading R18): the diagonals of
    conv_factors, s * column sums of squares of the input patches (bias entry
    s*M) and of the output-gradient rows."""
    P = im2col(x, kernel, stride, pad, dilation)
    R = output_rows(gy)
    if P.shape[0] != R.shape[0]:
        raise ValueError("input patches and output gradient rows differ")
    return diag_factor(R, 0, scale), diag_factor(P, has_bias, scale)


def diag_precondition(gw_hat, gs, as_, damping: float) -> np.ndarray:
    """P_ij = dW_ij / (g_i a_j + gamma)  (reading R7)."""
    return _f64(gw_hat) / (np.outer(_f64(gs), _f64(as_)) + damping)


# ---------------------------------------------------------------------------
# stale-factor schedule (Osawa et al. §5.4)

def stale_refresh(t: int, warmup: int, every_a: int, every_g: int):
    """Which factors a step t (1-based) recomputes and re-inverts (reading R19).

    Every step during the first ``warmup`` steps, while the Fisher changes
    fast; after that A every ``every_a`` steps and G every ``every_g`` steps
    (the page observes that A fluctuates less than G, so every_a >= every_g is
    the intended use), counted from the end of the warm-up.  Returns (A, G)."""
    if t <= warmup:
        return True, True
    u = t - warmup
    return u % every_a == 0, u % every_g == 0


# ---------------------------------------------------------------------------
# the whole per-layer step

class LayerState:
    """State of one layer: running factors, inverses, momentum and parameters."""

    def __init__(self, kind: str, d_out: int, d_in: int, has_bias: int, w0, b0=None):
        self.kind, self.o, self.d_in, self.has_bias = kind, d_out, d_in, has_bias
        self.n = d_in + has_bias
        self.W = grad_hat(w0, b0 if has_bias else None).copy()   # [o, n]
        self.m = np.zeros((d_out, self.n))
        self.t = 0
        if kind == "kron":
            self.A = np.zeros((self.n, self.n))
            self.G = np.zeros((d_out, d_out))
            self.Ainv = self.Ginv = None
        else:
            self.gs = np.zeros(d_out)
            self.as_ = np.zeros(self.n)
        self.P = None


class KfacOracle:
    """Per-layer K-FAC / diagonal step, in the order the pages give it.

    ``ema_init``: "zero" (reading R1) or "first" (F_1 = F_new).
    """

    def __init__(self, ema_decay, damping, lr, momentum, weight_decay,
                 invert_every: int = 1, ema_init: str = "zero"):
        self.xi, self.gamma = float(ema_decay), float(damping)
        self.lr, self.mu, self.wd = float(lr), float(momentum), float(weight_decay)
        self.k = int(invert_every)
        self.ema_init = ema_init

    def _blend(self, old, new, t):
        if t == 1 and self.ema_init == "first":
            return _f64(new).copy()
        return ema(old, new, self.xi)

    def step_kron(self, st: LayerState, a, g, grad_w, grad_b=None, scale=None):
        """One K-FAC step; returns the preconditioned gradient P [o, n]."""
        st.t += 1
        t = st.t
        st.A = self._blend(st.A, factor(a, st.has_bias, scale), t)
        st.G = self._blend(st.G, factor(g, 0, scale), t)
        if (t - 1) % self.k == 0:                      # reading R4
            st.Ainv = damped_inverse(st.A, self.gamma)
            st.Ginv = damped_inverse(st.G, self.gamma)
        P = precondition(st.Ginv, grad_hat(grad_w, grad_b if st.has_bias else None), st.Ainv)
        st.W, st.m = momentum_update(P, st.W, st.m, self.lr, self.mu, self.wd)
        st.P = P
        return P

    def step_kron_sched(self, st: LayerState, a, g, grad_w, grad_b=None, update=(True, True),
                        refresh=(True, True), scale=None, shared_a: "LayerState" = None):
        """One K-FAC step with an explicit per-factor schedule (Osawa et al. §5.4:
        stale factors).  update = (A, G): fold the new factor into the running
        one this step; refresh = (A, G): recompute that factor's damped inverse.
        A factor not updated keeps its running value, one not refreshed keeps
        the inverse of its latest refresh.  ``shared_a``: this layer has no A of
        its own and preconditions with that layer's current A inverse (layers
        fed the same input build the same A).  The EMA-first option counts each
        factor's own updates.  Returns P [o, n]."""
        st.t += 1
        if shared_a is None:
            if update[0]:
                st.ta = getattr(st, "ta", 0) + 1
                st.A = self._blend(st.A, factor(a, st.has_bias, scale), st.ta)
            if refresh[0]:
                st.Ainv = damped_inverse(st.A, self.gamma)
            Ainv = st.Ainv
        else:
            Ainv = shared_a.Ainv
        if update[1]:
            st.tg = getattr(st, "tg", 0) + 1
            st.G = self._blend(st.G, factor(g, 0, scale), st.tg)
        if refresh[1]:
            st.Ginv = damped_inverse(st.G, self.gamma)
        if Ainv is None or st.Ginv is None:
            raise ValueError("precondition before the first refresh of both factors")
        P = precondition(st.Ginv, grad_hat(grad_w, grad_b if st.has_bias else None), Ainv)
        st.W, st.m = momentum_update(P, st.W, st.m, self.lr, self.mu, self.wd)
        st.P = P
        return P

    def step_diag(self, st: LayerState, g_new, a_new, grad_w, grad_b=None):
        """One diagonal-Fisher step given the new diagonal factors; returns P."""
        st.t += 1
        st.gs = self._blend(st.gs, g_new, st.t)
        st.as_ = self._blend(st.as_, a_new, st.t)
        P = diag_precondition(grad_hat(grad_w, grad_b if st.has_bias else None),
                              st.gs, st.as_, self.gamma)
        st.W, st.m = momentum_update(P, st.W, st.m, self.lr, self.mu, self.wd)
        st.P = P
        return P
