"""The inverse-free refresh on the GPU against the float64 oracle.

Reading R20 (the "Structured Inverse-Free Natural Gradient" page gives only the
idea: an inverse-free K-FAC update by subtraction in the matrix-logarithm
space): K, with K K^T standing for (F + sqrt(gamma) I)^{-1}, is seeded by the
Cholesky refresh (K = L^{-T}) and stepped by K <- K (I - (beta/2)(K^T F_d K - I)).

Tolerances (relative Frobenius).  Each step is four 3xTF32 products (~1e-6
relative each) on operands rounded to TF32 halves (~2.4e-7), so T steps
accumulate about 4e-6 T: the inverses K K^T after 5 steps are held to 5e-5;
the preconditioned update W to 1e-4, as for the Cholesky path.  With the
products on bf16 tensor cores (KFAC_IKFAC_BF16; the page: stable in low
precision) the inverses and the preconditioned gradients are held to the bf16
path's 2e-2 against the float64 iteration.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_helpers import to_dev, to_np, rel_fro

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import second_order_optimizer_gb300 as K  # noqa: E402

HP = dict(ema_decay=0.9, damping=1e-2, lr=1e-2, momentum=0.9, weight_decay=5e-4)
RNG = np.random.default_rng(31)
GAMMA = HP["damping"]


def _draw(M, d, o, act="relu"):
    a = RNG.standard_normal((M, d))
    if act == "relu":
        a = np.maximum(a, 0)
    a = a.astype(np.float32)
    g = (RNG.standard_normal((M, o)) * 1e-2).astype(np.float32)
    gw = (RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)
    gb = (RNG.standard_normal(o) * 1e-3).astype(np.float32)
    return a, g, gw, gb


def test_seed_is_a_fixed_point():
    """Right after a Cholesky refresh K K^T is the inverse: one step leaves it."""
    M, d, o = 700, 299, 130
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32)], max_rows=M, ikfac=1, **HP)
    a, g, _, _ = _draw(M, d, o)
    h.update_factors(0, to_dev(a), to_dev(g))
    h.invert(0)
    A = to_np(h.state(0, K.KFAC_STATE_A))
    ref = np.linalg.inv(A + np.sqrt(GAMMA) * np.eye(d + 1))
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_AINV)), ref) <= 1e-5
    h.ikfac_update(0, beta=1.0)
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_AINV)), ref) <= 1e-5
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("beta", [0.5, 1.0])
def test_inverse_free_steps_match_oracle(beta):
    """Step 1: factors and a Cholesky refresh (seeds K).  Steps 2-6: new factors,
    one inverse-free step of every K, preconditioning with K K^T."""
    shapes = [(900, 1024, 1024), (600, 299, 130), (300, 64, 17)]   # (M, d_in, o)
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32) for _, d, o in shapes],
               max_rows=max(M for M, _, _ in shapes), ikfac=1, **HP)
    orc = O.KfacOracle(HP["ema_decay"], HP["damping"], HP["lr"], HP["momentum"],
                       HP["weight_decay"])
    idx = list(range(len(shapes)))
    st, pw, pb, KA, KG = [], [], [], [None] * 3, [None] * 3
    for M, d, o in shapes:
        w0 = (RNG.standard_normal((o, d)) * 0.1).astype(np.float32)
        b0 = (RNG.standard_normal(o) * 0.1).astype(np.float32)
        st.append(O.LayerState("kron", o, d, 1, w0, b0))
        pw.append(to_dev(w0))
        pb.append(to_dev(b0))
    for t in range(1, 7):
        ins = [_draw(M, d, o) for M, d, o in shapes]
        h.update_factors_batched(idx, [to_dev(x[0]) for x in ins], [to_dev(x[1]) for x in ins])
        if t == 1:
            h.invert(-1)
        else:
            h.ikfac_update(-1, beta=beta)
        h.precondition_batched(idx, [to_dev(x[2]) for x in ins], [to_dev(x[3]) for x in ins],
                               None, None, pw, pb)
        for i, x in enumerate(ins):
            s = st[i]
            s.A = O.ema(s.A, O.factor(x[0], 1), orc.xi)
            s.G = O.ema(s.G, O.factor(x[1], 0), orc.xi)
            if t == 1:
                KA[i], KG[i] = O.ikfac_init(s.A, GAMMA), O.ikfac_init(s.G, GAMMA)
            else:
                KA[i] = O.ikfac_update(KA[i], s.A, GAMMA, beta)
                KG[i] = O.ikfac_update(KG[i], s.G, GAMMA, beta)
            s.Ainv, s.Ginv = O.ikfac_inverse(KA[i]), O.ikfac_inverse(KG[i])
            P = O.precondition(s.Ginv, O.grad_hat(x[2], x[3]), s.Ainv)
            s.W, s.m = O.momentum_update(P, s.W, s.m, orc.lr, orc.mu, orc.wd)
            ea = rel_fro(to_np(h.state(i, K.KFAC_STATE_AINV)), s.Ainv)
            eg = rel_fro(to_np(h.state(i, K.KFAC_STATE_GINV)), s.Ginv)
            assert ea <= 5e-5 and eg <= 5e-5, (t, i, ea, eg)
            Wg = np.concatenate([to_np(pw[i]), to_np(pb[i])[:, None]], axis=1)
            assert rel_fro(Wg, s.W) <= 1e-4, (t, i, rel_fro(Wg, s.W))
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("beta", [0.5, 1.0])
def test_inverse_free_steps_bf16_match_oracle(beta):
    """The schedule above with the products on bf16 tensor cores: step 1 refreshes
    by Cholesky (seeds K), steps 2-6 take one bf16 inverse-free step of every K.
    The inverses K K^T and the preconditioned gradients P against the float64
    oracle's iteration from the same seed: 2e-2 (the bf16 path's tolerance)."""
    shapes = [(900, 1024, 1024), (600, 299, 130), (300, 64, 17)]   # (M, d_in, o)
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32) for _, d, o in shapes],
               max_rows=max(M for M, _, _ in shapes), ikfac=K.KFAC_IKFAC_BF16, **HP)
    idx = list(range(len(shapes)))
    A = [np.zeros((d + 1, d + 1)) for _, d, _ in shapes]
    G = [np.zeros((o, o)) for _, _, o in shapes]
    KA, KG = [None] * 3, [None] * 3
    pw = [to_dev(np.zeros((o, d), np.float32)) for _, d, o in shapes]
    pb = [to_dev(np.zeros(o, np.float32)) for _, _, o in shapes]
    worst = {"inv": 0.0, "P": 0.0}
    for t in range(1, 7):
        ins = [_draw(M, d, o) for M, d, o in shapes]
        h.update_factors_batched(idx, [to_dev(x[0]) for x in ins], [to_dev(x[1]) for x in ins])
        if t == 1:
            h.invert(-1)
        else:
            h.ikfac_update(-1, beta=beta)
        ow = [torch.empty(o, d, device="cuda") for _, d, o in shapes]
        ob = [torch.empty(o, device="cuda") for _, _, o in shapes]
        h.precondition_batched(idx, [to_dev(x[2]) for x in ins], [to_dev(x[3]) for x in ins],
                               ow, ob, pw, pb)
        for i, x in enumerate(ins):
            A[i] = O.ema(A[i], O.factor(x[0], 1), HP["ema_decay"])
            G[i] = O.ema(G[i], O.factor(x[1], 0), HP["ema_decay"])
            if t == 1:
                KA[i], KG[i] = O.ikfac_init(A[i], GAMMA), O.ikfac_init(G[i], GAMMA)
            else:
                KA[i] = O.ikfac_update(KA[i], A[i], GAMMA, beta)
                KG[i] = O.ikfac_update(KG[i], G[i], GAMMA, beta)
            Ainv, Ginv = O.ikfac_inverse(KA[i]), O.ikfac_inverse(KG[i])
            ea = rel_fro(to_np(h.state(i, K.KFAC_STATE_AINV)), Ainv)
            eg = rel_fro(to_np(h.state(i, K.KFAC_STATE_GINV)), Ginv)
            P = O.precondition(Ginv, O.grad_hat(x[2], x[3]), Ainv)
            ep = rel_fro(O.grad_hat(to_np(ow[i]), to_np(ob[i])), P)
            worst["inv"] = max(worst["inv"], ea, eg)
            worst["P"] = max(worst["P"], ep)
            assert ea <= 2e-2 and eg <= 2e-2 and ep <= 2e-2, (t, i, ea, eg, ep)
    print(f"bf16 inverse-free steps, beta {beta}: worst inverse {worst['inv']:.2e}, "
          f"worst P {worst['P']:.2e}")
    assert h.get_status()[0] == 0


def test_tied_a_steps_with_its_source():
    M, d, o = 400, 96, 48
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32)] * 2, max_rows=M, ikfac=1, **HP)
    h.tie_a_factor(1, 0)
    a, g0, _, _ = _draw(M, d, o)
    _, g1, _, _ = _draw(M, d, o)
    h.update_factors_batched([0, 1], [to_dev(a), None], [to_dev(g0), to_dev(g1)])
    h.invert(-1)
    a2, g2, _, _ = _draw(M, d, o)
    h.update_factors_batched([0, 1], [to_dev(a2), None], [to_dev(g2), to_dev(g1)])
    h.ikfac_update(-1, beta=1.0)
    A = 0.9 * 0.1 * O.factor(a, 1) + 0.1 * O.factor(a2, 1)
    KA = O.ikfac_update(O.ikfac_init(0.1 * O.factor(a, 1), GAMMA), A, GAMMA, 1.0)
    for li in (0, 1):
        assert rel_fro(to_np(h.state(li, K.KFAC_STATE_AINV)), O.ikfac_inverse(KA)) <= 5e-5
    assert h.state_info(1, K.KFAC_STATE_AINV) == h.state_info(0, K.KFAC_STATE_AINV)


def test_inverse_free_update_rules():
    L = (K.KFAC_KRON, 16, 32, 1, K.KFAC_F32)
    plain = K.Kfac([L], max_rows=64, **HP)
    with pytest.raises(K.KfacError) as e:
        plain.ikfac_update(0, beta=1.0)
    assert e.value.code == 7                        # not created with ikfac
    h = K.Kfac([L], max_rows=64, ikfac=1, **HP)
    with pytest.raises(K.KfacError) as e:
        h.ikfac_update(0, beta=1.0)
    assert e.value.code == 3                        # no refresh has seeded K yet
    h.update_factors(0, torch.rand(64, 32, device="cuda"), torch.randn(64, 16, device="cuda"))
    h.invert(0)
    for beta in (0.0, 2.0, -1.0):
        with pytest.raises(K.KfacError) as e:
            h.ikfac_update(0, beta=beta)
        assert e.value.code == 1
    hp = K.HParams(0.9, 1e-2, 1e-2, 0.9, 5e-4, 0, 0, 0)   # ikfac is fixed at creation
    assert K.LIB.kfac_set_hparams(h._h, ctypes.byref(hp)) == 1
    h.ikfac_update(0, beta=1.0)
    assert h.get_status()[0] == 0
