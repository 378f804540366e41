"""GPU parity of every kernel of the step against the float64 oracle, through the C ABI.

Tolerances (relative Frobenius unless stated):
  factors A, G (fp32 or bf16 inputs, oracle fed the same rounded inputs)  1e-5
  preconditioned gradient P and updated W                                 1e-4
  diagonal factors (elementwise)                                          1e-5
  diagonal step P, W, m, EMA vectors (same fp32 inputs and state)         1e-6 elementwise,
     relative to the magnitude of the terms forming each element (m and W are sums
     that can cancel); the free-running trajectory within 1e-6 relative Frobenius
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_helpers import to_dev, to_np, rel_fro, max_rel_elem, bf16_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import second_order_optimizer_gb300 as K  # noqa: E402

HP = dict(ema_decay=0.95, damping=1e-3, lr=1e-2, momentum=0.9, weight_decay=5e-4)
RNG = np.random.default_rng(7)


def _orc(**kw):
    hp = dict(HP)
    hp.update(kw)
    return O.KfacOracle(hp["ema_decay"], hp["damping"], hp["lr"], hp["momentum"],
                        hp["weight_decay"], kw.get("invert_every", 1))


def _inputs(M, d_in, o, act="relu", g_std=1e-3, dtype="f32"):
    a = RNG.standard_normal((M, d_in))
    if act == "relu":
        a = np.maximum(a, 0)
    a = W.round_input(a, dtype)
    g = W.round_input(RNG.standard_normal((M, o)) * g_std, dtype)
    return a, g


def _dev_in(x, dtype):
    return bf16_tensor(x) if dtype == "bf16" else to_dev(x)


# ------------------------------------------------------------------ K1 factors

@pytest.mark.parametrize("M,d_in,o,bias,dtype", [
    (1000, 300, 200, 1, "f32"), (129, 7, 130, 0, "f32"), (5000, 64, 16, 1, "f32"),
    (1, 1, 1, 1, "f32"), (777, 257, 129, 1, "bf16"), (20000, 27, 64, 1, "f32"),
    # bf16 column pairs: the ones column inside a pair (63 + 1), starting one (64 + 1),
    # a G width with an odd last pair (33), a single input column, a ragged row count
    (130, 63, 64, 1, "bf16"), (100, 64, 33, 1, "bf16"), (1000, 1, 3, 1, "bf16"),
    (4099, 130, 7, 0, "bf16"),
])
def test_factor_update_matches_oracle(M, d_in, o, bias, dtype):
    kd = K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32
    h = K.Kfac([(K.KFAC_KRON, o, d_in, bias, kd)], max_rows=M, **HP)
    A = np.zeros((d_in + bias,) * 2)
    G = np.zeros((o, o))
    for step in range(3):
        a, g = _inputs(M, d_in, o, dtype=dtype)
        h.update_factors(0, _dev_in(a, dtype), _dev_in(g, dtype))
        A = O.ema(A, O.factor(a, bias), 0.95)
        G = O.ema(G, O.factor(g, 0), 0.95)
        Ag, Gg = to_np(h.state(0, K.KFAC_STATE_A)), to_np(h.state(0, K.KFAC_STATE_G))
        assert rel_fro(Ag, A) <= 1e-5, (step, rel_fro(Ag, A))
        assert rel_fro(Gg, G) <= 1e-5, (step, rel_fro(Gg, G))
        assert np.array_equal(Ag, Ag.T) and np.array_equal(Gg, Gg.T)
    assert h.get_status()[0] == 0


def test_factor_ema_init_first_and_custom_scale():
    M, d_in, o = 300, 40, 24
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_F32)], max_rows=M,
               ema_init=K.KFAC_EMA_INIT_FIRST, **HP)
    a, g = _inputs(M, d_in, o)
    h.update_factors(0, to_dev(a), to_dev(g), scale=0.125)
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)), O.factor(a, 1, scale=0.125)) <= 1e-5
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_G)), O.factor(g, 0, scale=0.125)) <= 1e-5


def test_factor_constant_input_converges():
    """EMA of a constant factor converges to it (closed form C + xi^t (0 - C))."""
    M, d_in, o = 256, 33, 17
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_F32)], max_rows=M, **HP)
    a, g = _inputs(M, d_in, o)
    da, dg = to_dev(a), to_dev(g)
    C = O.factor(a, 1)
    for t in range(1, 121):
        h.update_factors(0, da, dg)
    Ag = to_np(h.state(0, K.KFAC_STATE_A))
    assert rel_fro(Ag, C * (1 - 0.95 ** 120)) <= 1e-5


@pytest.mark.parametrize("width", [71, 72])
def test_factor_strided_bf16_input(width):
    """bf16 inputs as column slices of a wider tensor: an odd row pitch (element-wise
    pack) and an even one (column-pair pack)."""
    M, d_in, o = 333, 50, 21
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_BF16)], max_rows=M, **HP)
    big_a, big_g = _inputs(M, width, width, dtype="bf16")
    ta, tg = _dev_in(big_a, "bf16"), _dev_in(big_g, "bf16")
    h.update_factors(0, ta[:, :d_in], tg[:, :o])
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)), 0.05 * O.factor(big_a[:, :d_in], 1)) <= 1e-5
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_G)), 0.05 * O.factor(big_g[:, :o], 0)) <= 1e-5


@pytest.mark.parametrize("d_in,o,bias,pad", [
    (3072, 3072, 1, 0),   # ones column from the ones matrix (a chunk of its own)
    (3008, 3100, 1, 8),   # strided rows (pitch d + 8), G with a ragged last chunk
    (3072, 3000, 0, 0),   # no bias
    (3000, 3100, 1, 0),   # d_in not a multiple of 64: A through the pack, G in place
    (3072, 3072, 1, 3),   # row pitch not a 16-byte multiple: both through the pack
])
def test_factor_bf16_in_place_syrk_matches_oracle(d_in, o, bias, pad):
    """bf16 factors wide enough for a wave of CTA pairs read the activations in place
    as MN-major operands (no pack); three EMA steps against the oracle, with a row
    count that leaves a ragged last k block."""
    M = 1000
    h = K.Kfac([(K.KFAC_KRON, o, d_in, bias, K.KFAC_BF16)], max_rows=M, **HP)
    A = np.zeros((d_in + bias,) * 2)
    G = np.zeros((o, o))
    for step in range(3):
        big_a, big_g = _inputs(M, d_in + pad, o + pad, dtype="bf16")
        ta, tg = _dev_in(big_a, "bf16"), _dev_in(big_g, "bf16")
        h.update_factors(0, ta[:, :d_in], tg[:, :o])
        A = O.ema(A, O.factor(big_a[:, :d_in], bias), 0.95)
        G = O.ema(G, O.factor(big_g[:, :o], 0), 0.95)
        Ag, Gg = to_np(h.state(0, K.KFAC_STATE_A)), to_np(h.state(0, K.KFAC_STATE_G))
        assert rel_fro(Ag, A) <= 1e-5, (step, rel_fro(Ag, A))
        assert rel_fro(Gg, G) <= 1e-5, (step, rel_fro(Gg, G))
        assert np.array_equal(Ag, Ag.T) and np.array_equal(Gg, Gg.T)
    assert h.get_status()[0] == 0


def test_factor_bf16_batched_in_place_and_packed_mix():
    """A batched bf16 call whose wide factors fill a wave of CTA pairs: those read in
    place, the rest (d_in not a multiple of 64) through the pack, one handle, two
    steps; batched equals per-layer calls and the oracle."""
    shapes = [(1024, 1024, 1)] * 5 + [(1000, 1030, 1), (1024, 700, 0)]
    descs = [(K.KFAC_KRON, o, d, b, K.KFAC_BF16) for d, o, b in shapes]
    M = 777
    hb = K.Kfac(descs, max_rows=M, **HP)
    hs = K.Kfac(descs, max_rows=M, **HP)
    ins = [_inputs(M, d, o, dtype="bf16") for (_, o, d, b, _) in descs]
    for step in range(2):
        a_l = [_dev_in(a, "bf16") for a, _ in ins]
        g_l = [_dev_in(g, "bf16") for _, g in ins]
        hb.update_factors_batched(list(range(len(descs))), a_l, g_l)
        for li in range(len(descs)):
            hs.update_factors(li, a_l[li], g_l[li])
    for li, (_, o, d, b, _) in enumerate(descs):
        a, g = ins[li]
        for which, ref in ((K.KFAC_STATE_A, O.factor(a, b)), (K.KFAC_STATE_G, O.factor(g, 0))):
            ref = ref * (1 - 0.95 ** 2)
            xb, xs = to_np(hb.state(li, which)), to_np(hs.state(li, which))
            assert rel_fro(xb, ref) <= 1e-5, (li, which, rel_fro(xb, ref))
            assert rel_fro(xs, ref) <= 1e-5, (li, which, rel_fro(xs, ref))
            assert np.array_equal(xb, xb.T)
    assert hb.get_status()[0] == 0


def test_factor_strided_input():
    M, d_in, o = 400, 50, 20
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_F32)], max_rows=M, **HP)
    big_a, big_g = _inputs(M, d_in + 13, o + 5)
    ta, tg = to_dev(big_a), to_dev(big_g)
    h.update_factors(0, ta[:, :d_in], tg[:, :o])
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)), 0.05 * O.factor(big_a[:, :d_in], 1)) <= 1e-5
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_G)), 0.05 * O.factor(big_g[:, :o], 0)) <= 1e-5


# ------------------------------------------------------------------ K2/K3 inverse

@pytest.mark.parametrize("n_in,o", [(0, 1), (27, 64), (63, 5), (64, 100), (128, 129), (299, 300),
                                    (512, 65), (1100, 1030), (1600, 700), (2048, 2049),
                                    (1800, 2300)])
def test_invert_matches_oracle(n_in, o):
    """Ainv/Ginv vs the oracle's textbook Cholesky inverse of the same (GPU) factor.
    Handles with a factor above 1536 take the blocked path (512-column outer
    panels, their second 256-column halves and the trailing block updated on the
    tensor cores): 1601 leaves a ragged last panel and block; 1801 with 2300 ends
    9 rows past a half-panel boundary while the other factor goes on."""
    bias = 1
    d_in = max(n_in, 1)
    M = 2 * (d_in + 1) + 3
    h = K.Kfac([(K.KFAC_KRON, o, d_in, bias, K.KFAC_F32)], max_rows=M, ema_init=K.KFAC_EMA_INIT_FIRST, **HP)
    a, g = _inputs(M, d_in, o, g_std=0.1)
    h.update_factors(0, to_dev(a), to_dev(g))
    h.invert(0)
    assert h.get_status()[0] == 0
    for wf, wi in ((K.KFAC_STATE_A, K.KFAC_STATE_AINV), (K.KFAC_STATE_G, K.KFAC_STATE_GINV)):
        F = to_np(h.state(0, wf))
        Finv = to_np(h.state(0, wi))
        ref = O.damped_inverse(F, HP["damping"])
        assert np.array_equal(Finv, Finv.T)
        assert rel_fro(Finv, ref) <= 1e-4, rel_fro(Finv, ref)


def test_invert_all_layers_batched():
    layers = [(K.KFAC_KRON, 70, 200, 1, K.KFAC_F32), (K.KFAC_DIAG, 8, 8, 1, K.KFAC_F32),
              (K.KFAC_KRON, 10, 3, 0, K.KFAC_F32), (K.KFAC_KRON, 300, 129, 1, K.KFAC_F32)]
    M = 700
    h = K.Kfac(layers, max_rows=M, **HP)
    for li, (kind, o, d_in, bias, _) in enumerate(layers):
        if kind == K.KFAC_KRON:
            a, g = _inputs(M, d_in, o, g_std=0.05)
            h.update_factors(li, to_dev(a), to_dev(g))
    h.invert(-1)
    assert h.get_status()[0] == 0
    for li, (kind, *_rest) in enumerate(layers):
        if kind != K.KFAC_KRON:
            continue
        for wf, wi in ((K.KFAC_STATE_A, K.KFAC_STATE_AINV), (K.KFAC_STATE_G, K.KFAC_STATE_GINV)):
            F = to_np(h.state(li, wf))
            assert rel_fro(to_np(h.state(li, wi)), O.damped_inverse(F, HP["damping"])) <= 1e-4


def test_invert_reports_not_positive_definite():
    """A factor made indefinite on the host: the device reports layer and column, no fault."""
    d_in, o = 100, 70
    h = K.Kfac([(K.KFAC_KRON, 5, 5, 1, K.KFAC_F32), (K.KFAC_KRON, o, d_in, 1, K.KFAC_F32)],
               max_rows=8, **HP)
    n = d_in + 1
    Abad = np.eye(n)
    Abad[77, 77] = -1.0
    h.state(1, K.KFAC_STATE_A).copy_(to_dev(Abad.astype(np.float32)))
    h.invert(-1)
    code, layer, info = h.get_status()
    assert (code, layer, info) == (4, 1, 77)
    assert h.get_status()[0] == 0          # cleared by the read
    h.state(1, K.KFAC_STATE_A).copy_(to_dev(np.eye(n, dtype=np.float32)))
    h.invert(1)
    assert h.get_status()[0] == 0
    ref = np.eye(n) / (1 + math.sqrt(HP["damping"]))
    assert rel_fro(to_np(h.state(1, K.KFAC_STATE_AINV)), ref) <= 1e-6


# ------------------------------------------------------------------ K4 precondition

@pytest.mark.parametrize("M,d_in,o,bias", [(600, 200, 150, 1), (300, 65, 1, 1), (90, 33, 70, 0)])
def test_precondition_and_update_match_oracle(M, d_in, o, bias):
    h = K.Kfac([(K.KFAC_KRON, o, d_in, bias, K.KFAC_F32)], max_rows=M, **HP)
    st = O.LayerState("kron", o, d_in, bias, np.zeros((o, d_in)), np.zeros(o) if bias else None)
    orc = _orc(invert_every=2)
    w0 = (RNG.standard_normal((o, d_in)) * 0.1).astype(np.float32)
    b0 = (RNG.standard_normal(o) * 0.1).astype(np.float32) if bias else None
    st.W = O.grad_hat(w0, b0).copy()
    pw, pb = to_dev(w0), (to_dev(b0) if bias else None)
    with pytest.raises(K.KfacError):
        h.precondition(0, to_dev(w0), pb, out_w=torch.empty_like(pw), out_b=pb)  # before invert
    for t in range(3):
        a, g = _inputs(M, d_in, o)
        gw = (RNG.standard_normal((o, d_in)) * 1e-3).astype(np.float32)
        gb = (RNG.standard_normal(o) * 1e-3).astype(np.float32) if bias else None
        h.update_factors(0, to_dev(a), to_dev(g))
        if t % 2 == 0:
            h.invert(0)
        ow = torch.empty(o, d_in, device="cuda")
        ob = torch.empty(o, device="cuda") if bias else None
        h.precondition(0, to_dev(gw), to_dev(gb) if bias else None, ow, ob, pw, pb)
        P = orc.step_kron(st, a, g, gw, gb)
        Pg = O.grad_hat(to_np(ow), to_np(ob) if bias else None)
        assert rel_fro(Pg, P) <= 1e-4, (t, rel_fro(Pg, P))
        Wg = O.grad_hat(to_np(pw), to_np(pb) if bias else None)
        assert rel_fro(Wg, st.W) <= 1e-4
        mw, mb = h.momentum(0)
        assert rel_fro(O.grad_hat(to_np(mw), to_np(mb) if bias else None), st.m) <= 1e-4
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("batched", [False, True])
def test_bf16_preconditioning_within_the_bf16_tolerance(batched):
    """hp.math = KFAC_MATH_BF16: the inverses (at each refresh), the gradient and
    X = dW-hat A^{-1} rounded to bf16, one bf16 tensor-core product each (fp32
    accumulate); factors, inverses and the update stay fp32.  P, m and W against
    the float64 oracle's step at the bf16 path's 2e-2 (relative Frobenius), three
    steps with a refresh at the first and third; ragged and bias-less shapes."""
    shapes = [(1000, 300, 200, 1), (600, 129, 70, 0), (1500, 1024, 1030, 1)]   # M, d_in, o, bias
    h = K.Kfac([(K.KFAC_KRON, o, d, b, K.KFAC_F32) for _, d, o, b in shapes],
               max_rows=max(M for M, *_ in shapes), math=K.KFAC_MATH_BF16, **HP)
    orc = _orc(invert_every=2)
    st, pw, pb = [], [], []
    for _, d, o, b in shapes:
        w0 = (RNG.standard_normal((o, d)) * 0.1).astype(np.float32)
        b0 = (RNG.standard_normal(o) * 0.1).astype(np.float32) if b else None
        st.append(O.LayerState("kron", o, d, b, w0, b0))
        pw.append(to_dev(w0))
        pb.append(to_dev(b0) if b else None)
    worst = 0.0
    for t in range(3):
        ins = []
        for M, d, o, b in shapes:
            a, g = _inputs(M, d, o)
            gw = (RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)
            gb = (RNG.standard_normal(o) * 1e-3).astype(np.float32) if b else None
            ins.append((a, g, gw, gb))
        for li, (a, g, _, _) in enumerate(ins):
            h.update_factors(li, to_dev(a), to_dev(g))
        if t % 2 == 0:
            h.invert(-1)
        ow = [torch.empty(o, d, device="cuda") for _, d, o, _ in shapes]
        ob = [torch.empty(o, device="cuda") if b else None for _, _, o, b in shapes]
        gws = [to_dev(x[2]) for x in ins]
        gbs = [to_dev(x[3]) if x[3] is not None else None for x in ins]
        if batched:
            h.precondition_batched(list(range(len(shapes))), gws, gbs, ow, ob, pw, pb)
        else:
            for li in range(len(shapes)):
                h.precondition(li, gws[li], gbs[li], ow[li], ob[li], pw[li], pb[li])
        for li, (a, g, gw, gb) in enumerate(ins):
            b = shapes[li][3]
            P = orc.step_kron(st[li], a, g, gw, gb)
            errs = [rel_fro(O.grad_hat(to_np(ow[li]), to_np(ob[li]) if b else None), P),
                    rel_fro(O.grad_hat(to_np(pw[li]), to_np(pb[li]) if b else None), st[li].W)]
            mw, mb = h.momentum(li)
            errs.append(rel_fro(O.grad_hat(to_np(mw), to_np(mb) if b else None), st[li].m))
            worst = max(worst, errs[0])
            assert max(errs) <= 2e-2, (t, li, errs)
    print(f"bf16 preconditioning ({'batched' if batched else 'per layer'}): worst P {worst:.2e}")
    assert h.get_status()[0] == 0


# ------------------------------------------------------------------ K5 / K6 diagonal

@pytest.mark.parametrize("M,d_in,o,bias,dtype", [(3000, 257, 100, 1, "f32"), (50, 3, 2, 0, "f32"),
                                                 (2500, 640, 64, 1, "bf16"),
                                                 # 16-byte-load form: ragged rows, a partial
                                                 # last column block
                                                 (3001, 256, 100, 1, "f32"),
                                                 (777, 328, 40, 0, "bf16"), (5, 8, 8, 1, "bf16")])
def test_diag_factors_match_oracle(M, d_in, o, bias, dtype):
    kd = K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32
    h = K.Kfac([(K.KFAC_DIAG, o, d_in, bias, kd)], max_rows=M, **HP)
    a, g = _inputs(M, d_in, o, act="normal", dtype=dtype)
    gn = torch.empty(o, device="cuda")
    an = torch.empty(d_in + bias, device="cuda")
    h.diag_factors(0, _dev_in(a, dtype), _dev_in(g, dtype), gn, an)
    # diagonal factors are factors: same 1e-5 bound, here held elementwise
    assert max_rel_elem(to_np(gn), O.diag_factor(g, 0), 0) <= 1e-5
    assert max_rel_elem(to_np(an), O.diag_factor(a, bias), 0) <= 1e-5


def _componentwise(x, ref, scale):
    """max |x - ref| / scale, scale = sum of the magnitudes of the terms forming ref."""
    x, ref, scale = (np.asarray(v, np.float64) for v in (x, ref, scale))
    return float(np.max(np.abs(x - ref) / np.maximum(scale, 1e-30)))


@pytest.mark.parametrize("o,d_in,bias", [(64, 256, 1), (33, 5, 1), (128, 1, 1), (7, 12, 0),
                                         (300, 1024, 1)])
def test_diag_step_elementwise(o, d_in, bias):
    """Each step starts both sides from the GPU's fp32 state; every element of P, m, W and
    of the EMA vectors must agree to 1e-6 relative to the magnitude of the terms that
    form it (P = dW/(g a + gamma) is a quotient, so that is |P|; m = mu m + P + lambda W
    is a sum, so that is mu|m| + |P| + lambda|W|; W - eta m expands to
    W - eta (mu m + P + lambda W): |W| + eta (mu|m| + |P| + lambda|W|))."""
    h = K.Kfac([(K.KFAC_DIAG, o, d_in, bias, K.KFAC_F32)], max_rows=1, **HP)
    n = d_in + bias
    xi, gam, eta, mu, lam = (HP[k] for k in ("ema_decay", "damping", "lr", "momentum",
                                             "weight_decay"))
    st = O.LayerState("diag", o, d_in, bias, np.zeros((o, d_in)), np.zeros(o) if bias else None)
    orc = _orc()
    w0 = (RNG.standard_normal((o, d_in)) * 0.1).astype(np.float32)
    b0 = (RNG.standard_normal(o) * 0.1).astype(np.float32) if bias else None
    pw, pb = to_dev(w0), (to_dev(b0) if bias else None)
    bo = lambda x, y: O.grad_hat(to_np(x), to_np(y) if bias else None)
    traj = O.LayerState("diag", o, d_in, bias, w0, b0)
    for t in range(4):
        mw, mb = h.momentum(0)
        st.W, st.m = bo(pw, pb), bo(mw, mb)
        st.gs = to_np(h.state(0, K.KFAC_STATE_GDIAG))
        st.as_ = to_np(h.state(0, K.KFAC_STATE_ADIAG))
        st.t = t
        W_old, m_old, gs_old, as_old = st.W.copy(), st.m.copy(), st.gs.copy(), st.as_.copy()
        gn = RNG.uniform(0, 2e-6, o).astype(np.float32)
        an = RNG.uniform(0, 2, n).astype(np.float32)
        gw = (RNG.standard_normal((o, d_in)) * 1e-3).astype(np.float32)
        gb = (RNG.standard_normal(o) * 1e-3).astype(np.float32) if bias else None
        ow = torch.empty(o, d_in, device="cuda")
        ob = torch.empty(o, device="cuda") if bias else None
        h.diag_step(0, to_dev(gn), to_dev(an), to_dev(gw), to_dev(gb) if bias else None, pw, pb,
                    ow, ob)
        P = orc.step_diag(st, gn, an, gw, gb)
        orc.step_diag(traj, gn, an, gw, gb)
        mw, mb = h.momentum(0)
        m_terms = mu * np.abs(m_old) + np.abs(P) + lam * np.abs(W_old)
        errs = {"P": _componentwise(bo(ow, ob), P, np.abs(P)),
                "m": _componentwise(bo(mw, mb), st.m, m_terms),
                "W": _componentwise(bo(pw, pb), st.W, np.abs(W_old) + eta * m_terms)}
        # the plain elementwise relative error |x - x*| / |x*|, reported beside the
        # bound above (they differ where m or W cancel to near zero)
        plain = {"P": _componentwise(bo(ow, ob), P, np.abs(P)),
                 "m": _componentwise(bo(mw, mb), st.m, np.abs(st.m)),
                 "W": _componentwise(bo(pw, pb), st.W, np.abs(st.W))}
        print(f"diag step o={o} d_in={d_in} t={t}: terms-relative "
              + " ".join(f"{k} {v:.2e}" for k, v in errs.items()) + "; plain relative "
              + " ".join(f"{k} {v:.2e}" for k, v in plain.items()))
        assert errs["P"] <= 1e-6 and errs["m"] <= 1e-6 and errs["W"] <= 1e-6, errs
        assert _componentwise(to_np(h.state(0, K.KFAC_STATE_GDIAG)), st.gs,
                              xi * np.abs(gs_old) + (1 - xi) * np.abs(gn)) <= 1e-6
        assert _componentwise(to_np(h.state(0, K.KFAC_STATE_ADIAG)), st.as_,
                              xi * np.abs(as_old) + (1 - xi) * np.abs(an)) <= 1e-6
    # and the free-running 4-step trajectory stays within 1e-6 (relative Frobenius)
    assert rel_fro(bo(pw, pb), traj.W) <= 1e-6


# ------------------------------------------------------------------ whole configs

def _run_config_small(cfg_name, steps, check_every=1):
    cfg = W.get_config(cfg_name)
    hp = cfg.hp
    kinds = [K.KFAC_KRON if l.kind == "kron" else K.KFAC_DIAG for l in cfg.layers]
    descs = [(k, l.d_out, l.d_in, l.has_bias, K.KFAC_BF16 if l.in_dtype == "bf16" else K.KFAC_F32)
             for k, l in zip(kinds, cfg.layers)]
    h = K.Kfac(descs, max_rows=max(l.rows for l in cfg.layers), ema_decay=hp.ema_decay,
               damping=hp.damping, lr=hp.lr, momentum=hp.momentum, weight_decay=hp.weight_decay)
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay,
                       cfg.invert_every)
    states, params = [], []
    for li, l in enumerate(cfg.layers):
        src = 0 if cfg_name == "c1" else li       # c1's two layers share one set of inputs
        w0, b0 = W.initial_params(cfg, src)
        states.append(O.LayerState(l.kind, l.d_out, l.d_in, l.has_bias, w0, b0))
        params.append((to_dev(w0), to_dev(b0) if l.has_bias else None))
    worst = {"A": 0.0, "G": 0.0, "P": 0.0, "W": 0.0, "Wdiag": 0.0}
    for t in range(1, steps + 1):
        for li, l in enumerate(cfg.layers):
            src = 0 if cfg_name == "c1" else li
            x = W.layer_inputs(cfg, src, t)
            gb = x["grad_b"]
            pw, pb = params[li]
            if l.kind == "kron":
                h.update_factors(li, to_dev(x["a"]), to_dev(x["g"]))
                if (t - 1) % cfg.invert_every == 0:
                    h.invert(li)
                ow = torch.empty(l.d_out, l.d_in, device="cuda")
                ob = torch.empty(l.d_out, device="cuda") if l.has_bias else None
                h.precondition(li, to_dev(x["grad_w"]), to_dev(gb) if l.has_bias else None,
                               ow, ob, pw, pb)
                P = orc.step_kron(states[li], x["a"], x["g"], x["grad_w"], gb)
                if t % check_every == 0 or t == steps:
                    worst["A"] = max(worst["A"], rel_fro(to_np(h.state(li, K.KFAC_STATE_A)), states[li].A))
                    worst["G"] = max(worst["G"], rel_fro(to_np(h.state(li, K.KFAC_STATE_G)), states[li].G))
                    worst["P"] = max(worst["P"], rel_fro(
                        O.grad_hat(to_np(ow), to_np(ob) if l.has_bias else None), P))
                    worst["W"] = max(worst["W"], rel_fro(
                        O.grad_hat(to_np(pw), to_np(pb) if l.has_bias else None), states[li].W))
            else:
                gn = torch.empty(l.d_out, device="cuda")
                an = torch.empty(l.n, device="cuda")
                h.diag_factors(li, to_dev(x["a"]), to_dev(x["g"]), gn, an)
                h.diag_step(li, gn, an, to_dev(x["grad_w"]), to_dev(gb), pw, pb)
                orc.step_diag(states[li], O.diag_factor(x["g"]), O.diag_factor(x["a"], l.has_bias),
                              x["grad_w"], gb)
                worst["Wdiag"] = max(worst["Wdiag"], rel_fro(
                    O.grad_hat(to_np(pw), to_np(pb)), states[li].W))
    assert h.get_status()[0] == 0
    return worst


def test_single_linear_layer_both_paths_10_steps():
    worst = _run_config_small("c1", 10)
    assert worst["A"] <= 1e-5 and worst["G"] <= 1e-5, worst
    assert worst["P"] <= 1e-4 and worst["W"] <= 1e-4, worst
    assert worst["Wdiag"] <= 1e-6, worst


def test_mlp4_full_size_two_refreshes():
    """4-layer MLP at full size (1024 wide, batch 1024), 11 steps: inverses refreshed at 1 and 11."""
    worst = _run_config_small("c2", 11, check_every=5)
    assert worst["A"] <= 1e-5 and worst["G"] <= 1e-5, worst
    assert worst["P"] <= 1e-4 and worst["W"] <= 1e-4, worst


# ------------------------------------------------------------------ batched entry points

def _mixed_layers(dtype):
    kd = K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32
    shapes = [(1024, 1024, 1), (300, 150, 1), (64, 10, 1), (33, 70, 0), (513, 1000, 1)]
    shapes += [(40 + 3 * i, 20 + 5 * i, i % 2) for i in range(15)]   # > 16 problems: 2+ groups
    return [(K.KFAC_KRON, o, d, b, kd) for d, o, b in shapes]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_update_factors_batched_matches_single_calls(dtype):
    descs = _mixed_layers(dtype)
    M = 700
    hb = K.Kfac(descs, max_rows=M, **HP)
    hs = K.Kfac(descs, max_rows=M, **HP)
    ins = [_inputs(M, d, o, dtype=dtype) for (_, o, d, b, _) in descs]
    for step in range(2):
        a_l = [_dev_in(a, dtype) for a, _ in ins]
        g_l = [_dev_in(g, dtype) for _, g in ins]
        hb.update_factors_batched(list(range(len(descs))), a_l, g_l)
        for li in range(len(descs)):
            hs.update_factors(li, a_l[li], g_l[li])
    for li, (_, o, d, b, _) in enumerate(descs):
        a, g = ins[li]
        Aref = O.factor(a, b) * (1 - 0.95 ** 2)
        for which, ref in ((K.KFAC_STATE_A, Aref), (K.KFAC_STATE_G, O.factor(g, 0) * (1 - 0.95 ** 2))):
            xb, xs = to_np(hb.state(li, which)), to_np(hs.state(li, which))
            assert rel_fro(xb, xs) <= 1e-6, (li, which)
            assert rel_fro(xb, ref) <= 1e-5, (li, which)
            assert np.array_equal(xb, xb.T)
    assert hb.get_status()[0] == 0


def test_precondition_batched_matches_single_calls():
    descs = _mixed_layers("f32")
    M = 500
    hb = K.Kfac(descs, max_rows=M, **HP)
    hs = K.Kfac(descs, max_rows=M, **HP)
    n_l = len(descs)
    ins = [_inputs(M, d, o, g_std=0.05) for (_, o, d, b, _) in descs]
    for h in (hb, hs):
        for li in range(n_l):
            h.update_factors(li, to_dev(ins[li][0]), to_dev(ins[li][1]))
        h.invert(-1)
    gws = [to_dev((RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)) for (_, o, d, b, _) in descs]
    gbs = [to_dev((RNG.standard_normal(o) * 1e-3).astype(np.float32)) if b else None
           for (_, o, d, b, _) in descs]
    w0 = [(RNG.standard_normal((o, d)) * 0.1).astype(np.float32) for (_, o, d, b, _) in descs]
    b0 = [(RNG.standard_normal(o) * 0.1).astype(np.float32) if b else None for (_, o, d, b, _) in descs]
    pw_b = [to_dev(w) for w in w0]
    pb_b = [to_dev(x) if x is not None else None for x in b0]
    pw_s = [to_dev(w) for w in w0]
    pb_s = [to_dev(x) if x is not None else None for x in b0]
    ow_b = [torch.empty(o, d, device="cuda") for (_, o, d, b, _) in descs]
    ob_b = [torch.empty(o, device="cuda") if b else None for (_, o, d, b, _) in descs]
    hb.precondition_batched(list(range(n_l)), gws, gbs, ow_b, ob_b, pw_b, pb_b)
    for li, (_, o, d, b, _) in enumerate(descs):
        ow = torch.empty(o, d, device="cuda")
        ob = torch.empty(o, device="cuda") if b else None
        hs.precondition(li, gws[li], gbs[li], ow, ob, pw_s[li], pb_s[li])
        gh = lambda w, x: O.grad_hat(to_np(w), to_np(x) if b else None)
        assert rel_fro(gh(ow_b[li], ob_b[li]), gh(ow, ob)) <= 1e-6, li
        assert rel_fro(gh(pw_b[li], pb_b[li]), gh(pw_s[li], pb_s[li])) <= 1e-6, li
        # and against the oracle's formula with the inverses in use
        Pref = O.precondition(to_np(hb.state(li, K.KFAC_STATE_GINV)),
                              gh(gws[li], gbs[li]), to_np(hb.state(li, K.KFAC_STATE_AINV)))
        assert rel_fro(gh(ow_b[li], ob_b[li]), Pref) <= 1e-4, li
    assert hb.get_status()[0] == 0


def test_batched_calls_reject_duplicates_and_mixed_dtypes():
    h = K.Kfac([(K.KFAC_KRON, 8, 8, 1, K.KFAC_F32), (K.KFAC_KRON, 8, 8, 1, K.KFAC_BF16)],
               max_rows=16, **HP)
    a = torch.zeros(16, 8, device="cuda")
    with pytest.raises(K.KfacError):
        h.update_factors_batched([0, 0], [a, a], [a, a])
    with pytest.raises(K.KfacError):
        h.update_factors_batched([0, 1], [a, a.bfloat16()], [a, a.bfloat16()])


def _diag_mix(n_layers, seed):
    """Mixed shapes: d_in multiple of 4 or not (vector and scalar paths), with and without
    bias, BatchNorm-like (d_in = 1), and a few large ones."""
    rng = np.random.default_rng(seed)
    shapes = [(1024, 1024, 1), (1, 256, 1), (1, 64, 1), (96, 50, 0), (1000, 7, 1)]
    while len(shapes) < n_layers:
        d = int(rng.integers(1, 200))
        shapes.append((d, int(rng.integers(1, 120)), int(rng.integers(0, 2))))
    return shapes


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_diag_factors_batched_matches_single_calls(dtype):
    """70 layers (two launches of at most 64): against the single call and the oracle."""
    kd = K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32
    shapes = _diag_mix(70, 5)
    descs = [(K.KFAC_DIAG if i % 3 else K.KFAC_KRON, o, d, b, kd) for i, (d, o, b) in enumerate(shapes)]
    M = 600
    h = K.Kfac(descs, max_rows=M, **HP)
    ins = [_inputs(M, d, o, act="normal", dtype=dtype) for (d, o, b) in shapes]
    a_l = [_dev_in(a, dtype) for a, _ in ins]
    g_l = [_dev_in(g, dtype) for _, g in ins]
    gn_b = [torch.empty(o, device="cuda") for (d, o, b) in shapes]
    an_b = [torch.empty(d + b, device="cuda") for (d, o, b) in shapes]
    h.diag_factors_batched(list(range(len(shapes))), a_l, g_l, gn_b, an_b)
    for li, (d, o, b) in enumerate(shapes):
        gn = torch.empty(o, device="cuda")
        an = torch.empty(d + b, device="cuda")
        h.diag_factors(li, a_l[li], g_l[li], gn, an)
        a, g = ins[li]
        assert max_rel_elem(to_np(gn_b[li]), to_np(gn), 0) <= 1e-6, li
        assert max_rel_elem(to_np(an_b[li]), to_np(an), 0) <= 1e-6, li
        assert max_rel_elem(to_np(gn_b[li]), O.diag_factor(g, 0), 0) <= 1e-5, li
        assert max_rel_elem(to_np(an_b[li]), O.diag_factor(a, b), 0) <= 1e-5, li
    assert h.get_status()[0] == 0


def test_diag_step_batched_bitwise_equals_single_calls():
    """70 DIAG layers, three steps: every output, parameter, momentum and EMA vector of the
    batched launch equals the per-layer launch bit for bit (same arithmetic per element);
    one layer is also followed against the oracle's step formulas."""
    shapes = _diag_mix(70, 6)
    descs = [(K.KFAC_DIAG, o, d, b, K.KFAC_F32) for (d, o, b) in shapes]
    hb = K.Kfac(descs, max_rows=1, **HP)
    hs = K.Kfac(descs, max_rows=1, **HP)
    L = list(range(len(shapes)))
    w0 = [(RNG.standard_normal((o, d)) * 0.1).astype(np.float32) for (d, o, b) in shapes]
    b0 = [(RNG.standard_normal(o) * 0.1).astype(np.float32) if b else None for (d, o, b) in shapes]
    pw_b, pw_s = [to_dev(w) for w in w0], [to_dev(w) for w in w0]
    pb_b = [to_dev(x) if x is not None else None for x in b0]
    pb_s = [to_dev(x) if x is not None else None for x in b0]
    probe = 0   # the 1024 x 1024 layer
    d0, o0, bb0 = shapes[probe]
    traj = O.LayerState("diag", o0, d0, bb0, w0[probe].astype(np.float64),
                        b0[probe].astype(np.float64))
    orc = _orc()
    for t in range(3):
        gn = [to_dev(RNG.uniform(0, 2e-6, o).astype(np.float32)) for (d, o, b) in shapes]
        an = [to_dev(RNG.uniform(0, 2, d + b).astype(np.float32)) for (d, o, b) in shapes]
        gw = [to_dev((RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)) for (d, o, b) in shapes]
        gb = [to_dev((RNG.standard_normal(o) * 1e-3).astype(np.float32)) if b else None
              for (d, o, b) in shapes]
        ow_b = [torch.empty(o, d, device="cuda") for (d, o, b) in shapes]
        ob_b = [torch.empty(o, device="cuda") if b else None for (d, o, b) in shapes]
        hb.diag_step_batched(L, gn, an, gw, gb, pw_b, pb_b, ow_b, ob_b)
        for li, (d, o, b) in enumerate(shapes):
            ow = torch.empty(o, d, device="cuda")
            ob = torch.empty(o, device="cuda") if b else None
            hs.diag_step(li, gn[li], an[li], gw[li], gb[li], pw_s[li], pb_s[li], ow, ob)
            assert torch.equal(ow_b[li], ow) and torch.equal(pw_b[li], pw_s[li]), (t, li)
            if b:
                assert torch.equal(ob_b[li], ob) and torch.equal(pb_b[li], pb_s[li]), (t, li)
            for which in (K.KFAC_STATE_MOMENTUM, K.KFAC_STATE_GDIAG, K.KFAC_STATE_ADIAG):
                assert torch.equal(hb.state(li, which), hs.state(li, which)), (t, li, which)
        orc.step_diag(traj, to_np(gn[probe]), to_np(an[probe]), to_np(gw[probe]),
                      to_np(gb[probe]))
    got = O.grad_hat(to_np(pw_b[probe]), to_np(pb_b[probe]))
    assert rel_fro(got, traj.W) <= 1e-6
    assert hb.get_status()[0] == 0


def test_batched_diag_calls_reject_duplicates_and_wrong_kinds():
    h = K.Kfac([(K.KFAC_DIAG, 8, 8, 1, K.KFAC_F32), (K.KFAC_KRON, 8, 8, 1, K.KFAC_F32)],
               max_rows=16, **HP)
    a = torch.zeros(16, 8, device="cuda")
    v8, v9 = torch.zeros(8, device="cuda"), torch.zeros(9, device="cuda")
    w = torch.zeros(8, 8, device="cuda")
    with pytest.raises(K.KfacError):
        h.diag_factors_batched([0, 0], [a, a], [a, a], [v8, v8], [v9, v9])
    with pytest.raises(K.KfacError):   # K6 is for DIAG layers only
        h.diag_step_batched([0, 1], [v8, v8], [v9, v9], [w, w], [v8, v8], [w, w], [v8, v8])
    with pytest.raises(K.KfacError):
        h.diag_step_batched([0, 0], [v8, v8], [v9, v9], [w, w], [v8, v8], [w, w], [v8, v8])


def test_factor_update_concurrent_with_preconditioning_and_diag_step():
    """The factor update, preconditioning and the diagonal path use disjoint scratch:
    run on three streams at once they leave exactly the state of running them in order
    (split-K products included: a wide, short layer forces them in both phases)."""
    descs = [(K.KFAC_KRON, 64, 700, 1, K.KFAC_F32), (K.KFAC_KRON, 300, 200, 1, K.KFAC_F32),
             (K.KFAC_DIAG, 96, 128, 1, K.KFAC_F32)]
    M = 4096
    hs = [K.Kfac(descs, max_rows=M, **HP) for _ in range(2)]
    ins = [_inputs(M, d, o) for (_, o, d, b, _) in descs]
    a_l = [to_dev(a) for a, _ in ins]
    g_l = [to_dev(g) for _, g in ins]
    for h in hs:
        h.update_factors_batched([0, 1], a_l[:2], g_l[:2])
        h.invert(-1)
    gws = [to_dev((RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)) for (_, o, d, b, _) in descs]
    gbs = [to_dev((RNG.standard_normal(o) * 1e-3).astype(np.float32)) for (_, o, d, b, _) in descs]
    w0 = [(RNG.standard_normal((o, d)) * 0.1).astype(np.float32) for (_, o, d, b, _) in descs]
    b0 = [(RNG.standard_normal(o) * 0.1).astype(np.float32) for (_, o, d, b, _) in descs]
    pw = [[to_dev(w) for w in w0] for _ in range(2)]
    pb = [[to_dev(x) for x in b0] for _ in range(2)]
    gn = to_dev(RNG.uniform(0, 1e-6, 96).astype(np.float32))
    an = to_dev(RNG.uniform(0, 2, 129).astype(np.float32))
    # in order, one stream
    h = hs[0]
    h.update_factors_batched([0, 1], a_l[:2], g_l[:2])
    h.precondition_batched([0, 1], gws[:2], gbs[:2], None, None, pw[0][:2], pb[0][:2])
    k5 = [(torch.empty(96, device="cuda"), torch.empty(129, device="cuda")) for _ in range(2)]
    h.diag_factors(2, a_l[2], g_l[2], k5[0][0], k5[0][1])
    h.diag_step(2, gn, an, gws[2], gbs[2], pw[0][2], pb[0][2])
    torch.cuda.synchronize()
    # overlapped: factor update, preconditioning and the diagonal path on three streams
    h = hs[1]
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        h.update_factors_batched([0, 1], a_l[:2], g_l[:2])
    with torch.cuda.stream(s2):
        h.precondition_batched([0, 1], gws[:2], gbs[:2], None, None, pw[1][:2], pb[1][:2])
    with torch.cuda.stream(s3):
        h.diag_factors(2, a_l[2], g_l[2], k5[1][0], k5[1][1])
        h.diag_step(2, gn, an, gws[2], gbs[2], pw[1][2], pb[1][2])
    torch.cuda.synchronize()
    assert torch.equal(k5[0][0], k5[1][0]) and torch.equal(k5[0][1], k5[1][1])
    for li in range(2):
        for which in (K.KFAC_STATE_A, K.KFAC_STATE_G, K.KFAC_STATE_MOMENTUM):
            assert torch.equal(hs[0].state(li, which), hs[1].state(li, which)), (li, which)
    for li in range(3):
        assert torch.equal(pw[0][li], pw[1][li]) and torch.equal(pb[0][li], pb[1][li]), li
    assert hs[0].get_status()[0] == 0 and hs[1].get_status()[0] == 0


def test_hyperparameter_schedules_through_set_hparams():
    """Warm-up damping gamma(t), an lr/momentum schedule and a BatchNorm-style damping
    rho_BN * gamma(t) for the diagonal layer, all applied with kfac_set_hparams between
    calls (the values are read when a call is enqueued): 8 steps against the oracle
    following the same schedule."""
    d_in, o, M, rho_bn = 96, 48, 256, 4.0
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_F32), (K.KFAC_DIAG, o, d_in, 1, K.KFAC_F32)],
               max_rows=M, **HP)
    orc_k, orc_d = _orc(invert_every=2), _orc()
    w0 = (RNG.standard_normal((o, d_in)) * 0.1).astype(np.float32)
    b0 = (RNG.standard_normal(o) * 0.1).astype(np.float32)
    st_k = O.LayerState("kron", o, d_in, 1, w0, b0)
    st_d = O.LayerState("diag", o, d_in, 1, w0, b0)
    params = [(to_dev(w0), to_dev(b0)) for _ in range(2)]
    for t in range(1, 9):
        gamma = 1e-3 * (1.0 + 20.0 * 0.5 ** t)          # decaying warm-up damping
        lr, mu = 1e-2 * min(1.0, t / 4), 0.9 if t > 2 else 0.5
        a, g = _inputs(M, d_in, o)
        gw = (g.T @ np.hstack([a, np.ones((M, 1))]) / M).astype(np.float32)
        gwd, gbd = to_dev(np.ascontiguousarray(gw[:, :d_in])), to_dev(np.ascontiguousarray(gw[:, d_in]))
        # K-FAC layer
        h.set_hparams(damping=gamma, lr=lr, momentum=mu)
        orc_k.gamma, orc_k.lr, orc_k.mu = gamma, lr, mu
        h.update_factors(0, to_dev(a), to_dev(g))
        if (t - 1) % 2 == 0:
            h.invert(0)
        h.precondition(0, gwd, gbd, None, None, *params[0])
        orc_k.step_kron(st_k, a, g, gw[:, :d_in], gw[:, d_in])
        # diagonal layer with its own damping
        h.set_hparams(damping=rho_bn * gamma)
        orc_d.gamma, orc_d.lr, orc_d.mu = rho_bn * gamma, lr, mu
        gn = torch.empty(o, device="cuda")
        an = torch.empty(d_in + 1, device="cuda")
        h.diag_factors(1, to_dev(a), to_dev(g), gn, an)
        h.diag_step(1, gn, an, gwd, gbd, *params[1])
        orc_d.step_diag(st_d, O.diag_factor(g), O.diag_factor(a, 1), gw[:, :d_in], gw[:, d_in])
    Wk = O.grad_hat(to_np(params[0][0]), to_np(params[0][1]))
    Wd = O.grad_hat(to_np(params[1][0]), to_np(params[1][1]))
    assert rel_fro(Wk, st_k.W) <= 1e-4
    assert rel_fro(Wd, st_d.W) <= 1e-6
    assert h.get_status()[0] == 0


def test_bounded_wait_reports_timeout_and_the_context_stays_usable():
    """Failure detection without a fault: a kernel waits, through the library's
    bounded mbarrier wait, for a phase nothing completes; after ~1 ms of SM clocks
    it records KFAC_ERR_TIMEOUT and returns.  The status is reported once, then
    cleared, and the handle computes correctly afterwards."""
    M, d_in, o = 256, 40, 24
    h = K.Kfac([(K.KFAC_KRON, o, d_in, 1, K.KFAC_F32)], max_rows=M, **HP)
    h.selftest_timeout(2_000_000)
    code, layer, info = h.get_status()
    assert (code, layer, info) == (5, -1, 1)
    assert h.get_status()[0] == 0                      # reported once, then cleared
    a, g = _inputs(M, d_in, o)
    h.update_factors(0, to_dev(a), to_dev(g))
    assert h.get_status()[0] == 0
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)), 0.05 * O.factor(a, 1)) <= 1e-5
    with pytest.raises(K.KfacError):
        h.selftest_timeout(0)
