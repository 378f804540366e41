"""Stale factors and shared A factors on the GPU against the float64 oracle.

Osawa et al. §5.4: after a warm-up the factors are recomputed and re-inverted
less often, A (which fluctuates less) less often than G.  The library provides
per-factor updates (a NULL input leaves that factor as it is), per-factor
refreshes (kfac_invert_factors) and A factors shared by layers fed the same
input (kfac_tie_a_factor); the schedule is the caller's.  Tolerances as for
the plain step: P and W relative Frobenius 1e-4, factors 1e-5.
"""
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
RNG = np.random.default_rng(23)


def _orc():
    return O.KfacOracle(HP["ema_decay"], HP["damping"], HP["lr"], HP["momentum"],
                        HP["weight_decay"])


def _params(o, d):
    return ((RNG.standard_normal((o, d)) * 0.1).astype(np.float32),
            (RNG.standard_normal(o) * 0.1).astype(np.float32))


def _draw(M, d, o):
    a = np.maximum(RNG.standard_normal((M, d)), 0).astype(np.float32)
    g = (RNG.standard_normal((M, o)) * 1e-2).astype(np.float32)
    gw = (RNG.standard_normal((o, d)) * 1e-3).astype(np.float32)
    gb = (RNG.standard_normal(o) * 1e-3).astype(np.float32)
    return a, g, gw, gb


@pytest.mark.parametrize("warmup,every_a,every_g", [(3, 4, 2), (2, 3, 3), (1, 1, 2)])
def test_stale_schedule_matches_oracle(warmup, every_a, every_g):
    shapes = [(600, 150, 90), (300, 700, 40), (257, 33, 129)]   # (M, d_in, o)
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32) for _, d, o in shapes],
               max_rows=max(M for M, _, _ in shapes), **HP)
    orc = _orc()
    states, dev_p = [], []
    for M, d, o in shapes:
        w0, b0 = _params(o, d)
        states.append(O.LayerState("kron", o, d, 1, w0, b0))
        dev_p.append((to_dev(w0), to_dev(b0)))
    idx = list(range(len(shapes)))
    for t in range(1, 12):
        ra, rg = O.stale_refresh(t, warmup, every_a, every_g)
        ins = [_draw(M, d, o) for M, d, o in shapes]
        if ra or rg:
            h.update_factors_batched(idx, [to_dev(x[0]) if ra else None for x in ins],
                                     [to_dev(x[1]) if rg else None for x in ins])
            h.invert(-1, which=(K.KFAC_FACTOR_A if ra else 0) | (K.KFAC_FACTOR_G if rg else 0))
        outs = [torch.empty(o, d, device="cuda") for _, d, o in shapes]
        outb = [torch.empty(o, device="cuda") for _, _, o in shapes]
        h.precondition_batched(idx, [to_dev(x[2]) for x in ins], [to_dev(x[3]) for x in ins],
                               outs, outb, [p[0] for p in dev_p], [p[1] for p in dev_p])
        for i, (st, x) in enumerate(zip(states, ins)):
            P = orc.step_kron_sched(st, x[0], x[1], x[2], x[3], update=(ra, rg), refresh=(ra, rg))
            Pg = np.concatenate([to_np(outs[i]), to_np(outb[i])[:, None]], axis=1)
            assert rel_fro(Pg, P) <= 1e-4, (t, i, rel_fro(Pg, P))
            Wg = np.concatenate([to_np(dev_p[i][0]), to_np(dev_p[i][1])[:, None]], axis=1)
            assert rel_fro(Wg, st.W) <= 1e-4, (t, i)
            assert rel_fro(to_np(h.state(i, K.KFAC_STATE_A)), st.A) <= 1e-5
            assert rel_fro(to_np(h.state(i, K.KFAC_STATE_G)), st.G) <= 1e-5
    assert h.get_status()[0] == 0


def test_skipped_factor_is_left_bitwise_and_ema_first_counts_per_factor():
    M, d, o = 200, 40, 24
    h = K.Kfac([(K.KFAC_KRON, o, d, 1, K.KFAC_F32)], max_rows=M,
               ema_init=K.KFAC_EMA_INIT_FIRST, **HP)
    a, g, _, _ = _draw(M, d, o)
    h.update_factors(0, to_dev(a), None)            # A's first update replaces it
    A1 = h.state(0, K.KFAC_STATE_A).clone()
    assert rel_fro(to_np(A1), O.factor(a, 1)) <= 1e-5
    assert not torch.any(h.state(0, K.KFAC_STATE_G))
    a2, g2, _, _ = _draw(M, d, o)
    h.update_factors(0, None, to_dev(g2))           # G's first update replaces it; A untouched
    assert torch.equal(h.state(0, K.KFAC_STATE_A), A1)
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_G)), O.factor(g2, 0)) <= 1e-5
    h.update_factors(0, to_dev(a2), None)           # A's second update is an EMA
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)),
                   0.9 * O.factor(a, 1) + 0.1 * O.factor(a2, 1)) <= 1e-5
    with pytest.raises(K.KfacError):
        h.update_factors(0, None, None, rows=M)
    # precondition needs both inverses
    with pytest.raises(K.KfacError) as e:
        h.precondition(0, torch.zeros(o, d, device="cuda"), torch.zeros(o, device="cuda"),
                       torch.empty(o, d, device="cuda"), torch.empty(o, device="cuda"))
    assert e.value.code == 3
    h.invert(0, which=K.KFAC_FACTOR_A)
    with pytest.raises(K.KfacError) as e:
        h.precondition(0, torch.zeros(o, d, device="cuda"), torch.zeros(o, device="cuda"),
                       torch.empty(o, d, device="cuda"), torch.empty(o, device="cuda"))
    assert e.value.code == 3
    Ainv = h.state(0, K.KFAC_STATE_AINV).clone()
    h.invert(0, which=K.KFAC_FACTOR_G)
    assert torch.equal(h.state(0, K.KFAC_STATE_AINV), Ainv)      # G refresh leaves A's inverse
    h.precondition(0, torch.zeros(o, d, device="cuda"), torch.zeros(o, device="cuda"),
                   torch.empty(o, d, device="cuda"), torch.empty(o, device="cuda"))
    with pytest.raises(K.KfacError):
        h.invert(0, which=0)
    assert h.get_status()[0] == 0


def test_conv_stale_input_leaves_factor_bitwise():
    h = K.Kfac([(K.KFAC_KRON, 8, 27, 1, K.KFAC_F32)], max_rows=2 * 36, **HP)
    x = torch.rand(2, 3, 6, 6, device="cuda")
    gy = torch.randn(2, 8, 6, 6, device="cuda")
    h.update_factors_conv2d(0, x, gy, 3, 1, 1)
    A1 = h.state(0, K.KFAC_STATE_A).clone()
    G1 = h.state(0, K.KFAC_STATE_G).clone()
    h.update_factors_conv2d(0, None, gy * 2, 3, 1, 1, in_shape=x.shape)
    assert torch.equal(h.state(0, K.KFAC_STATE_A), A1)
    assert not torch.equal(h.state(0, K.KFAC_STATE_G), G1)


def test_tied_a_factors_match_oracle():
    """Query, key and value projections fed the same input: one A, built and
    inverted once, preconditions all three."""
    M, d, o, T = 512, 96, 96, 4
    layers = [(K.KFAC_KRON, o, d, 1, K.KFAC_F32)] * 3 + [(K.KFAC_KRON, 2 * o, d, 1, K.KFAC_F32)]
    h = K.Kfac(layers, max_rows=M, **HP)
    h.tie_a_factor(1, 0)
    h.tie_a_factor(2, 0)
    h.tie_a_factor(3, 0)        # a different o, the same n: allowed
    orc = _orc()
    outs = [o, o, o, 2 * o]
    states, dev_p = [], []
    for oo in outs:
        w0, b0 = _params(oo, d)
        states.append(O.LayerState("kron", oo, d, 1, w0, b0))
        dev_p.append((to_dev(w0), to_dev(b0)))
    idx = [0, 1, 2, 3]
    launches = []
    for t in range(1, T + 1):
        a = np.maximum(RNG.standard_normal((M, d)), 0).astype(np.float32)
        gs = [(RNG.standard_normal((M, oo)) * 1e-2).astype(np.float32) for oo in outs]
        gws = [(RNG.standard_normal((oo, d)) * 1e-3).astype(np.float32) for oo in outs]
        gbs = [(RNG.standard_normal(oo) * 1e-3).astype(np.float32) for oo in outs]
        h.update_factors_batched(idx, [to_dev(a), None, None, None], [to_dev(g) for g in gs])
        n0 = K.launch_count()
        h.invert(-1)
        launches.append(K.launch_count() - n0)
        h.precondition_batched(idx, [to_dev(x) for x in gws], [to_dev(x) for x in gbs], None,
                               None, [p[0] for p in dev_p], [p[1] for p in dev_p])
        orc.step_kron_sched(states[0], a, gs[0], gws[0], gbs[0])
        for i in (1, 2, 3):
            orc.step_kron_sched(states[i], None, gs[i], gws[i], gbs[i], shared_a=states[0])
        for i in idx:
            Wg = np.concatenate([to_np(dev_p[i][0]), to_np(dev_p[i][1])[:, None]], axis=1)
            assert rel_fro(Wg, states[i].W) <= 1e-4, (t, i, rel_fro(Wg, states[i].W))
    for i in (1, 2, 3):
        assert h.state_info(i, K.KFAC_STATE_A) == h.state_info(0, K.KFAC_STATE_A)
        assert h.state_info(i, K.KFAC_STATE_AINV) == h.state_info(0, K.KFAC_STATE_AINV)
    assert h.get_status()[0] == 0


def test_tie_rules():
    L = (K.KFAC_KRON, 16, 32, 1, K.KFAC_F32)
    h = K.Kfac([L, L, L, (K.KFAC_KRON, 16, 31, 1, K.KFAC_F32), (K.KFAC_DIAG, 16, 32, 1,
                                                                K.KFAC_F32)],
               max_rows=64, **HP)
    # itself; different n; a DIAG layer either way; no such layer
    for layer, src in [(0, 0), (3, 0), (4, 0), (0, 4), (0, 9)]:
        with pytest.raises(K.KfacError) as e:
            h.tie_a_factor(layer, src)
        assert e.value.code == 1, (layer, src)
    h.tie_a_factor(1, 0)
    # source already tied; layer is a source; layer already tied
    for layer, src in [(2, 1), (0, 2), (1, 2)]:
        with pytest.raises(K.KfacError) as e:
            h.tie_a_factor(layer, src)
        assert e.value.code == 1, (layer, src)
    a = torch.rand(64, 32, device="cuda")
    g = torch.randn(64, 16, device="cuda")
    with pytest.raises(K.KfacError) as e:
        h.update_factors(1, a, g)               # a tied layer takes no a
    assert e.value.code == 1
    h.update_factors(1, None, g)
    h.update_factors(0, a, g)
    with pytest.raises(K.KfacError) as e:       # the source has state now: too late to tie
        h.tie_a_factor(2, 0)
    assert e.value.code == 3
    h.invert(1, which=K.KFAC_FACTOR_A)          # a tied layer has no A of its own: nothing to do
    h.invert(-1)
    h.precondition(1, torch.zeros(16, 32, device="cuda"), torch.zeros(16, device="cuda"),
                   torch.empty(16, 32, device="cuda"), torch.empty(16, device="cuda"))
    assert h.get_status()[0] == 0


def test_features_together_against_oracle():
    """One handle mixing the features: a convolution from NCHW tensors, two linear
    layers sharing one A, inverse-free refreshes, a stale A, a G-only Cholesky
    refresh, and a convolution on the diagonal path.  Six steps against the oracle."""
    gam = HP["damping"]
    B, C, H, Wd, o_c = 4, 6, 9, 9, 10                  # conv 3x3, pad 1: 324 rows, n = 55
    M, d, o = 324, 40, 24                               # two linear layers fed the same input
    layers = [(K.KFAC_KRON, o_c, C * 9, 1, K.KFAC_F32), (K.KFAC_KRON, o, d, 1, K.KFAC_F32),
              (K.KFAC_KRON, o, d, 1, K.KFAC_F32), (K.KFAC_DIAG, o_c, C * 9, 1, K.KFAC_F32)]
    h = K.Kfac(layers, max_rows=M, ikfac=1, **HP)
    h.tie_a_factor(2, 1)
    orc = _orc()
    shapes = [(o_c, C * 9), (o, d), (o, d), (o_c, C * 9)]
    st, dev_p = [], []
    for kind, (oo, dd) in zip(["kron", "kron", "kron", "diag"], shapes):
        w0, b0 = _params(oo, dd)
        st.append(O.LayerState(kind, oo, dd, 1, w0, b0))
        dev_p.append((to_dev(w0), to_dev(b0)))
    KA, KG = {}, {}
    gn = torch.empty(o_c, device="cuda")
    an = torch.empty(C * 9 + 1, device="cuda")
    for t in range(1, 7):
        x = np.maximum(RNG.standard_normal((B, C, H, Wd)), 0).astype(np.float32)
        gy = (RNG.standard_normal((B, o_c, H, Wd)) * 1e-2).astype(np.float32)
        a = np.maximum(RNG.standard_normal((M, d)), 0).astype(np.float32)
        g1, g2 = [(RNG.standard_normal((M, o)) * 1e-2).astype(np.float32) for _ in range(2)]
        grads = [((RNG.standard_normal((oo, dd)) * 1e-3).astype(np.float32),
                  (RNG.standard_normal(oo) * 1e-3).astype(np.float32)) for oo, dd in shapes]
        stale_a = t == 3                                 # A factors left as they are at step 3
        # --- GPU
        h.update_factors_conv2d(0, None if stale_a else to_dev(x), to_dev(gy), 3, 1, 1,
                                in_shape=x.shape)
        h.update_factors_batched([1, 2], [None if stale_a else to_dev(a), None],
                                 [to_dev(g1), to_dev(g2)])
        if t == 1:
            h.invert(-1)
        elif t == 4:
            h.invert(-1, which=K.KFAC_FACTOR_G)          # Cholesky for G; A keeps its K
        else:
            h.ikfac_update(-1, beta=1.0)
        h.precondition_batched([0, 1, 2], [to_dev(g[0]) for g in grads[:3]],
                               [to_dev(g[1]) for g in grads[:3]], None, None,
                               [p[0] for p in dev_p[:3]], [p[1] for p in dev_p[:3]])
        h.diag_factors_conv2d(3, to_dev(x), to_dev(gy), gn, an, 3, 1, 1)
        h.diag_step(3, gn, an, to_dev(grads[3][0]), to_dev(grads[3][1]), dev_p[3][0], dev_p[3][1])
        # --- oracle
        An_c, Gn_c = O.conv_factors(x, gy, (3, 3), (1, 1), (1, 1), (1, 1), 1)
        ins = {0: (An_c, Gn_c), 1: (O.factor(a, 1), O.factor(g1, 0)), 2: (None, O.factor(g2, 0))}
        for i in (0, 1, 2):
            s = st[i]
            if i != 2 and not stale_a:
                s.A = O.ema(s.A, ins[i][0], orc.xi)
            s.G = O.ema(s.G, ins[i][1], orc.xi)
        for i in (0, 1, 2):
            s, src = st[i], st[1] if i == 2 else st[i]
            if t == 1:
                if i != 2:
                    KA[i] = O.ikfac_init(s.A, gam)
                KG[i] = O.ikfac_init(s.G, gam)
            elif t == 4:
                KG[i] = O.ikfac_init(s.G, gam)
            else:
                if i != 2:
                    KA[i] = O.ikfac_update(KA[i], s.A, gam, 1.0)
                KG[i] = O.ikfac_update(KG[i], s.G, gam, 1.0)
        for i in (0, 1, 2):
            s = st[i]
            Ainv = O.ikfac_inverse(KA[1 if i == 2 else i])
            P = O.precondition(O.ikfac_inverse(KG[i]), O.grad_hat(*grads[i]), Ainv)
            s.W, s.m = O.momentum_update(P, s.W, s.m, orc.lr, orc.mu, orc.wd)
        gd, ad = O.conv_diag_factors(x, gy, (3, 3), (1, 1), (1, 1), (1, 1), 1)
        orc.step_diag(st[3], gd, ad, *grads[3])
        for i in range(4):
            Wg = np.concatenate([to_np(dev_p[i][0]), to_np(dev_p[i][1])[:, None]], axis=1)
            tol = 1e-4 if i < 3 else 1e-6
            assert rel_fro(Wg, st[i].W) <= tol, (t, i, rel_fro(Wg, st[i].W))
    assert h.get_status()[0] == 0
