"""Full-size parity: the ResNet-18 (CIFAR), ResNet-50 (fp32 and bf16 inputs) and
transformer-block layer sets.

Gate (`test_widest_layers_match_the_oracle_step`): for each set's widest A and
widest G layer, one K-FAC step on the GPU (factor update, refresh, precondition
with the fused update) against the float64 oracle's own step on the same
rounded inputs -- the oracle builds A and G from the inputs, inverts them with
its textbook Cholesky and substitutions, and forms P, m and W.  Every element is
compared: factors <= 1e-5 and P, m, W <= 1e-4 relative Frobenius.  The handle
starts its running factors from the first update (EMA-first), so the factors
carry their full spread and cond(F + sqrt(gamma) I) is the largest the layer
reaches; it is printed beside each error.

Whole sets (`test_full_layer_set`): every layer through one handle exactly as
the benchmark calls the library, two steps with one refresh:
  * factor entries are sampled and each one is formed by the oracle's own
    `factor` on the two columns it involves; the whole factor must be exactly
    symmetric;
  * preconditioned gradients: sampled rows of P against the oracle's
    precondition() applied to the inverses in use (a check of the K4 products
    at full size given their inputs; the inverses themselves are gated above);
  * diagonal-path elements (K5 columns, K6 m and W entries) are sampled and
    formed one by one by the oracle, K6 to 1e-6 componentwise.
"""
import math

import numpy as np
import pytest

import oracle as O
import workloads as W

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import second_order_optimizer_gb300 as K  # noqa: E402

NS = 24  # sampled entries per factor


def _np(t):
    return t.detach().double().cpu().numpy()


def _handle(cfg):
    hp = cfg.hp
    descs = [(K.KFAC_KRON if l.kind == "kron" else K.KFAC_DIAG, l.d_out, l.d_in, l.has_bias,
              K.KFAC_BF16 if l.in_dtype == "bf16" else K.KFAC_F32) for l in cfg.layers]
    return K.Kfac(descs, ema_decay=hp.ema_decay, damping=hp.damping, lr=hp.lr,
                  momentum=hp.momentum, weight_decay=hp.weight_decay,
                  max_rows=max(l.rows for l in cfg.layers))


def _sample_pairs(n, rng, has_bias):
    pairs = [(0, 0), (n - 1, n - 1), (0, n - 1)]
    if has_bias:
        pairs += [(int(rng.integers(0, n - 1)), n - 1) for _ in range(3)]
    pairs += [(int(i), int(i)) for i in rng.integers(0, n, 4)]
    while len(pairs) < NS:
        i, j = sorted(int(v) for v in rng.integers(0, n, 2))
        pairs.append((i, j))
    return pairs


def _check_factor(F_gpu, x, has_bias, decay_weight, rng, tag):
    """Sampled entries of the factor against the oracle, each formed from its two columns."""
    n = F_gpu.shape[0]
    pairs = _sample_pairs(n, rng, has_bias)
    d = x.shape[1]
    cols = sorted({c for p in pairs for c in p if c < d})
    sub = _np(x[:, cols])                         # the oracle reads the same rounded inputs
    pos = {c: k for k, c in enumerate(cols)}
    Fs = _np(F_gpu)
    worst = 0.0
    for i, j in pairs:
        ci = [pos[c] for c in (i, j) if c < d]
        xi = sub[:, sorted(set(ci))]
        Fo = O.factor(xi, has_bias if (i >= d or j >= d) else 0)
        # map (i, j) into the small factor
        idx = {c: k for k, c in enumerate(sorted({c for c in (i, j) if c < d}))}
        ii = idx[i] if i < d else Fo.shape[0] - 1
        jj = idx[j] if j < d else Fo.shape[0] - 1
        ref = decay_weight * Fo[ii, jj]
        di = decay_weight * (Fo[ii, ii])
        dj = decay_weight * (Fo[jj, jj])
        err = abs(Fs[i, j] - ref) / max(math.sqrt(di * dj), 1e-30)
        worst = max(worst, err)
    assert worst <= 1e-5, (tag, worst)
    assert np.array_equal(Fs, Fs.T), tag


def _run_config(name, steps=2):
    """The whole layer set for `steps` steps, as the benchmark runs it; the inverses are
    refreshed after the step-1 factor update.  Checked on sampled elements:
      K4: P rows against the oracle's precondition() with the inverses in use;
      K5: diagonal factors, one column at a time by the oracle;
      K6: m and W elements, from the same fp32 state, by the oracle's step formulas."""
    cfg = W.get_config(name)
    hp = cfg.hp
    dev = torch.device("cuda")
    h = _handle(cfg)
    rng = np.random.default_rng(99)
    params = [W.initial_params_torch(cfg, li, dev) for li in range(len(cfg.layers))]
    report = {"precond": 0.0, "diag_step": 0.0, "diag_factor": 0.0}
    kron = [i for i, l in enumerate(cfg.layers) if l.kind == "kron"]
    tallest = max(kron, key=lambda i: (cfg.layers[i].rows, cfg.layers[i].n))
    for t in range(1, steps + 1):
        grads = {}
        for li, l in enumerate(cfg.layers):
            x = W.layer_inputs_torch(cfg, li, t, dev)
            if l.kind == "kron":
                h.update_factors(li, x["a"], x["g"])
                grads[li] = (x["grad_w"], x["grad_b"])
                if t == 1 and li == tallest:   # longest reduction: sampled entries
                    w1 = 1 - hp.ema_decay
                    _check_factor(h.state(li, K.KFAC_STATE_A), x["a"], l.has_bias, w1, rng,
                                  (name, l.name, "A"))
                    _check_factor(h.state(li, K.KFAC_STATE_G), x["g"], 0, w1, rng,
                                  (name, l.name, "G"))
                continue
            pw, pb = params[li]
            if l.act == "bn":
                gn, an = x["g_new"], x["a_new"]
            else:
                gn = torch.empty(l.d_out, device=dev)
                an = torch.empty(l.n, device=dev)
                h.diag_factors(li, x["a"], x["g"], gn, an)
                for c in sorted({0, l.d_in - 1, int(rng.integers(0, l.d_in))}):
                    ref = O.diag_factor(_np(x["a"][:, c:c + 1]), 0)[0]
                    e = abs(_np(an[c:c + 1])[0] - ref) / ref
                    report["diag_factor"] = max(report["diag_factor"], e)
                    assert e <= 1e-5, (name, l.name, c, e)
                c = int(rng.integers(0, l.d_out))
                ref = O.diag_factor(_np(x["g"][:, c:c + 1]), 0)[0]
                e = abs(_np(gn[c:c + 1])[0] - ref) / ref
                assert e <= 1e-5, (name, l.name, "g", e)
            gs0 = _np(h.state(li, K.KFAC_STATE_GDIAG))
            as0 = _np(h.state(li, K.KFAC_STATE_ADIAG))
            mw, _ = h.momentum(li)
            rows = rng.integers(0, l.d_out, 4)
            cols = rng.integers(0, l.d_in, 4)
            w0, m0 = _np(pw[rows][:, cols]), _np(mw[rows][:, cols])
            gw = _np(x["grad_w"][rows][:, cols])
            gnn, ann = _np(gn), _np(an)
            h.diag_step(li, gn, an, x["grad_w"], x["grad_b"], pw, pb)
            gs = O.ema(gs0, gnn, hp.ema_decay)
            as_ = O.ema(as0, ann, hp.ema_decay)
            P = O.diag_precondition(gw, gs[rows], as_[cols], hp.damping)
            Wn, mn = O.momentum_update(P, w0, m0, hp.lr, hp.momentum, hp.weight_decay)
            mw, _ = h.momentum(li)
            scale_m = hp.momentum * np.abs(m0) + np.abs(P) + hp.weight_decay * np.abs(w0)
            e = max(np.max(np.abs(_np(mw[rows][:, cols]) - mn) / scale_m),
                    np.max(np.abs(_np(pw[rows][:, cols]) - Wn) / (np.abs(w0) + hp.lr * scale_m)))
            report["diag_step"] = max(report["diag_step"], float(e))
            assert e <= 1e-6, (name, l.name, e)
        if t == 1:
            h.invert(-1)
        for li, (gw_t, gb_t) in grads.items():
            l = cfg.layers[li]
            pw, pb = params[li]
            ow = torch.empty(l.d_out, l.d_in, device=dev)
            ob = torch.empty(l.d_out, device=dev)
            h.precondition(li, gw_t, gb_t, ow, ob, pw, pb)
            A, G = h.state(li, K.KFAC_STATE_A), h.state(li, K.KFAC_STATE_G)
            assert torch.equal(A, A.T) and torch.equal(G, G.T)
            if t != steps:
                continue
            rows = sorted(set(int(v) for v in rng.integers(0, l.d_out, 3)))
            Pref = O.precondition(_np(h.state(li, K.KFAC_STATE_GINV)[rows]),
                                  O.grad_hat(_np(gw_t), _np(gb_t)),
                                  _np(h.state(li, K.KFAC_STATE_AINV)))
            Pgot = O.grad_hat(_np(ow[rows]), _np(ob[rows]))
            e = np.linalg.norm(Pgot - Pref) / np.linalg.norm(Pref)
            report["precond"] = max(report["precond"], float(e))
            assert e <= 1e-4, (name, l.name, e)
    return h, report


def _cond2(Fd, Finv, iters=60):
    """2-norm condition number of the SPD matrix Fd from power iterations on Fd and on
    its inverse (the oracle's)."""
    rng = np.random.default_rng(5)

    def top(M):
        v = rng.standard_normal(M.shape[0])
        lam = 0.0
        for _ in range(iters):
            w = M @ v
            lam = float(np.linalg.norm(w))
            v = w / lam
        return lam
    return top(Fd) * top(Finv)


def _gate_layer(cfg, li):
    """One step of layer li alone on the GPU (EMA-first) against the oracle's step."""
    l = cfg.layers[li]
    hp = cfg.hp
    dev = torch.device("cuda")
    h = K.Kfac([(K.KFAC_KRON, l.d_out, l.d_in, l.has_bias,
                 K.KFAC_BF16 if l.in_dtype == "bf16" else K.KFAC_F32)],
               ema_decay=hp.ema_decay, damping=hp.damping, lr=hp.lr, momentum=hp.momentum,
               weight_decay=hp.weight_decay, ema_init=K.KFAC_EMA_INIT_FIRST, max_rows=l.rows)
    x = W.layer_inputs_torch(cfg, li, 1, dev)
    pw, pb = W.initial_params_torch(cfg, li, dev)
    w0, b0 = _np(pw), (_np(pb) if pb is not None else None)
    h.update_factors(0, x["a"], x["g"])
    h.invert(0)
    ow = torch.empty(l.d_out, l.d_in, device=dev)
    ob = torch.empty(l.d_out, device=dev) if l.has_bias else None
    h.precondition(0, x["grad_w"], x["grad_b"], ow, ob, pw, pb)
    torch.cuda.synchronize()
    assert h.get_status()[0] == 0
    got = {"A": _np(h.state(0, K.KFAC_STATE_A)), "G": _np(h.state(0, K.KFAC_STATE_G)),
           "Ainv": _np(h.state(0, K.KFAC_STATE_AINV)), "Ginv": _np(h.state(0, K.KFAC_STATE_GINV)),
           "P": O.grad_hat(_np(ow), _np(ob) if ob is not None else None),
           "W": O.grad_hat(_np(pw), _np(pb) if pb is not None else None)}
    mw, mb = h.momentum(0)
    got["m"] = O.grad_hat(_np(mw), _np(mb) if mb is not None else None)
    h.close()
    del h, mw, mb
    # the oracle's step on the same rounded inputs (promoted to float64)
    orc = O.KfacOracle(hp.ema_decay, hp.damping, hp.lr, hp.momentum, hp.weight_decay, 1,
                       ema_init="first")
    st = O.LayerState("kron", l.d_out, l.d_in, l.has_bias, w0, b0)
    a, g = _np(x["a"]), _np(x["g"])
    gw, gb = _np(x["grad_w"]), (_np(x["grad_b"]) if x["grad_b"] is not None else None)
    del x
    torch.cuda.empty_cache()
    P = orc.step_kron(st, a, g, gw, gb)
    del a, g
    rel = lambda k, ref: float(np.linalg.norm(got[k] - ref) / np.linalg.norm(ref))
    sg = math.sqrt(hp.damping)
    res = {"layer": l.name, "n": l.n, "o": l.d_out, "rows": l.rows,
           "cond_A": _cond2(O.damped(st.A, hp.damping), st.Ainv),
           "cond_G": _cond2(O.damped(st.G, hp.damping), st.Ginv),
           "A": rel("A", st.A), "G": rel("G", st.G), "Ainv": rel("Ainv", st.Ainv),
           "Ginv": rel("Ginv", st.Ginv), "P": rel("P", P), "m": rel("m", st.m),
           "W": rel("W", st.W)}
    del sg
    return res


def _gate_layers(cfg):
    kron = [i for i, l in enumerate(cfg.layers) if l.kind == "kron"]
    widest_a = max(kron, key=lambda i: (cfg.layers[i].n, cfg.layers[i].rows))
    widest_g = max(kron, key=lambda i: (cfg.layers[i].d_out, cfg.layers[i].rows))
    return sorted({widest_a, widest_g})


@pytest.mark.parametrize("name", ["c3", "c4", "c4bf16", "c5"])
def test_widest_layers_match_the_oracle_step(name):
    cfg = W.get_config(name)
    for li in _gate_layers(cfg):
        r = _gate_layer(cfg, li)
        print(name, {k: (f"{v:.3g}" if isinstance(v, float) else v) for k, v in r.items()})
        assert r["A"] <= 1e-5 and r["G"] <= 1e-5, (name, r)
        assert r["P"] <= 1e-4 and r["m"] <= 1e-4 and r["W"] <= 1e-4, (name, r)


@pytest.mark.parametrize("name", ["c3", "c4", "c4bf16", "c5"])
def test_full_layer_set(name):
    h, report = _run_config(name)
    assert h.get_status()[0] == 0
    print(name, report)
