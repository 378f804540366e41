"""GPU parity of the convolution factor update (input patches gathered from NCHW
tensors inside the library) against the float64 oracle's im2col factors.

Tolerances: factors A, G relative Frobenius 1e-5 (fp32 or bf16 inputs; the
oracle is fed the same rounded values), as for row-major inputs.  The gathered
path runs the same products as kfac_update_factors_batched on the unfolded
matrices, so the two must agree bit for bit.
"""
import ctypes

import numpy as np
import pytest

import oracle as O
import workloads as W
from gpu_helpers import to_dev, to_np, rel_fro, bf16_tensor

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import second_order_optimizer_gb300 as K  # noqa: E402

HP = dict(ema_decay=0.95, damping=1e-3, lr=1e-2, momentum=0.9, weight_decay=5e-4)
RNG = np.random.default_rng(11)

# (B, C, H, W, o, kh, kw, sh, sw, ph, pw, dh, dw, bias)
GEOMS = [
    (4, 3, 17, 13, 16, 3, 3, 1, 1, 1, 1, 1, 1, 1),     # ragged rows (884), 3 channels
    (2, 64, 16, 16, 64, 3, 3, 2, 2, 1, 1, 1, 1, 1),    # stride 2, n = 577, 128 rows
    (3, 5, 9, 11, 7, 3, 2, 2, 1, 2, 0, 2, 1, 0),       # dilation, asymmetric, no bias
    (8, 40, 8, 8, 33, 1, 1, 1, 1, 0, 0, 1, 1, 1),      # 1x1
    (2, 3, 30, 30, 8, 7, 7, 2, 2, 3, 3, 1, 1, 1),      # 7x7 stem, stride 2
    (1, 2, 1, 1, 3, 3, 3, 1, 1, 1, 1, 1, 1, 1),        # one pixel: every tap but the centre pads
    (16, 32, 20, 20, 48, 3, 3, 1, 1, 1, 1, 1, 1, 1),   # 6400 rows: many pack tiles
]


def _draw(B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, dtype):
    Ho = O.conv_out_size(H, kh, sh, ph, dh)
    Wo = O.conv_out_size(Wd, kw, sw, pw, dw)
    x = W.round_input(np.maximum(RNG.standard_normal((B, C, H, Wd)), 0), dtype)
    gy = W.round_input(RNG.standard_normal((B, o, Ho, Wo)) * 1e-3, dtype)
    return x, gy


def _dev(x, dtype):
    return bf16_tensor(x) if dtype == "bf16" else to_dev(x)


def _layer(geom, dtype):
    B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, bias = geom
    kd = K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32
    return (K.KFAC_KRON, o, C * kh * kw, bias, kd)


@pytest.mark.parametrize("geom", GEOMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_factors_match_oracle(geom, dtype):
    B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, bias = geom
    M = B * O.conv_out_size(H, kh, sh, ph, dh) * O.conv_out_size(Wd, kw, sw, pw, dw)
    h = K.Kfac([_layer(geom, dtype)], max_rows=M, **HP)
    A = np.zeros((C * kh * kw + bias,) * 2)
    G = np.zeros((o, o))
    for step in range(2):
        x, gy = _draw(B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, dtype)
        h.update_factors_conv2d(0, _dev(x, dtype), _dev(gy, dtype), (kh, kw), (sh, sw),
                                (ph, pw), (dh, dw))
        An, Gn = O.conv_factors(x, gy, (kh, kw), (sh, sw), (ph, pw), (dh, dw), bias)
        A, G = O.ema(A, An, 0.95), O.ema(G, Gn, 0.95)
        Ag, Gg = to_np(h.state(0, K.KFAC_STATE_A)), to_np(h.state(0, K.KFAC_STATE_G))
        assert rel_fro(Ag, A) <= 1e-5, (step, rel_fro(Ag, A))
        assert rel_fro(Gg, G) <= 1e-5, (step, rel_fro(Gg, G))
        assert np.array_equal(Ag, Ag.T) and np.array_equal(Gg, Gg.T)
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_gather_equals_unfolded_input_bitwise(dtype):
    """The gathered pack feeds the products exactly the values of the unfolded matrix."""
    geoms = [GEOMS[0], GEOMS[2], GEOMS[4]]
    layers = [_layer(g, dtype) for g in geoms]
    Ms, xs, gys, ref_a, ref_g, cg = [], [], [], [], [], []
    for g in geoms:
        B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, bias = g
        x, gy = _draw(B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, dtype)
        xs.append(_dev(x, dtype))
        gys.append(_dev(gy, dtype))
        cg.append(K.conv2d_geom(x.shape, (kh, kw), (sh, sw), (ph, pw), (dh, dw)))
        ref_a.append(_dev(O.im2col(x, (kh, kw), (sh, sw), (ph, pw), (dh, dw)).astype(np.float32),
                          dtype))
        ref_g.append(_dev(O.output_rows(gy).astype(np.float32), dtype))
        Ms.append(ref_a[-1].shape[0])
    h1 = K.Kfac(layers, max_rows=max(Ms), **HP)
    h2 = K.Kfac(layers, max_rows=max(Ms), **HP)
    idx = list(range(len(geoms)))
    for _ in range(2):
        h1.update_factors_conv2d_batched(idx, xs, gys, cg)
        h2.update_factors_batched(idx, ref_a, ref_g)
    torch.cuda.synchronize()
    for i in idx:
        for which in (K.KFAC_STATE_A, K.KFAC_STATE_G):
            assert torch.equal(h1.state(i, which), h2.state(i, which)), (i, which)


def test_conv_batched_matches_oracle_and_single_calls():
    geoms = [GEOMS[1], GEOMS[3], GEOMS[6]]
    layers = [_layer(g, "f32") for g in geoms]
    data = []
    for g in geoms:
        B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, bias = g
        x, gy = _draw(B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, "f32")
        data.append((x, gy, (kh, kw), (sh, sw), (ph, pw), (dh, dw), bias))
    M = max(O.im2col(d[0], *d[2:6]).shape[0] for d in data)
    hb = K.Kfac(layers, max_rows=M, **HP)
    hs = K.Kfac(layers, max_rows=M, **HP)
    xs = [to_dev(d[0]) for d in data]
    gys = [to_dev(d[1]) for d in data]
    hb.update_factors_conv2d_batched([0, 1, 2], xs, gys,
                                     [K.conv2d_geom(d[0].shape, *d[2:6]) for d in data])
    for i, d in enumerate(data):
        hs.update_factors_conv2d(i, xs[i], gys[i], *d[2:6])
    for i, d in enumerate(data):
        An, Gn = O.conv_factors(d[0], d[1], *d[2:6], d[6])
        for hh in (hb, hs):
            assert rel_fro(to_np(hh.state(i, K.KFAC_STATE_A)), 0.05 * An) <= 1e-5
            assert rel_fro(to_np(hh.state(i, K.KFAC_STATE_G)), 0.05 * Gn) <= 1e-5


def test_conv_rejects_bad_geometry():
    h = K.Kfac([(K.KFAC_KRON, 8, 27, 1, K.KFAC_F32), (K.KFAC_DIAG, 8, 27, 1, K.KFAC_F32)],
               max_rows=2 * 6 * 6, **HP)
    x = torch.zeros(2, 3, 6, 6, device="cuda")
    gy = torch.zeros(2, 8, 6, 6, device="cuda")
    ok = dict(kernel=3, stride=1, padding=1)
    h.update_factors_conv2d(0, x, gy, **ok)            # a valid call first
    bad = [
        (0, torch.zeros(2, 4, 6, 6, device="cuda"), gy, ok),     # C*kh*kw != d_in
        (0, x, gy, dict(kernel=3, stride=0, padding=1)),         # stride 0
        (0, x, gy, dict(kernel=3, stride=1, padding=-1)),        # negative pad
        (0, x, gy, dict(kernel=3, stride=1, padding=0, dilation=4)),  # no output position
        (0, torch.zeros(3, 3, 6, 6, device="cuda"), gy, ok),     # M = 108 > max_rows
        (1, x, gy, ok),                                          # a DIAG layer
        (5, x, gy, ok),                                          # no such layer
    ]
    for layer, xx, gg, kw in bad:
        with pytest.raises(K.KfacError) as e:
            h.update_factors_conv2d(layer, xx, gg, **kw)
        assert e.value.code == 1, (layer, kw)
    with pytest.raises(K.KfacError):
        h.update_factors_conv2d_batched([0, 0], [x, x], [gy, gy],
                                        [K.conv2d_geom(x.shape, 3, 1, 1)] * 2)
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("cfg_name,li,dtype", [("c3", 2, "f32"), ("c4bf16", 0, "bf16")])
def test_conv_full_size_layers_match_oracle(cfg_name, li, dtype):
    """A ResNet-18 stage-1 3x3 convolution (batch 128, 64 channels, 32 x 32: 131072
    rows, n = 577) and the ResNet-50 7x7 stem in bf16 (batch 32, 224 x 224, stride
    2: 401408 rows, n = 148) at full size, from NCHW draws, against the oracle."""
    cfg = W.get_config(cfg_name)
    L = cfg.layers[li]
    cg = L.conv
    d = W.conv_inputs(cfg, li, 1)
    h = K.Kfac([(K.KFAC_KRON, L.d_out, L.d_in, 1,
                 K.KFAC_BF16 if dtype == "bf16" else K.KFAC_F32)], max_rows=L.rows, **HP)
    h.update_factors_conv2d(0, _dev(d["x"], dtype), _dev(d["gy"], dtype), (cg.kh, cg.kw),
                            (cg.sh, cg.sw), (cg.ph, cg.pw), (cg.dh, cg.dw))
    An, Gn = O.conv_factors(d["x"], d["gy"], (cg.kh, cg.kw), (cg.sh, cg.sw), (cg.ph, cg.pw),
                            (cg.dh, cg.dw), 1)
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_A)), 0.05 * An) <= 1e-5
    assert rel_fro(to_np(h.state(0, K.KFAC_STATE_G)), 0.05 * Gn) <= 1e-5
    assert h.get_status()[0] == 0


@pytest.mark.parametrize("geom", GEOMS)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_conv_diag_factors_match_oracle(geom, dtype):
    """K5 from NCHW tensors: the diagonals of the convolution factors (elementwise
    1e-5, as for row-major inputs)."""
    from gpu_helpers import max_rel_elem
    B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, bias = geom
    M = B * O.conv_out_size(H, kh, sh, ph, dh) * O.conv_out_size(Wd, kw, sw, pw, dw)
    layer = _layer(geom, dtype)
    h = K.Kfac([(K.KFAC_DIAG,) + tuple(layer[1:])], max_rows=M, **HP)
    x, gy = _draw(B, C, H, Wd, o, kh, kw, sh, sw, ph, pw, dh, dw, dtype)
    gn = torch.empty(o, device="cuda")
    an = torch.empty(C * kh * kw + bias, device="cuda")
    for _ in range(2):   # twice: the ticket and partials are left ready for reuse
        h.diag_factors_conv2d(0, _dev(x, dtype), _dev(gy, dtype), gn, an, (kh, kw), (sh, sw),
                              (ph, pw), (dh, dw))
    g_ref, a_ref = O.conv_diag_factors(x, gy, (kh, kw), (sh, sw), (ph, pw), (dh, dw), bias)
    assert max_rel_elem(to_np(an), a_ref) <= 1e-5, max_rel_elem(to_np(an), a_ref)
    assert max_rel_elem(to_np(gn), g_ref) <= 1e-5, max_rel_elem(to_np(gn), g_ref)
    assert h.get_status()[0] == 0


def test_conv_diag_factors_full_size_stage1_layer():
    """A ResNet-18 stage-1 3x3 convolution (batch 128, 64 channels, 32 x 32) on the
    diagonal path, at full size."""
    from gpu_helpers import max_rel_elem
    cfg = W.get_config("c3")
    L = cfg.layers[2]
    cg = L.conv
    d = W.conv_inputs(cfg, 2, 1)
    h = K.Kfac([(K.KFAC_DIAG, L.d_out, L.d_in, 1, K.KFAC_F32)], max_rows=L.rows, **HP)
    gn = torch.empty(L.d_out, device="cuda")
    an = torch.empty(L.n, device="cuda")
    h.diag_factors_conv2d(0, to_dev(d["x"]), to_dev(d["gy"]), gn, an, (cg.kh, cg.kw),
                          (cg.sh, cg.sw), (cg.ph, cg.pw), (cg.dh, cg.dw))
    g_ref, a_ref = O.conv_diag_factors(d["x"], d["gy"], (cg.kh, cg.kw), (cg.sh, cg.sw),
                                       (cg.ph, cg.pw), (cg.dh, cg.dw), 1)
    assert max_rel_elem(to_np(an), a_ref) <= 1e-5
    assert max_rel_elem(to_np(gn), g_ref) <= 1e-5
    assert h.get_status()[0] == 0


def test_conv_diag_factors_large_kernel_and_limits():
    """Any kernel size (a 9 x 9 one against the oracle); an image beyond the
    shared-memory limit (240 x 240) is refused."""
    from gpu_helpers import max_rel_elem
    h = K.Kfac([(K.KFAC_DIAG, 4, 3 * 81, 1, K.KFAC_F32), (K.KFAC_DIAG, 4, 27, 1, K.KFAC_F32)],
               max_rows=2 * 240 * 240, **HP)
    x = torch.rand(2, 3, 10, 10, device="cuda")
    gy = torch.randn(2, 4, 10, 10, device="cuda")
    gn, an = torch.empty(4, device="cuda"), torch.empty(3 * 81 + 1, device="cuda")
    h.diag_factors_conv2d(0, x, gy, gn, an, 9, 1, 4)
    g_ref, a_ref = O.conv_diag_factors(to_np(x), to_np(gy), (9, 9), (1, 1), (4, 4), (1, 1), 1)
    assert max_rel_elem(to_np(an), a_ref) <= 1e-5 and max_rel_elem(to_np(gn), g_ref) <= 1e-5
    big = torch.zeros(2, 3, 240, 240, device="cuda")
    with pytest.raises(K.KfacError) as e:
        h.diag_factors_conv2d(1, big, torch.zeros(2, 4, 240, 240, device="cuda"), gn,
                              torch.empty(28, device="cuda"), 3, 1, 1)
    assert e.value.code == 7
    x = torch.zeros(2, 3, 10, 10, device="cuda")
    geom = K.conv2d_geom(x.shape, 3, 1, 1)                # no output gradient
    assert K.LIB.kfac_diag_factors_conv2d(h._h, 1, x.data_ptr(), None, ctypes.byref(geom), 0.0,
                                          gn.data_ptr(), an.data_ptr(), None) == 1
    assert h.get_status()[0] == 0
