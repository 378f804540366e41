"""Python binding of libkfac (the GB300 Kronecker-factored optimizer step).

Argument marshalling only: every step of the optimizer runs in the library's
CUDA kernels.  Tensors supply device pointers; the stream is torch's current
stream unless one is given.  There is no CPU path: if the shared library is
missing, importing this package raises.

Function names follow the C ABI in include/kfac.h.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

from ._lib import (LIB, KFAC_KRON, KFAC_DIAG, KFAC_F32, KFAC_BF16, KFAC_MATH_3XTF32,
                   KFAC_IKFAC_OFF, KFAC_IKFAC_TF32, KFAC_IKFAC_BF16,
                   KFAC_FACTOR_A, KFAC_FACTOR_G,
                   KFAC_MATH_BF16, KFAC_EMA_INIT_ZERO, KFAC_EMA_INIT_FIRST, KFAC_STATE_A,
                   KFAC_STATE_G, KFAC_STATE_AINV, KFAC_STATE_GINV, KFAC_STATE_MOMENTUM,
                   KFAC_STATE_GDIAG, KFAC_STATE_ADIAG, LayerDesc, HParams, Conv2dGeom, KfacError,
                   status_string, launch_count)

__all__ = ["Kfac", "diag_factors_static", "conv2d_geom", "LayerDesc", "HParams", "Conv2dGeom",
           "KfacError", "status_string", "launch_count",
           "KFAC_KRON", "KFAC_DIAG", "KFAC_F32", "KFAC_BF16", "KFAC_MATH_3XTF32",
           "KFAC_MATH_BF16", "KFAC_EMA_INIT_ZERO", "KFAC_EMA_INIT_FIRST", "KFAC_FACTOR_A",
           "KFAC_IKFAC_OFF", "KFAC_IKFAC_TF32", "KFAC_IKFAC_BF16",
           "KFAC_FACTOR_G", "LIB"]


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _pair(v):
    return (int(v), int(v)) if isinstance(v, int) else (int(v[0]), int(v[1]))


def conv2d_geom(x_shape, kernel, stride=1, padding=0, dilation=1) -> Conv2dGeom:
    """kfac_conv2d_geom for an NCHW input of shape x_shape (int or pair arguments,
    as torch.nn.Conv2d takes them)."""
    B, C, H, W = (int(v) for v in x_shape)
    (kh, kw), (sh, sw), (ph, pw), (dh, dw) = (_pair(kernel), _pair(stride), _pair(padding),
                                              _pair(dilation))
    return Conv2dGeom(B, C, H, W, kh, kw, sh, sw, ph, pw, dh, dw)


def _check(code: int, what: str):
    if code != 0:
        raise KfacError(code, what)


class Kfac:
    """One handle over a workspace tensor that holds all optimizer state.

    ``layers``: sequence of (kind, d_out, d_in, has_bias, in_dtype) tuples or LayerDesc.
    """

    def __init__(self, layers: Sequence, ema_decay=0.95, damping=1e-3, lr=1e-2, momentum=0.9,
                 weight_decay=5e-4, ema_init=KFAC_EMA_INIT_ZERO, math=KFAC_MATH_3XTF32,
                 max_rows: int = 1, device=None, ikfac: int = 0):
        import torch
        descs = [l if isinstance(l, LayerDesc) else LayerDesc(*l) for l in layers]
        self.n_layers = len(descs)
        self._descs = (LayerDesc * self.n_layers)(*descs)
        self._hp = HParams(ema_decay, damping, lr, momentum, weight_decay, ema_init, math,
                           int(ikfac))
        self.max_rows = int(max_rows)
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        nbytes = ctypes.c_size_t(0)
        with torch.cuda.device(dev):   # the plan depends on the device's SM count
            _check(LIB.kfac_workspace_size(self._descs, self.n_layers, ctypes.byref(self._hp),
                                           self.max_rows, ctypes.byref(nbytes)),
                   "kfac_workspace_size")
        self.workspace_bytes = nbytes.value
        # 256-byte alignment: torch's caching allocator returns 512-byte aligned blocks
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=dev)
        self._h = ctypes.c_void_p()
        with torch.cuda.device(dev):
            _check(LIB.kfac_create(self._descs, self.n_layers, ctypes.byref(self._hp), self.max_rows,
                                   ctypes.c_void_p(self.workspace.data_ptr()),
                                   self.workspace_bytes, ctypes.byref(self._h)), "kfac_create")

    # -- lifecycle -----------------------------------------------------------
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            LIB.kfac_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def set_hparams(self, ema_decay=None, damping=None, lr=None, momentum=None,
                    weight_decay=None):
        hp = self._hp
        for name, v in (("ema_decay", ema_decay), ("damping", damping), ("lr", lr),
                        ("momentum", momentum), ("weight_decay", weight_decay)):
            if v is not None:
                setattr(hp, name, float(v))
        _check(LIB.kfac_set_hparams(self._h, ctypes.byref(hp)), "kfac_set_hparams")

    # -- the five verbs ---------------------------------------------------------
    def update_factors(self, layer: int, a, g, rows: Optional[int] = None, scale: float = 0.0,
                       stream=None, lda: Optional[int] = None, ldg: Optional[int] = None):
        """a or g may be None: that factor is left as it is."""
        rows = (a if a is not None else g).shape[0] if rows is None else rows
        lda = (a.stride(0) if a is not None else 0) if lda is None else lda
        ldg = (g.stride(0) if g is not None else 0) if ldg is None else ldg
        _check(LIB.kfac_update_factors(self._h, layer, _ptr(a), lda, _ptr(g), ldg, rows,
                                       float(scale), _stream(stream)), "kfac_update_factors")

    def update_factors_batched(self, layers, a_list, g_list, scale: float = 0.0, stream=None):
        """kfac_update_factors_batched over parallel lists of layers and input tensors
        (an entry of a_list or g_list may be None: that factor is left as it is)."""
        k = len(layers)
        I64 = ctypes.c_int64 * k
        P = ctypes.c_void_p * k
        st = lambda x: x.stride(0) if x is not None else 0
        rows = [(x if x is not None else y).shape[0] for x, y in zip(a_list, g_list)]
        _check(LIB.kfac_update_factors_batched(
            self._h, k, (ctypes.c_int * k)(*layers), P(*[_ptr(x) for x in a_list]),
            I64(*[st(x) for x in a_list]), P(*[_ptr(x) for x in g_list]),
            I64(*[st(x) for x in g_list]), I64(*rows),
            float(scale), _stream(stream)), "kfac_update_factors_batched")

    def update_factors_conv2d(self, layer: int, x, gy, kernel, stride=1, padding=0, dilation=1,
                              scale: float = 0.0, stream=None, in_shape=None):
        """kfac_update_factors_conv2d: x [B, C, H, W] and gy [B, o, Ho, Wo], both contiguous.
        Either may be None to leave that factor as it is; with x None the geometry
        takes the input's shape from in_shape."""
        geom = conv2d_geom(x.shape if x is not None else in_shape, kernel, stride, padding,
                           dilation)
        _check(LIB.kfac_update_factors_conv2d(self._h, layer, _ptr(x), _ptr(gy),
                                              ctypes.byref(geom), float(scale), _stream(stream)),
               "kfac_update_factors_conv2d")

    def update_factors_conv2d_batched(self, layers, x_list, gy_list, geoms, scale: float = 0.0,
                                      stream=None):
        """kfac_update_factors_conv2d_batched; geoms: Conv2dGeom per layer (see conv2d_geom)."""
        k = len(layers)
        P = ctypes.c_void_p * k
        _check(LIB.kfac_update_factors_conv2d_batched(
            self._h, k, (ctypes.c_int * k)(*layers), P(*[_ptr(x) for x in x_list]),
            P(*[_ptr(x) for x in gy_list]), (Conv2dGeom * k)(*geoms), float(scale),
            _stream(stream)), "kfac_update_factors_conv2d_batched")

    def diag_factors(self, layer: int, a, g, g_new, a_new, rows: Optional[int] = None,
                     scale: float = 0.0, stream=None):
        rows = a.shape[0] if rows is None else rows
        _check(LIB.kfac_diag_factors(self._h, layer, _ptr(a), a.stride(0), _ptr(g), g.stride(0),
                                     rows, float(scale), _ptr(g_new), _ptr(a_new),
                                     _stream(stream)), "kfac_diag_factors")

    def diag_factors_conv2d(self, layer: int, x, gy, g_new, a_new, kernel, stride=1, padding=0,
                            dilation=1, scale: float = 0.0, stream=None):
        """kfac_diag_factors_conv2d: x [B, C, H, W] and gy [B, o, Ho, Wo], both contiguous."""
        geom = conv2d_geom(x.shape, kernel, stride, padding, dilation)
        _check(LIB.kfac_diag_factors_conv2d(self._h, layer, _ptr(x), _ptr(gy), ctypes.byref(geom),
                                            float(scale), _ptr(g_new), _ptr(a_new),
                                            _stream(stream)), "kfac_diag_factors_conv2d")

    def diag_factors_batched(self, layers, a_list, g_list, g_new, a_new, scale: float = 0.0,
                             stream=None):
        """kfac_diag_factors_batched over parallel lists of layers, inputs and output vectors."""
        k = len(layers)
        I64 = ctypes.c_int64 * k
        P = ctypes.c_void_p * k
        _check(LIB.kfac_diag_factors_batched(
            self._h, k, (ctypes.c_int * k)(*layers), P(*[_ptr(x) for x in a_list]),
            I64(*[x.stride(0) for x in a_list]), P(*[_ptr(x) for x in g_list]),
            I64(*[x.stride(0) for x in g_list]), I64(*[x.shape[0] for x in a_list]),
            float(scale), P(*[_ptr(x) for x in g_new]), P(*[_ptr(x) for x in a_new]),
            _stream(stream)), "kfac_diag_factors_batched")

    def invert(self, layer: int = -1, stream=None, which: int = KFAC_FACTOR_A | KFAC_FACTOR_G):
        """kfac_invert, or kfac_invert_factors for which = KFAC_FACTOR_A or KFAC_FACTOR_G."""
        if which == KFAC_FACTOR_A | KFAC_FACTOR_G:
            _check(LIB.kfac_invert(self._h, layer, _stream(stream)), "kfac_invert")
        else:
            _check(LIB.kfac_invert_factors(self._h, layer, which, _stream(stream)),
                   "kfac_invert_factors")

    def ikfac_update(self, layer: int = -1, beta: float = 1.0, stream=None):
        """kfac_ikfac_update: one inverse-free step of the inverse factors (handle
        created with ikfac=KFAC_IKFAC_TF32 or KFAC_IKFAC_BF16); the layer's inverses
        become K K^T."""
        _check(LIB.kfac_ikfac_update(self._h, layer, float(beta), _stream(stream)),
               "kfac_ikfac_update")

    def tie_a_factor(self, layer: int, source: int):
        """kfac_tie_a_factor: layer uses source's A (same input); synchronous."""
        _check(LIB.kfac_tie_a_factor(self._h, layer, source), "kfac_tie_a_factor")

    def precondition(self, layer: int, grad_w, grad_b=None, out_w=None, out_b=None,
                     param_w=None, param_b=None, stream=None):
        _check(LIB.kfac_precondition(self._h, layer, _ptr(grad_w), grad_w.stride(0), _ptr(grad_b),
                                     _ptr(out_w), _ptr(out_b), _ptr(param_w), _ptr(param_b),
                                     _stream(stream)), "kfac_precondition")

    def precondition_batched(self, layers, grad_w, grad_b=None, out_w=None, out_b=None,
                             param_w=None, param_b=None, stream=None):
        """kfac_precondition_batched over parallel lists (None, or lists that may hold None)."""
        k = len(layers)
        P = ctypes.c_void_p * k
        arr = lambda xs: None if xs is None else P(*[_ptr(x) for x in xs])
        _check(LIB.kfac_precondition_batched(
            self._h, k, (ctypes.c_int * k)(*layers), arr(grad_w),
            (ctypes.c_int64 * k)(*[x.stride(0) for x in grad_w]), arr(grad_b), arr(out_w),
            arr(out_b), arr(param_w), arr(param_b), _stream(stream)), "kfac_precondition_batched")

    def diag_step(self, layer: int, g_new, a_new, grad_w, grad_b, param_w, param_b,
                  out_w=None, out_b=None, stream=None):
        _check(LIB.kfac_diag_step(self._h, layer, _ptr(g_new), _ptr(a_new), _ptr(grad_w),
                                  _ptr(grad_b), _ptr(param_w), _ptr(param_b), _ptr(out_w),
                                  _ptr(out_b), _stream(stream)), "kfac_diag_step")

    def diag_step_batched(self, layers, g_new, a_new, grad_w, grad_b, param_w, param_b,
                          out_w=None, out_b=None, stream=None):
        """kfac_diag_step_batched over parallel lists (None, or lists that may hold None)."""
        k = len(layers)
        P = ctypes.c_void_p * k
        arr = lambda xs: None if xs is None else P(*[_ptr(x) for x in xs])
        _check(LIB.kfac_diag_step_batched(
            self._h, k, (ctypes.c_int * k)(*layers), arr(g_new), arr(a_new), arr(grad_w),
            arr(grad_b), arr(param_w), arr(param_b), arr(out_w), arr(out_b), _stream(stream)),
            "kfac_diag_step_batched")

    # -- status and state --------------------------------------------------------
    def selftest_timeout(self, wait_cycles: int, stream=None):
        """kfac_selftest_timeout: a kernel whose bounded wait runs out; the status
        word then holds KFAC_ERR_TIMEOUT (read it with get_status)."""
        _check(LIB.kfac_selftest_timeout(self._h, int(wait_cycles), _stream(stream)),
               "kfac_selftest_timeout")

    def get_status(self):
        """Synchronises; returns (code, layer, info) of the first device error (code 0: none)."""
        layer, info = ctypes.c_int(-1), ctypes.c_int(0)
        code = LIB.kfac_get_status(self._h, ctypes.byref(layer), ctypes.byref(info))
        return code, layer.value, info.value

    def state_info(self, layer: int, which: int):
        off, nb = ctypes.c_size_t(0), ctypes.c_size_t(0)
        _check(LIB.kfac_state_info(self._h, layer, which, ctypes.byref(off), ctypes.byref(nb)),
               "kfac_state_info")
        return off.value, nb.value

    def state(self, layer: int, which: int):
        """A float32 view of one piece of layer state inside the workspace (no copy)."""
        import torch
        off, nb = self.state_info(layer, which)
        d = self._descs[layer]
        n = d.d_in + d.has_bias
        v = self.workspace[off:off + nb].view(torch.float32)
        shapes = {KFAC_STATE_A: (n, n), KFAC_STATE_G: (d.d_out, d.d_out),
                  KFAC_STATE_AINV: (n, n), KFAC_STATE_GINV: (d.d_out, d.d_out),
                  KFAC_STATE_GDIAG: (d.d_out,), KFAC_STATE_ADIAG: (n,)}
        if which == KFAC_STATE_MOMENTUM:
            return v  # [o*d_in] weight part then [o] bias part
        return v.view(*shapes[which])

    def momentum(self, layer: int):
        """(m_w [o, d_in], m_b [o] or None) views of the momentum buffer."""
        d = self._descs[layer]
        v = self.state(layer, KFAC_STATE_MOMENTUM)
        mw = v[:d.d_out * d.d_in].view(d.d_out, d.d_in)
        mb = v[d.d_out * d.d_in:] if d.has_bias else None
        return mw, mb


def diag_factors_static(a, g, g_new, a_new, has_bias: int = 1, rows: Optional[int] = None,
                        scale: float = 0.0, stream=None):
    """kfac_diag_factors_static: the diagonal factors of one layer without a handle or
    workspace (for callers that cannot allocate device memory; see include/kfac.h)."""
    import torch
    rows = a.shape[0] if rows is None else rows
    dt = KFAC_BF16 if a.dtype == torch.bfloat16 else KFAC_F32
    _check(LIB.kfac_diag_factors_static(_ptr(a), a.stride(0), _ptr(g), g.stride(0), rows,
                                        a.shape[1], g.shape[1], has_bias, dt, float(scale),
                                        _ptr(g_new), _ptr(a_new), _stream(stream)),
           "kfac_diag_factors_static")
