"""ctypes declarations of libkfac's C ABI (include/kfac.h)."""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libkfac.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it with `python -c \"import __graft_entry__ as g; g.build()\"` "
        "(there is no CPU implementation of this library)")

LIB = ctypes.CDLL(LIB_PATH)

KFAC_KRON, KFAC_DIAG = 0, 1
KFAC_F32, KFAC_BF16 = 0, 1
KFAC_MATH_3XTF32, KFAC_MATH_BF16 = 0, 1
KFAC_EMA_INIT_ZERO, KFAC_EMA_INIT_FIRST = 0, 1
KFAC_IKFAC_OFF, KFAC_IKFAC_TF32, KFAC_IKFAC_BF16 = 0, 1, 2
KFAC_FACTOR_A, KFAC_FACTOR_G = 1, 2
(KFAC_STATE_A, KFAC_STATE_G, KFAC_STATE_AINV, KFAC_STATE_GINV, KFAC_STATE_MOMENTUM,
 KFAC_STATE_GDIAG, KFAC_STATE_ADIAG) = range(7)

STATUS_NAMES = {0: "KFAC_OK", 1: "KFAC_ERR_INVALID_ARG", 2: "KFAC_ERR_WORKSPACE",
                3: "KFAC_ERR_STATE", 4: "KFAC_ERR_NOT_PD", 5: "KFAC_ERR_TIMEOUT",
                6: "KFAC_ERR_CUDA", 7: "KFAC_ERR_UNSUPPORTED"}


class LayerDesc(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int), ("d_out", ctypes.c_int), ("d_in", ctypes.c_int),
                ("has_bias", ctypes.c_int), ("in_dtype", ctypes.c_int)]


class HParams(ctypes.Structure):
    _fields_ = [("ema_decay", ctypes.c_double), ("damping", ctypes.c_double),
                ("lr", ctypes.c_double), ("momentum", ctypes.c_double),
                ("weight_decay", ctypes.c_double), ("ema_init", ctypes.c_int),
                ("math", ctypes.c_int), ("ikfac", ctypes.c_int)]


class Conv2dGeom(ctypes.Structure):
    _fields_ = [(nm, ctypes.c_int) for nm in
                ("batch", "in_channels", "in_h", "in_w", "kernel_h", "kernel_w", "stride_h",
                 "stride_w", "pad_h", "pad_w", "dilation_h", "dilation_w")]


class KfacError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        msg = f"{what}: {STATUS_NAMES.get(code, code)} ({status_string(code)})"
        if STATUS_NAMES.get(code) == "KFAC_ERR_CUDA":
            msg += f": {LIB.kfac_last_cuda_error().decode()}"
        super().__init__(msg)


_vp, _i, _i64, _d, _sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_size_t
_pLD, _pHP = ctypes.POINTER(LayerDesc), ctypes.POINTER(HParams)
_pCG = ctypes.POINTER(Conv2dGeom)

# (name, restype, argtypes): one line per entry point of include/kfac.h
SIGNATURES = [
    ("kfac_workspace_size", _i, [_pLD, _i, _pHP, _i64, ctypes.POINTER(_sz)]),
    ("kfac_create", _i, [_pLD, _i, _pHP, _i64, _vp, _sz, ctypes.POINTER(_vp)]),
    ("kfac_set_hparams", _i, [_vp, _pHP]),
    ("kfac_update_factors", _i, [_vp, _i, _vp, _i64, _vp, _i64, _i64, _d, _vp]),
    ("kfac_update_factors_batched", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _d, _vp]),
    ("kfac_update_factors_conv2d", _i, [_vp, _i, _vp, _vp, _pCG, _d, _vp]),
    ("kfac_update_factors_conv2d_batched", _i, [_vp, _i, _vp, _vp, _vp, _pCG, _d, _vp]),
    ("kfac_diag_factors", _i, [_vp, _i, _vp, _i64, _vp, _i64, _i64, _d, _vp, _vp, _vp]),
    ("kfac_diag_factors_conv2d", _i, [_vp, _i, _vp, _vp, _pCG, _d, _vp, _vp, _vp]),
    ("kfac_diag_factors_batched", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _d, _vp, _vp,
                                       _vp]),
    ("kfac_invert", _i, [_vp, _i, _vp]),
    ("kfac_invert_factors", _i, [_vp, _i, _i, _vp]),
    ("kfac_ikfac_update", _i, [_vp, _i, _d, _vp]),
    ("kfac_tie_a_factor", _i, [_vp, _i, _i]),
    ("kfac_precondition", _i, [_vp, _i, _vp, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("kfac_precondition_batched", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("kfac_diag_step", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("kfac_diag_step_batched", _i, [_vp, _i, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                    _vp]),
    ("kfac_selftest_timeout", _i, [_vp, _i64, _vp]),
    ("kfac_get_status", _i, [_vp, ctypes.POINTER(_i), ctypes.POINTER(_i)]),
    ("kfac_state_info", _i, [_vp, _i, _i, ctypes.POINTER(_sz), ctypes.POINTER(_sz)]),
    ("kfac_destroy", _i, [_vp]),
    ("kfac_status_string", ctypes.c_char_p, [_i]),
    ("kfac_launch_count", ctypes.c_ulonglong, []),
    ("kfac_last_cuda_error", ctypes.c_char_p, []),
    ("kfac_diag_factors_static", _i, [_vp, _i64, _vp, _i64, _i64, _i, _i, _i, _i, _d, _vp, _vp,
                                      _vp]),
]

for _name, _res, _args in SIGNATURES:
    _f = getattr(LIB, _name)
    _f.restype = _res
    _f.argtypes = _args


def status_string(code: int) -> str:
    return LIB.kfac_status_string(code).decode()


def launch_count() -> int:
    return int(LIB.kfac_launch_count())
