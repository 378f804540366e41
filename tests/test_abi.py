"""CPU checks of the C ABI: the library loads, exports every declared entry point,
and the host-only calls (sizing, argument checks, status strings) behave.
No compute call is made here (there is no GPU on this side)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kfac.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import second_order_optimizer_gb300._lib as L
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(kfac_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_five_verbs():
    names = declared_functions()
    for verb in ("kfac_create", "kfac_update_factors", "kfac_invert", "kfac_precondition",
                 "kfac_diag_step"):
        assert verb in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib.LIB, n), n
    # and the binding declares a signature for each
    assert {s[0] for s in lib.SIGNATURES} >= set(names)


def test_binding_covers_exactly_the_header(lib):
    assert {s[0] for s in lib.SIGNATURES} == set(declared_functions())


def _descs(lib, layers):
    arr = (lib.LayerDesc * len(layers))(*[lib.LayerDesc(*l) for l in layers])
    return arr


def _hp(lib, **kw):
    d = dict(ema_decay=0.95, damping=1e-3, lr=1e-2, momentum=0.9, weight_decay=5e-4,
             ema_init=0, math=0)
    d.update(kw)
    return lib.HParams(**d)


def test_workspace_size_grows_with_layers(lib):
    hp = _hp(lib)
    out = ctypes.c_size_t(0)
    small = _descs(lib, [(0, 32, 64, 1, 0)])
    assert lib.LIB.kfac_workspace_size(small, 1, ctypes.byref(hp), 128, ctypes.byref(out)) == 0
    s1 = out.value
    assert s1 % 256 == 0
    # at least the fp32 state: A, G, Ainv, Ginv, m
    n, o = 65, 32
    assert s1 >= 4 * (2 * n * n + 2 * o * o + o * n)
    big = _descs(lib, [(0, 32, 64, 1, 0), (1, 1024, 1024, 1, 0)])
    assert lib.LIB.kfac_workspace_size(big, 2, ctypes.byref(hp), 128, ctypes.byref(out)) == 0
    assert out.value > s1 + 4 * 1024 * 1025


def test_workspace_size_rejects_bad_arguments(lib):
    hp = _hp(lib)
    out = ctypes.c_size_t(0)
    bad = [
        ([(0, 0, 64, 1, 0)], hp),            # d_out = 0
        ([(0, 4, 0, 1, 0)], hp),             # d_in = 0
        ([(2, 4, 4, 1, 0)], hp),             # kind
        ([(0, 4, 4, 2, 0)], hp),             # has_bias
        ([(0, 4, 4, 1, 5)], hp),             # dtype
        ([(0, 4, 4, 1, 0)], _hp(lib, ema_decay=1.0)),
        ([(0, 4, 4, 1, 0)], _hp(lib, damping=0.0)),
        ([(0, 4, 4, 1, 0)], _hp(lib, damping=float("nan"))),
        ([(0, 4, 4, 1, 0)], _hp(lib, math=7)),
        ([(0, 4, 4, 1, 0)], _hp(lib, ikfac=3)),
    ]
    for layers, h in bad:
        d = _descs(lib, layers)
        assert lib.LIB.kfac_workspace_size(d, 1, ctypes.byref(h), 16, ctypes.byref(out)) == 1
    d = _descs(lib, [(0, 4, 4, 1, 0)])
    assert lib.LIB.kfac_workspace_size(d, 0, ctypes.byref(hp), 16, ctypes.byref(out)) == 1
    assert lib.LIB.kfac_workspace_size(d, 1, ctypes.byref(hp), 0, ctypes.byref(out)) == 1


def test_null_handle_calls_fail_cleanly(lib):
    L = lib.LIB
    assert L.kfac_invert(None, -1, None) == 1
    assert L.kfac_destroy(None) == 1
    assert L.kfac_get_status(None, None, None) == 1
    assert L.kfac_update_factors(None, 0, None, 1, None, 1, 1, 0.0, None) == 1
    geom = lib.Conv2dGeom(1, 1, 3, 3, 3, 3, 1, 1, 1, 1, 1, 1)
    assert L.kfac_update_factors_conv2d(None, 0, None, None, ctypes.byref(geom), 0.0, None) == 1
    assert L.kfac_update_factors_conv2d(None, 0, None, None, None, 0.0, None) == 1
    assert L.kfac_selftest_timeout(None, 1000, None) == 1
    assert L.kfac_invert_factors(None, -1, 3, None) == 1
    assert L.kfac_tie_a_factor(None, 1, 0) == 1
    assert L.kfac_precondition(None, 0, None, 1, None, None, None, None, None, None) == 1
    assert L.kfac_diag_step(None, 0, None, None, None, None, None, None, None, None, None) == 1


def test_create_rejects_small_or_misaligned_workspace(lib):
    hp = _hp(lib)
    d = _descs(lib, [(0, 8, 8, 1, 0)])
    h = ctypes.c_void_p()
    # too small: rejected before touching the device
    assert lib.LIB.kfac_create(d, 1, ctypes.byref(hp), 16, ctypes.c_void_p(0x1000), 16,
                               ctypes.byref(h)) == 2
    assert lib.LIB.kfac_create(d, 1, ctypes.byref(hp), 16, ctypes.c_void_p(0x1001), 1 << 30,
                               ctypes.byref(h)) == 2
    assert h.value is None


def test_status_strings(lib):
    for code in range(8):
        s = lib.status_string(code)
        assert isinstance(s, str) and s
    assert lib.status_string(0) == "ok"


def test_package_refuses_to_load_without_the_library(tmp_path):
    """No CPU fallback: a copy of the package without libkfac.so fails to import."""
    import shutil
    import subprocess
    import sys
    pkg = os.path.join(ROOT, "second_order_optimizer_gb300")
    dst = tmp_path / "second_order_optimizer_gb300"
    dst.mkdir()
    for f in ("__init__.py", "_lib.py"):
        shutil.copy(os.path.join(pkg, f), dst / f)
    r = subprocess.run([sys.executable, "-c", "import second_order_optimizer_gb300"],
                       cwd=tmp_path, capture_output=True, text=True)
    assert r.returncode != 0
    assert "libkfac.so is missing" in r.stderr


def test_workspace_holds_the_inverse_factors_when_asked(lib):
    """ikfac = 1 adds the inverse factors and their scratch: 8 arrays of n x np
    floats per n x n factor (np = n rounded up to 4)."""
    d = _descs(lib, [(0, 100, 299, 1, 0)])            # A: 300 x 300, G: 100 x 100
    out0, out1 = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert lib.LIB.kfac_workspace_size(d, 1, ctypes.byref(_hp(lib)), 64, ctypes.byref(out0)) == 0
    assert lib.LIB.kfac_workspace_size(d, 1, ctypes.byref(_hp(lib, ikfac=1)), 64,
                                       ctypes.byref(out1)) == 0
    want = 8 * 4 * (300 * 300 + 100 * 100)
    assert want <= out1.value - out0.value <= want + 16 * 256


def test_header_is_plain_c(tmp_path):
    """include/kfac.h compiles as C99 (no C++ in the boundary): its structs and
    enums initialise and a declared function is called from a C translation unit."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    cuda_inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    if not cc or not os.path.exists(os.path.join(cuda_inc, "cuda_runtime_api.h")):
        pytest.skip("no C compiler or CUDA headers")
    src = tmp_path / "use_kfac.c"
    src.write_text('#include "kfac.h"\n'
                   "int main(void) {\n"
                   "  kfac_conv2d_geom g = {1, 1, 3, 3, 3, 3, 1, 1, 1, 1, 1, 1};\n"
                   "  kfac_hparams hp = {0.95, 1e-3, 1e-2, 0.9, 5e-4, KFAC_EMA_INIT_ZERO,\n"
                   "                     KFAC_MATH_3XTF32, 0};\n"
                   "  (void)g; (void)hp;\n"
                   "  return (int)kfac_launch_count();\n"
                   "}\n")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror=implicit-function-declaration",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, "-fsyntax-only",
                        str(src)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
