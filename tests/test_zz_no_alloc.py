"""The workspace-free diagonal-factor entry point (kfac_diag_factors_static).

It exists for callers that cannot allocate device memory (no cudaMalloc and no
workspace of their own to hand over, e.g. code running under another
framework's allocator or inside a plug-in whose host owns every allocation).
Its scratch is a static device array inside the library.  These tests call it
through the C ABI and check it against the handle-based kfac_diag_factors and
against the float64 oracle on the same inputs, twice in a row, so that state the
shared array keeps between calls cannot leak into the next result; two more
cases reach the array's edges: the most row splits (one column block, rows
enough for four CTAs per SM) and the largest layer width it takes.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import oracle as O  # noqa: E402
import second_order_optimizer_gb300 as K  # noqa: E402
from second_order_optimizer_gb300._lib import LIB  # noqa: E402


def _max_rel(x, ref):
    x = x.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    return float(np.max(np.abs(x - ref) / np.maximum(np.abs(ref), 1e-30)))


CASES = [(3000, 257, 100, 1, "f32"), (2500, 640, 64, 1, "bf16"), (77, 5, 3, 0, "f32")]


def _static_call(a, g, M, d_in, o, bias, kd, gn, an):
    stream = torch.cuda.current_stream().cuda_stream
    return LIB.kfac_diag_factors_static(
        ctypes.c_void_p(a.data_ptr()), a.stride(0), ctypes.c_void_p(g.data_ptr()), g.stride(0),
        M, d_in, o, bias, kd, 0.0, ctypes.c_void_p(gn.data_ptr()), ctypes.c_void_p(an.data_ptr()),
        ctypes.c_void_p(stream))


def _oracle_err(gn, an, a, g, bias):
    """max elementwise relative error against the oracle's diagonal factors, formed
    from the same rounded inputs"""
    a64 = a.double().cpu().numpy()
    g64 = g.double().cpu().numpy()
    eg = _max_rel(gn, torch.from_numpy(O.diag_factor(g64, 0)))
    ea = _max_rel(an, torch.from_numpy(O.diag_factor(a64, bias)))
    return max(eg, ea)


def test_static_entry_point_matches_handle_entry_point_twice():
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        for M, d_in, o, bias, dt in CASES:
            tdt = torch.bfloat16 if dt == "bf16" else torch.float32
            kd = K.KFAC_BF16 if dt == "bf16" else K.KFAC_F32
            a = torch.randn(M, d_in, generator=gen, device="cuda").to(tdt)
            g = (torch.randn(M, o, generator=gen, device="cuda") * 1e-3).to(tdt)
            h = K.Kfac([(K.KFAC_DIAG, o, d_in, bias, kd)], max_rows=M)
            gn_ref = torch.empty(o, device="cuda")
            an_ref = torch.empty(d_in + bias, device="cuda")
            h.diag_factors(0, a, g, gn_ref, an_ref)
            gn = torch.full((o,), float("nan"), device="cuda")
            an = torch.full((d_in + bias,), float("nan"), device="cuda")
            rc = LIB.kfac_diag_factors_static(
                ctypes.c_void_p(a.data_ptr()), a.stride(0), ctypes.c_void_p(g.data_ptr()),
                g.stride(0), M, d_in, o, bias, kd, 0.0, ctypes.c_void_p(gn.data_ptr()),
                ctypes.c_void_p(an.data_ptr()), ctypes.c_void_p(stream))
            assert rc == 0, K.status_string(rc)
            torch.cuda.synchronize()
            # same tolerance as the diagonal-factor parity tests (factors: 1e-5)
            assert _max_rel(gn, gn_ref) <= 1e-5, (call, M, d_in, o)
            assert _max_rel(an, an_ref) <= 1e-5, (call, M, d_in, o)
            assert _oracle_err(gn, an, a, g, bias) <= 1e-5, (call, M, d_in, o)
            h.close()


@pytest.mark.parametrize("M,d_in,o", [(20000, 200, 56), (64, 200000, 62144)])
def test_static_entry_point_at_the_edges_of_its_array(M, d_in, o):
    """(20000, 200 + 56): one column block split over the most rows the array
    holds (four CTAs per SM); (64, 200000 + 62144): the widest layer it takes
    (d_in + d_out = 262144).  Both against the oracle, twice in a row."""
    gen = torch.Generator(device="cuda")
    gen.manual_seed(77)
    a = torch.randn(M, d_in, generator=gen, device="cuda")
    g = torch.randn(M, o, generator=gen, device="cuda") * 1e-3
    for call in range(2):
        gn = torch.full((o,), float("nan"), device="cuda")
        an = torch.full((d_in + 1,), float("nan"), device="cuda")
        rc = _static_call(a, g, M, d_in, o, 1, K.KFAC_F32, gn, an)
        assert rc == 0, K.status_string(rc)
        torch.cuda.synchronize()
        assert _oracle_err(gn, an, a, g, 1) <= 1e-5, (call, M, d_in, o)


def test_static_entry_point_rejects_oversize_and_bad_arguments():
    x = torch.zeros(4, 4, device="cuda")
    v = torch.zeros(8, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    # d_in + d_out beyond the static scratch: rejected before any launch
    rc = LIB.kfac_diag_factors_static(p(x), 300000, p(x), 4, 4, 300000, 4, 1, K.KFAC_F32, 0.0,
                                      p(v), p(v), None)
    assert rc == 2  # KFAC_ERR_WORKSPACE
    rc = LIB.kfac_diag_factors_static(None, 4, p(x), 4, 4, 4, 4, 1, K.KFAC_F32, 0.0, p(v), p(v),
                                      None)
    assert rc == 1
    rc = LIB.kfac_diag_factors_static(p(x), 4, p(x), 4, 0, 4, 4, 1, K.KFAC_F32, 0.0, p(v), p(v),
                                      None)
    assert rc == 1
