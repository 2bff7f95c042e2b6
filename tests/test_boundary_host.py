"""Host-side checks of the C ABI: the library loads, exports every declared
symbol, validates arguments before touching the GPU, and reports injected
failures.  None of these tests needs a GPU."""
import os
import re

import pytest

from fft_gemm_ifft_gb300 import capi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
F32, F16 = capi.FNO_F32, capi.FNO_F16


@pytest.fixture(scope="module")
def L():
    from fft_gemm_ifft_gb300 import build
    build.build()
    return capi.lib()


def declared_functions():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fno_\w+)\s*\(", text))
    return names


def test_exports_every_declared_symbol(L):
    decl = declared_functions()
    assert decl, "no declarations found"
    for name in decl:
        assert hasattr(L, name), f"libfno.so does not export {name}"
    assert set(capi.EXPORTS) == decl


def test_status_strings(L):
    for code in range(0, 9):
        s = capi.fno_status_string(code)
        assert s.startswith("FNO_")
    assert "UNKNOWN" in capi.fno_status_string(99)
    assert capi.fno_version() >= 10000


Q = capi.fno_spectral_conv_query


@pytest.mark.parametrize("args,wbytes", [
    ((1, [256], [16], 4, 16, 16, F32), 1 * 16 * 16 * 16 * 8),
    ((2, [128, 128], [16, 16], 8, 32, 32, F32), 2 * 32 * 32 * 256 * 8),
    ((2, [256, 256], [32, 32], 32, 64, 64, F16), 2 * 64 * 64 * 1024 * 4),
    ((2, [256, 256], [32, 32], 32, 64, 64, capi.FNO_BF16), 2 * 64 * 64 * 1024 * 4),
    ((3, [64, 64, 64], [16, 16, 16], 4, 32, 32, F32), 4 * 32 * 32 * 4096 * 8),
    ((2, [8, 8], [4, 5], 1, 1, 1, F32), 2 * 1 * 1 * 20 * 8),     # all modes, Nyquist kept
])
def test_query_valid(L, args, wbytes):
    st, ws, wb = Q(*args)
    assert st == capi.FNO_OK
    assert wb == wbytes


@pytest.mark.parametrize("args,code", [
    ((0, [8], [2], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),           # rank 0
    ((4, [8] * 4, [2] * 4, 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),   # rank 4
    ((1, [12], [2], 1, 1, 1, F32), capi.FNO_OK),                       # any extent
    ((1, [12], [8], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),          # m > N/2 + 1
    ((1, [1], [1], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),           # N < 2
    ((1, [16], [0], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),          # m = 0
    ((1, [16], [10], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),         # m > N/2 + 1
    ((2, [16, 16], [9, 4], 1, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),   # corners overlap
    ((2, [16, 16], [8, 9], 1, 1, 1, F32), capi.FNO_OK),
    ((1, [16], [4], 0, 1, 1, F32), capi.FNO_ERR_INVALID_ARG),          # batch 0
    ((1, [16], [4], 1, 0, 1, F32), capi.FNO_ERR_INVALID_ARG),          # cin 0
    ((1, [16], [4], 1, 1, -2, F32), capi.FNO_ERR_INVALID_ARG),         # cout < 0
    ((1, [16], [4], 1, 1, 1, 7), capi.FNO_ERR_INVALID_ARG),            # dtype
    ((1, [16], [4], 1, 1, 1, 3), capi.FNO_ERR_INVALID_ARG),            # dtype
    ((1, [4096], [4], 1, 1, 1, F32), capi.FNO_OK),
    ((1, [4097], [4], 1, 1, 1, F32), capi.FNO_ERR_UNSUPPORTED),        # N too large
])
def test_query_rejects(L, args, code):
    st, _, _ = Q(*args)
    assert st == code


def test_query_rejects_unknown_flags_and_nulls(L):
    st, _, _ = Q(1, [16], [4], 1, 1, 1, F32, flags=0x1000)
    assert st == capi.FNO_ERR_INVALID_ARG
    # bit 4 (a former tensor-core switch that did nothing) is not a flag
    st, _, _ = Q(2, [128, 128], [16, 16], 8, 32, 32, F32, flags=4)
    assert st == capi.FNO_ERR_INVALID_ARG
    # the tensor-core mixing request is a flag (ignored where it does not apply)
    for shape in (([128, 128], [16, 16]), ([64], [8])):
        st, _, _ = Q(len(shape[0]), shape[0], shape[1], 8, 32, 32, F32,
                     flags=capi.FNO_PLAN_TENSOR_EXTRA)
        assert st == capi.FNO_OK
    import ctypes
    assert L.fno_spectral_conv_query(1, None, None, 1, 1, 1, 0, 0, None, None) == \
        capi.FNO_ERR_INVALID_ARG
    assert L.fno_spectral_conv_plan(None, 1, None, None, 1, 1, 1, 0, 0) == \
        capi.FNO_ERR_INVALID_ARG
    h = ctypes.c_void_p(0)
    st = L.fno_spectral_conv_plan(ctypes.byref(h), 2, None, None, 1, 1, 1, 0, 0)
    assert st == capi.FNO_ERR_INVALID_ARG and not h.value


def test_null_handles(L):
    assert capi.fno_plan_destroy(None) == capi.FNO_OK
    assert capi.fno_model_destroy(None) == capi.FNO_OK
    assert capi.fno_spectral_conv_forward(None, 16, 16, 16, 16, None) == capi.FNO_ERR_INVALID_ARG
    assert capi.fno_plan_get_device_error(None, None) == capi.FNO_ERR_INVALID_ARG
    assert capi.fno_spectral_conv_workspace_size(None)[0] == capi.FNO_ERR_INVALID_ARG
    assert capi.fno_model_plan(capi.fno_model_desc_t())[0] == capi.FNO_ERR_INVALID_ARG


def test_invalid_plan_makes_no_cuda_call(L, monkeypatch):
    # validation happens before any CUDA call: an invalid description is
    # rejected the same way with or without a device
    st, h = capi.fno_spectral_conv_plan(2, [16, 16], [9, 4], 1, 1, 1, F32)
    assert st == capi.FNO_ERR_INVALID_ARG and not h


def test_fault_injection_plan_alloc(L, monkeypatch):
    monkeypatch.setenv("FNO_FAULT_INJECT", "plan_alloc")
    st, h = capi.fno_spectral_conv_plan(2, [16, 16], [4, 4], 1, 2, 2, F32)
    assert st == capi.FNO_ERR_OUT_OF_MEMORY and not h
    d = capi.fno_model_desc_t()
    d.batch, d.cin_lift, d.width, d.nlayers, d.hidden, d.cout = 1, 3, 4, 1, 4, 1
    d.h, d.w = 16, 16
    d.modes[0], d.modes[1] = 4, 4
    st, h = capi.fno_model_plan(d)
    assert st == capi.FNO_ERR_OUT_OF_MEMORY and not h


def test_model_desc_validation(L):
    d = capi.fno_model_desc_t()
    d.batch, d.cin_lift, d.width, d.nlayers, d.hidden, d.cout = 1, 3, 4, 1, 4, 1
    d.h, d.w = 16, 16
    d.modes[0], d.modes[1] = 9, 4          # corner blocks would overlap
    assert capi.fno_model_plan(d)[0] == capi.FNO_ERR_INVALID_ARG
    d.modes[0] = 4
    d.cout = 9                             # more outputs than the projection kernel holds
    assert capi.fno_model_plan(d)[0] == capi.FNO_ERR_UNSUPPORTED
    d.cout = 1
    d.dtype = 7                            # not a storage type
    assert capi.fno_model_plan(d)[0] == capi.FNO_ERR_INVALID_ARG
    d.dtype = F32
    d.h, d.w = 5, 6                        # h*w not a multiple of 4
    d.modes[0], d.modes[1] = 2, 3
    assert capi.fno_model_plan(d)[0] == capi.FNO_ERR_UNSUPPORTED


def test_backward_flag_adds_workspace(L):
    st, ws0, wb = Q(2, [128, 128], [16, 16], 8, 32, 16, F32)
    assert st == capi.FNO_OK
    st, ws1, wb1 = Q(2, [128, 128], [16, 16], 8, 32, 16, F32, flags=capi.FNO_PLAN_BACKWARD)
    assert st == capi.FNO_OK and wb1 == wb
    # the adjoint weights, the kept modes of x (8*32*512) and dy (8*16*512)
    assert ws1 >= wb + 8 * 32 * 512 * 8 + 8 * 16 * 512 * 8
    st, _, _ = Q(1, [16], [4], 1, 1, 1, F32, flags=capi.FNO_PLAN_BACKWARD | 0x1000)
    assert st == capi.FNO_ERR_INVALID_ARG


def test_packed_weights_flag_validation(L):
    P = capi.FNO_PLAN_PACKED_WEIGHTS
    assert Q(2, [128, 128], [16, 16], 8, 32, 32, F32, flags=P)[0] == capi.FNO_OK
    assert Q(1, [16], [5], 1, 2, 2, F32, flags=P)[0] == capi.FNO_ERR_INVALID_ARG   # |K| = 5
    assert Q(1, [16], [8], 1, 2, 2, F32, flags=P | capi.FNO_PLAN_BACKWARD)[0] == \
        capi.FNO_ERR_INVALID_ARG
    # same weight bytes in both layouts
    assert Q(2, [32, 32], [4, 4], 1, 3, 5, F32, flags=P)[2] == \
        Q(2, [32, 32], [4, 4], 1, 3, 5, F32)[2]
    assert capi.fno_spectral_conv_pack_weights(None, None, None, None) == capi.FNO_ERR_INVALID_ARG


def test_padded_query_validation(L):
    QP = capi.fno_spectral_conv_query_padded
    # modes are counted on the padded transform length: 2 m <= n + pad
    assert QP(1, [12], [4], [8], 1, 2, 2, F32)[0] == capi.FNO_OK          # m <= 16/2 + 1
    assert QP(1, [12], [4], [10], 1, 2, 2, F32)[0] == capi.FNO_ERR_INVALID_ARG
    assert QP(2, [6, 10], [2, 6], [4, 9], 1, 2, 2, F32)[0] == capi.FNO_OK
    assert QP(2, [6, 10], [1, 6], [4, 9], 1, 2, 2, F32)[0] == capi.FNO_ERR_INVALID_ARG
    assert QP(1, [12], [-1], [4], 1, 2, 2, F32)[0] == capi.FNO_ERR_INVALID_ARG
    assert QP(1, [4000], [200], [4], 1, 2, 2, F32)[0] == capi.FNO_ERR_UNSUPPORTED
    # an extent of one sample is fine once padded; the backward is not offered
    assert QP(1, [1], [7], [3], 1, 2, 2, F32)[0] == capi.FNO_OK
    assert QP(1, [12], [4], [4], 1, 2, 2, F32,
              flags=capi.FNO_PLAN_BACKWARD)[0] == capi.FNO_ERR_UNSUPPORTED
    # NULL or zero padding is the periodic layer, with the same sizes
    a = QP(2, [128, 128], None, [16, 16], 8, 32, 32, F32)
    b = QP(2, [128, 128], [0, 0], [16, 16], 8, 32, 32, F32)
    c = Q(2, [128, 128], [16, 16], 8, 32, 32, F32)
    assert a == b == c
    # a padded layer runs on the separate kernels: its workspace is theirs
    d = QP(2, [100, 120], [28, 8], [16, 16], 8, 32, 32, F32)
    e = Q(2, [128, 128], [16, 16], 8, 32, 32, F32, flags=capi.FNO_PLAN_UNFUSED)
    assert d[0] == capi.FNO_OK and d[1] <= e[1] and d[2] == e[2]


def test_index_checking_build_exports_the_same_symbols():
    # the FNO_DEBUG_BOUNDS variant is the same library with index checks:
    # built from the same sources, it exports every declared entry point
    import ctypes
    from fft_gemm_ifft_gb300 import build
    path = build.build(debug_bounds=True)
    assert path.endswith("libfno_bounds.so") and os.path.exists(path)
    B = ctypes.CDLL(path)
    for name in declared_functions():
        assert hasattr(B, name), f"libfno_bounds.so does not export {name}"
