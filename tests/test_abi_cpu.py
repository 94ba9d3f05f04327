"""Host-side checks of the C ABI (no GPU needed).

The library loads and exports every function include/fp4.h declares; argument
errors are reported before anything touches a device (fake pointer values are
never dereferenced because every check fails first).
"""

import ctypes
import os
import shutil

import pytest

from fp4_block_scaled_amax_gb300 import fp4


def _need_lib():
    if not os.path.exists(fp4.LIB_PATH):
        if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
            pytest.skip("libfp4.so not built and no nvcc")
        from fp4_block_scaled_amax_gb300 import build
        build.build()
    return fp4._lib()


def test_exports_every_header_function():
    lib = _need_lib()
    names = fp4.header_functions()
    assert len(names) >= 13
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(fp4._SIGS), "binding and header disagree"


def test_group_size_and_storage_bytes():
    _need_lib()
    assert fp4.fp4_group_size("E4M3") == 16
    assert fp4.fp4_group_size("UE5M3") == 16
    assert fp4.fp4_group_size("E8M0") == 32
    assert fp4.fp4_group_size("E1M6") == 16
    for f in ("E2M5", "E3M4", "E5M2", "E6M1", "E7M0"):
        assert fp4.fp4_group_size(f) == 16
    assert fp4.fp4_group_size("NVINT4") == 16
    assert fp4.fp4_group_size("MXINT4") == 32
    assert fp4._lib().fp4_group_size(11) == 0
    cb, sb = fp4.fp4_storage_bytes(64, 1024, "E4M3")
    assert (cb + sb) * 8 / (64 * 1024) == 4.5
    cb, sb = fp4.fp4_storage_bytes(64, 1024, "E8M0")
    assert (cb + sb) * 8 / (64 * 1024) == 4.25
    with pytest.raises(fp4.Fp4Error) as e:
        fp4.fp4_storage_bytes(4, 40, "E8M0")
    assert e.value.status == fp4.FP4_ERR_SHAPE


def test_status_strings():
    _need_lib()
    for s in range(9):
        assert fp4.fp4_status_string(s)
    assert fp4.fp4_status_string(42) == "unknown status"


P = 0x10000  # a fake, 16-byte aligned "device" address; never dereferenced


def q(**kw):
    lib = _need_lib()
    a = dict(x=P, M=64, K=64, ldx=64, f=0, r=0, seed=0, g=P, tr=0, sfl=0, codes=P, scales=P, amax=None,
             shift=None, st=None)
    a.update(kw)
    return lib.fp4_quantize(a["x"], a["M"], a["K"], a["ldx"], a["f"], a["r"], a["seed"], a["g"], a["tr"],
                            a["sfl"], a["codes"], a["scales"], a["amax"], a["shift"], a["st"], None)


def test_quantize_argument_errors():
    assert q(f=11) == fp4.FP4_ERR_INVALID_ARG
    assert q(r=3) == fp4.FP4_ERR_INVALID_ARG
    assert q(tr=2) == fp4.FP4_ERR_INVALID_ARG
    assert q(K=40, ldx=40) == fp4.FP4_ERR_SHAPE           # K not a multiple of 16
    assert q(f=2, K=48, ldx=48) == fp4.FP4_ERR_SHAPE      # MXFP4 needs 32
    assert q(ldx=32) == fp4.FP4_ERR_SHAPE                 # ldx < K
    assert q(x=P + 8) == fp4.FP4_ERR_ALIGNMENT
    assert q(ldx=68) == fp4.FP4_ERR_ALIGNMENT             # row pitch 136 bytes
    assert q(codes=None) == fp4.FP4_ERR_INVALID_ARG
    assert q(scales=P + 4) == fp4.FP4_ERR_ALIGNMENT
    assert q(tr=1, M=48) == fp4.FP4_ERR_SHAPE             # transpose needs M % 32
    assert q(sfl=1) == fp4.FP4_ERR_SHAPE                  # MMA layout needs rows % 128
    assert q(g=None, amax=None) == fp4.FP4_ERR_INVALID_ARG  # fresh amax needs amax_out
    # the UE5M3 shift by-product exists for UE5M3 scales only (checked before any launch)
    for f in (0, 2, 3):
        assert q(f=f, shift=P) == fp4.FP4_ERR_UNSUPPORTED
        assert lib_dual(f=f, shift=P) == fp4.FP4_ERR_UNSUPPORTED


def lib_dual(**kw):
    lib = _need_lib()
    a = dict(f=0, M=64, K=64, shift=None)
    a.update(kw)
    return lib.fp4_quantize_dual(P, a["M"], a["K"], a["K"], a["f"], 0, 0, 0, 0, P, 0, P, P, P, P, None, a["shift"],
                                 None, None)


def test_gemm_argument_errors():
    lib = _need_lib()

    def g(**kw):
        a = dict(M=128, N=256, K=256, f=0, lay=0, od=0, ldc=256, A=P, C=P, ta=None)
        a.update(kw)
        return lib.fp4_gemm(a["A"], P, P, P, P, P, a["ta"], a["ta"], a["M"], a["N"], a["K"], a["f"], a["lay"],
                            a["od"], a["C"], a["ldc"], None, None)

    assert g(lay=1) == fp4.FP4_ERR_INVALID_ARG
    assert g(f=3) == fp4.FP4_ERR_UNSUPPORTED              # E1M6 has no GEMM
    assert g(f=1) == fp4.FP4_ERR_INVALID_ARG              # UE5M3 needs tA, tB
    assert g(M=100) == fp4.FP4_ERR_SHAPE
    assert g(N=192, ldc=192) == fp4.FP4_ERR_SHAPE          # N must be a multiple of 128
    assert g(K=128) == fp4.FP4_ERR_SHAPE
    assert g(ldc=100) == fp4.FP4_ERR_SHAPE
    assert g(A=P + 1) == fp4.FP4_ERR_ALIGNMENT
    assert g(od=1, ldc=260) == fp4.FP4_ERR_ALIGNMENT      # 520-byte bf16 rows
    assert g(C=None) == fp4.FP4_ERR_INVALID_ARG


def test_gemm_quantize_dual_argument_errors():
    lib = _need_lib()

    def g(**kw):
        a = dict(M=256, N=256, K=256, rr=0, rc=0, sfl=0, C=P, Cs=P, Ct=P, Cts=P, A=P)
        a.update(kw)
        return lib.fp4_gemm_quantize_dual(a["A"], P, P, P, P, P, None, None, a["M"], a["N"], a["K"], 0, 0, P,
                                          a["rr"], 0, a["rc"], 0, a["sfl"], a["C"], a["Cs"], a["Ct"], a["Cts"],
                                          None, None, None)

    assert g(C=None, Cs=None, Ct=None, Cts=None) == fp4.FP4_ERR_INVALID_ARG  # no output at all
    assert g(Cs=None) == fp4.FP4_ERR_INVALID_ARG                            # half a pair
    assert g(Cts=None) == fp4.FP4_ERR_INVALID_ARG
    assert g(rc=2) == fp4.FP4_ERR_INVALID_ARG
    assert g(sfl=2) == fp4.FP4_ERR_INVALID_ARG
    assert g(M=128) == fp4.FP4_ERR_UNSUPPORTED                              # CTA pairs only
    assert g(K=128) == fp4.FP4_ERR_SHAPE
    assert g(Ct=P + 8) == fp4.FP4_ERR_ALIGNMENT
    assert g(A=P + 1) == fp4.FP4_ERR_ALIGNMENT


def test_gemv_and_misc_argument_errors():
    lib = _need_lib()
    assert lib.fp4_gemv_w4a16(P, P, P, P, 0, 128, 256, 0, P, None, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_gemv_w4a16(P, P, P, P, 65, 128, 256, 0, P, None, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_gemv_w4a16(P, P, P, P, 1, 128, 48, 0, P, None, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_gemv_w4a16(P, P, None, P, 1, 128, 256, 0, P, None, None) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_amax(P, 4, 12, 12, P, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_amax(P, 4, 16, 16, None, None) == fp4.FP4_ERR_INVALID_ARG
    arr = lambda t, *v: (t * len(v))(*v)
    xs = arr(ctypes.c_void_p, P, P)
    i64 = ctypes.c_int64
    assert lib.fp4_amax_n(9, xs, arr(i64, 4, 4), arr(i64, 16, 16), arr(i64, 16, 16), P, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_amax_n(2, xs, arr(i64, 4, 4), arr(i64, 16, 12), arr(i64, 16, 16), P, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_amax_n(2, xs, arr(i64, 4, 4), arr(i64, 16, 16), arr(i64, 16, 16), None, None) == \
        fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_amax_n(2, arr(ctypes.c_void_p, P, P + 8), arr(i64, 4, 4), arr(i64, 16, 16), arr(i64, 16, 16), P,
                          None) == fp4.FP4_ERR_ALIGNMENT
    assert lib.fp4_amax_n(0, None, None, None, None, None, None) == fp4.FP4_OK
    assert lib.fp4_dequantize(P, P, 0, 4, 24, 0, P, 0, P, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_ue5m3_to_e4m3(P, 16, None, P, None, None) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_ue5m3_windows(P, 16, P, None, P, None, None) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_ue5m3_reencode(P, 16, None, P, None, None) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_ue5m3_reencode(P, -1, P, P, None, None) == fp4.FP4_ERR_SHAPE
    assert lib.fp4_ue5m3_windows(P, -1, P, P, P, None, None) == fp4.FP4_ERR_SHAPE
    w = lambda M=256, N=256, K=256, A=P, C=P, ldc=256, nA=P: lib.fp4_gemm_ue5m3_windows(
        A, P, P, nA, P, P, P, P, P, P, M, N, K, C, ldc, None, None)
    assert w(nA=None) == fp4.FP4_ERR_INVALID_ARG
    assert w(C=None) == fp4.FP4_ERR_INVALID_ARG
    assert w(M=100) == fp4.FP4_ERR_SHAPE
    assert w(N=192) == fp4.FP4_ERR_SHAPE
    assert w(ldc=100) == fp4.FP4_ERR_SHAPE
    assert w(A=P + 1) == fp4.FP4_ERR_ALIGNMENT
    assert w(ldc=258) == fp4.FP4_ERR_ALIGNMENT           # 1032-byte float32 rows
    assert lib.fp4_encode_scales(P, 4, 11, P, P, None) == fp4.FP4_ERR_INVALID_ARG
    assert lib.fp4_philox_bits16(1, 0, -1, P, None) == fp4.FP4_ERR_SHAPE
    # empty tensors are valid no-ops
    assert lib.fp4_dequantize(None, None, 0, 0, 32, 0, None, 0, None, None) == fp4.FP4_OK


def test_sweep_formats_rows_only():
    # E2M5 .. E7M0 and the INT4 grids quantize along rows only: the transposed and dual layouts and
    # the GEMM report FP4_ERR_UNSUPPORTED before anything is launched
    lib = _need_lib()
    for f in (fp4.FP4_SF_E2M5, fp4.FP4_SF_E3M4, fp4.FP4_SF_E5M2, fp4.FP4_SF_E6M1, fp4.FP4_SF_E7M0,
              fp4.FP4_SF_NVINT4):
        assert q(f=f, tr=1) == fp4.FP4_ERR_UNSUPPORTED
        assert lib_dual(f=f) == fp4.FP4_ERR_UNSUPPORTED
        assert lib.fp4_gemm(P, P, P, P, P, P, None, None, 128, 256, 256, f, 0, 0, P, 256, None,
                            None) == fp4.FP4_ERR_UNSUPPORTED
