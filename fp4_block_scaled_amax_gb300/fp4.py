"""ctypes binding of libfp4.so: the C ABI of include/fp4.h under the same names.

Argument marshalling only: tensors become device pointers and sizes, the stream
is torch's current CUDA stream, and a non-zero fp4_status raises Fp4Error.
Every computation happens in the library's CUDA kernels; there is no CPU path.
The library loads on the first call and a missing library raises at once.
"""

from __future__ import annotations

import ctypes
import os
import re

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfp4.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fp4.h")

# enums of include/fp4.h
FP4_OK, FP4_ERR_INVALID_ARG, FP4_ERR_SHAPE, FP4_ERR_ALIGNMENT, FP4_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
FP4_ERR_NONFINITE, FP4_ERR_UE5M3_RANGE, FP4_ERR_TIMEOUT, FP4_ERR_CUDA = 5, 6, 7, 8
FP4_SF_E4M3, FP4_SF_UE5M3, FP4_SF_E8M0, FP4_SF_E1M6 = 0, 1, 2, 3
FP4_SF_E2M5, FP4_SF_E3M4, FP4_SF_E5M2, FP4_SF_E6M1, FP4_SF_E7M0 = 4, 5, 6, 7, 8
FP4_SF_NVINT4, FP4_SF_MXINT4 = 9, 10
FP4_ROUND_RNE, FP4_ROUND_STOCHASTIC = 0, 1
FP4_SFLAYOUT_PLAIN, FP4_SFLAYOUT_MMA = 0, 1
FP4_OUT_F32, FP4_OUT_BF16 = 0, 1
FP4_LAYOUT_TN = 0

FMT = {"E4M3": FP4_SF_E4M3, "UE5M3": FP4_SF_UE5M3, "E8M0": FP4_SF_E8M0, "E1M6": FP4_SF_E1M6,
       "E2M5": FP4_SF_E2M5, "E3M4": FP4_SF_E3M4, "E5M2": FP4_SF_E5M2, "E6M1": FP4_SF_E6M1, "E7M0": FP4_SF_E7M0,
       "NVINT4": FP4_SF_NVINT4, "MXINT4": FP4_SF_MXINT4}
GROUP = {f: (32 if f in (FP4_SF_E8M0, FP4_SF_MXINT4) else 16) for f in FMT.values()}


class Fp4Error(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: fp4_status {status}"
        try:
            msg += f" ({_lib().fp4_status_string(status).decode()})"
            if status == FP4_ERR_CUDA:
                msg += f", cudaError {_lib().fp4_last_cuda_error()}"
        except Exception:  # noqa: BLE001 - message only
            pass
        super().__init__(msg)


_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_I32 = ctypes.c_int
_SZP = ctypes.POINTER(ctypes.c_size_t)

_SIGS = {
    "fp4_group_size": (_I32, [_I32]),
    "fp4_storage_bytes": (_I32, [_I64, _I64, _I32, _SZP, _SZP]),
    "fp4_amax": (_I32, [_VP, _I64, _I64, _I64, _VP, _VP]),
    "fp4_amax_n": (_I32, [_I32, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp4_quantize": (_I32, [_VP, _I64, _I64, _I64, _I32, _I32, _U64, _VP, _I32, _I32, _VP, _VP, _VP, _VP, _VP,
                            _VP]),
    "fp4_quantize_rht": (_I32, [_VP, _I64, _I64, _I64, _I32, _I32, _U64, ctypes.c_uint32, _VP, _I32, _VP, _VP, _VP,
                                _VP, _VP]),
    "fp4_quantize_dual_rht": (_I32, [_VP, _I64, _I64, _I64, _I32, _I32, _U64, _I32, _U64, ctypes.c_uint32, _VP, _VP,
                                     _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp4_quantize_dual": (_I32, [_VP, _I64, _I64, _I64, _I32, _I32, _U64, _I32, _U64, _VP, _I32,
                                 _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp4_dequantize": (_I32, [_VP, _VP, _I32, _I64, _I64, _I32, _VP, _I32, _VP, _VP]),
    "fp4_ue5m3_to_e4m3": (_I32, [_VP, _I64, _VP, _VP, _VP, _VP]),
    "fp4_ue5m3_reencode": (_I32, [_VP, _I64, _VP, _VP, _VP, _VP]),
    "fp4_gemm": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I32, _I32, _I32, _VP, _I64,
                        _VP, _VP]),
    "fp4_gemm_quantize": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I32, _I32, _VP, _I32,
                                 _U64, _I32, _VP, _VP, _VP, _VP, _VP]),
    "fp4_gemm_quantize_dual": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _I32, _I32, _VP,
                                      _I32, _U64, _I32, _U64, _I32, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp4_ue5m3_windows": (_I32, [_VP, _I64, _VP, _VP, _VP, _VP, _VP]),
    "fp4_gemm_ue5m3_windows": (_I32, [_VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _I64, _I64, _I64, _VP, _I64,
                                      _VP, _VP]),
    "fp4_gemv_w4a16": (_I32, [_VP, _VP, _VP, _VP, _I64, _I64, _I64, _I32, _VP, _VP, _VP]),
    "fp4_encode_scales": (_I32, [_VP, _I64, _I32, _VP, _VP, _VP]),
    "fp4_philox_bits16": (_I32, [_U64, _U64, _I64, _VP, _VP]),
    "fp4_status_string": (ctypes.c_char_p, [_I32]),
    "fp4_last_cuda_error": (_I32, []),
}

_handle = None


def header_functions() -> list:
    """Names of the functions include/fp4.h declares."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4_[a-z0-9_]+)\s*\(", text)))


def _lib():
    global _handle
    if _handle is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m fp4_block_scaled_amax_gb300.build`")
        h = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(h, name)
            fn.restype = res
            fn.argtypes = args
        _handle = h
    return _handle


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor arguments must be CUDA tensors")
    return t.data_ptr()


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(status: int, where: str):
    if status != FP4_OK:
        raise Fp4Error(status, where)


def _fmt(f) -> int:
    return FMT[f] if isinstance(f, str) else int(f)


# ---------------------------------------------------------------------------
# C ABI, same names
# ---------------------------------------------------------------------------

def fp4_group_size(fmt) -> int:
    return _lib().fp4_group_size(_fmt(fmt))


def fp4_storage_bytes(rows: int, cols: int, fmt) -> tuple:
    cb, sb = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib().fp4_storage_bytes(rows, cols, _fmt(fmt), ctypes.byref(cb), ctypes.byref(sb)),
           "fp4_storage_bytes")
    return cb.value, sb.value


def fp4_amax(x, amax_out, stream=None):
    M, K = x.shape
    _check(_lib().fp4_amax(_ptr(x), M, K, x.stride(0), _ptr(amax_out), _stream(stream)), "fp4_amax")


def fp4_amax_n(xs, amax_out, stream=None):
    """xs: a sequence of bf16 [M, K] CUDA tensors; amax_out: CUDA float32 tensor of len(xs)."""
    n = len(xs)
    ptrs = (ctypes.c_void_p * max(n, 1))(*[_ptr(x) for x in xs])
    Ms = (ctypes.c_int64 * max(n, 1))(*[x.shape[0] for x in xs])
    Ks = (ctypes.c_int64 * max(n, 1))(*[x.shape[1] for x in xs])
    lds = (ctypes.c_int64 * max(n, 1))(*[x.stride(0) for x in xs])
    _check(_lib().fp4_amax_n(n, ptrs, Ms, Ks, lds, _ptr(amax_out), _stream(stream)), "fp4_amax_n")


def fp4_quantize(x, fmt, rounding, seed, global_amax, transpose, sfl, codes, scales,
                 amax_out=None, dev_status=None, stream=None, ue5m3_shift_out=None):
    M, K = x.shape
    _check(_lib().fp4_quantize(_ptr(x), M, K, x.stride(0), _fmt(fmt), int(rounding), int(seed),
                               _ptr(global_amax), int(transpose), int(sfl), _ptr(codes), _ptr(scales),
                               _ptr(amax_out), _ptr(ue5m3_shift_out), _ptr(dev_status), _stream(stream)),
           "fp4_quantize")


def fp4_quantize_rht(x, fmt, rounding, seed, rht_mask, global_amax, sf_layout, codes, scales, amax_out=None,
                     dev_status=None, stream=None):
    M, K = x.shape
    _check(_lib().fp4_quantize_rht(_ptr(x), M, K, x.stride(0), _fmt(fmt), int(rounding), int(seed), int(rht_mask),
                                   _ptr(global_amax), int(sf_layout), _ptr(codes), _ptr(scales), _ptr(amax_out),
                                   _ptr(dev_status), _stream(stream)), "fp4_quantize_rht")


def fp4_quantize_dual_rht(x, fmt, r_row, seed_row, r_col, seed_col, rht_mask, g_row, g_col, sf_layout, codes_row,
                          scales_row, codes_col, scales_col, amax_row_out=None, amax_col_out=None, dev_status=None,
                          stream=None):
    M, K = x.shape
    _check(_lib().fp4_quantize_dual_rht(_ptr(x), M, K, x.stride(0), _fmt(fmt), int(r_row), int(seed_row), int(r_col),
                                        int(seed_col), int(rht_mask), _ptr(g_row), _ptr(g_col), int(sf_layout),
                                        _ptr(codes_row), _ptr(scales_row), _ptr(codes_col), _ptr(scales_col),
                                        _ptr(amax_row_out), _ptr(amax_col_out), _ptr(dev_status), _stream(stream)),
           "fp4_quantize_dual_rht")


def fp4_quantize_dual(x, fmt, r_row, seed_row, r_col, seed_col, global_amax, sfl, codes_row, scales_row,
                      codes_col, scales_col, amax_out=None, dev_status=None, stream=None, ue5m3_shift_out=None):
    M, K = x.shape
    _check(_lib().fp4_quantize_dual(_ptr(x), M, K, x.stride(0), _fmt(fmt), int(r_row), int(seed_row),
                                    int(r_col), int(seed_col), _ptr(global_amax), int(sfl),
                                    _ptr(codes_row), _ptr(scales_row), _ptr(codes_col), _ptr(scales_col),
                                    _ptr(amax_out), _ptr(ue5m3_shift_out), _ptr(dev_status), _stream(stream)),
           "fp4_quantize_dual")


def fp4_dequantize(codes, scales, sfl, M, K, fmt, global_amax, out_dtype, out, stream=None):
    _check(_lib().fp4_dequantize(_ptr(codes), _ptr(scales), int(sfl), M, K, _fmt(fmt), _ptr(global_amax),
                                 int(out_dtype), _ptr(out), _stream(stream)), "fp4_dequantize")


def fp4_ue5m3_to_e4m3(scales, t_out, e4m3_out, dev_status=None, stream=None):
    _check(_lib().fp4_ue5m3_to_e4m3(_ptr(scales), scales.numel(), _ptr(t_out), _ptr(e4m3_out),
                                    _ptr(dev_status), _stream(stream)), "fp4_ue5m3_to_e4m3")


def fp4_ue5m3_reencode(scales, t, e4m3_out, dev_status=None, stream=None):
    _check(_lib().fp4_ue5m3_reencode(_ptr(scales), scales.numel(), _ptr(t), _ptr(e4m3_out), _ptr(dev_status),
                                     _stream(stream)), "fp4_ue5m3_reencode")


def fp4_gemm(Aq, As, Bq, Bs, ga, gb, tA, tB, M, N, K, fmt, out_dtype, C, ldc=None, dev_status=None,
             stream=None):
    _check(_lib().fp4_gemm(_ptr(Aq), _ptr(As), _ptr(Bq), _ptr(Bs), _ptr(ga), _ptr(gb), _ptr(tA), _ptr(tB),
                           M, N, K, _fmt(fmt), FP4_LAYOUT_TN, int(out_dtype), _ptr(C),
                           N if ldc is None else ldc, _ptr(dev_status), _stream(stream)), "fp4_gemm")


def fp4_gemm_quantize(Aq, As, Bq, Bs, ga, gb, tA, tB, M, N, K, fmt, g_out, rounding, seed, sf_layout, C_codes,
                      C_scales, C_amax_out=None, dev_status=None, stream=None):
    _check(_lib().fp4_gemm_quantize(_ptr(Aq), _ptr(As), _ptr(Bq), _ptr(Bs), _ptr(ga), _ptr(gb), _ptr(tA), _ptr(tB),
                                    M, N, K, _fmt(fmt), FP4_LAYOUT_TN, _ptr(g_out), int(rounding), int(seed),
                                    int(sf_layout), _ptr(C_codes), _ptr(C_scales), _ptr(C_amax_out),
                                    _ptr(dev_status), _stream(stream)), "fp4_gemm_quantize")


def fp4_gemm_quantize_dual(Aq, As, Bq, Bs, ga, gb, tA, tB, M, N, K, fmt, g_out, r_row, seed_row, r_col, seed_col,
                           sf_layout, C_codes, C_scales, Ct_codes, Ct_scales, C_amax_out=None, dev_status=None,
                           stream=None):
    _check(_lib().fp4_gemm_quantize_dual(_ptr(Aq), _ptr(As), _ptr(Bq), _ptr(Bs), _ptr(ga), _ptr(gb), _ptr(tA),
                                         _ptr(tB), M, N, K, _fmt(fmt), FP4_LAYOUT_TN, _ptr(g_out), int(r_row),
                                         int(seed_row), int(r_col), int(seed_col), int(sf_layout), _ptr(C_codes),
                                         _ptr(C_scales), _ptr(Ct_codes), _ptr(Ct_scales), _ptr(C_amax_out),
                                         _ptr(dev_status), _stream(stream)), "fp4_gemm_quantize_dual")


def fp4_ue5m3_windows(scales, t_out, n_windows_out, out, dev_status=None, stream=None):
    _check(_lib().fp4_ue5m3_windows(_ptr(scales), scales.numel(), _ptr(t_out), _ptr(n_windows_out), _ptr(out),
                                    _ptr(dev_status), _stream(stream)), "fp4_ue5m3_windows")


def fp4_gemm_ue5m3_windows(Aq, As_windows, tA, nA, Bq, Bs_windows, tB, nB, ga, gb, M, N, K, C, ldc=None,
                           dev_status=None, stream=None):
    _check(_lib().fp4_gemm_ue5m3_windows(_ptr(Aq), _ptr(As_windows), _ptr(tA), _ptr(nA), _ptr(Bq), _ptr(Bs_windows),
                                         _ptr(tB), _ptr(nB), _ptr(ga), _ptr(gb), M, N, K, _ptr(C),
                                         N if ldc is None else ldc, _ptr(dev_status), _stream(stream)),
           "fp4_gemm_ue5m3_windows")


def fp4_gemv_w4a16(Wq, Ws, gw, x, batch, N, K, out_dtype, y, dev_status=None, stream=None):
    _check(_lib().fp4_gemv_w4a16(_ptr(Wq), _ptr(Ws), _ptr(gw), _ptr(x), batch, N, K, int(out_dtype), _ptr(y),
                                 _ptr(dev_status), _stream(stream)), "fp4_gemv_w4a16")


def fp4_encode_scales(s, fmt, codes, decoded, stream=None):
    _check(_lib().fp4_encode_scales(_ptr(s), s.numel(), _fmt(fmt), _ptr(codes), _ptr(decoded),
                                    _stream(stream)), "fp4_encode_scales")


def fp4_philox_bits16(seed, start, n, out, stream=None):
    _check(_lib().fp4_philox_bits16(int(seed), int(start), n, _ptr(out), _stream(stream)), "fp4_philox_bits16")


def fp4_status_string(status: int) -> str:
    return _lib().fp4_status_string(int(status)).decode()


def fp4_last_cuda_error() -> int:
    return _lib().fp4_last_cuda_error()


# ---------------------------------------------------------------------------
# Output allocation helpers (torch device memory; the calls above do the work)
# ---------------------------------------------------------------------------

def empty_quantized(rows: int, cols: int, fmt, device="cuda"):
    """(codes [rows, cols/2] uint8, scales [rows*cols/G] uint8) for an output layout [rows, cols]."""
    G = GROUP[_fmt(fmt)]
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device=device)
    scales = torch.empty((rows, cols // G), dtype=torch.uint8, device=device)
    return codes, scales


def quantize(x, fmt="E4M3", rounding=FP4_ROUND_RNE, seed=0, global_amax=None, transpose=False,
             sfl=FP4_SFLAYOUT_PLAIN, amax_out=None, dev_status=None, stream=None):
    M, K = x.shape
    rows, cols = (K, M) if transpose else (M, K)
    codes, scales = empty_quantized(rows, cols, fmt, x.device)
    if global_amax is None and amax_out is None:
        amax_out = torch.empty(1, dtype=torch.float32, device=x.device)
    fp4_quantize(x, fmt, rounding, seed, global_amax, transpose, sfl, codes, scales, amax_out, dev_status, stream)
    return codes, scales, amax_out
