"""fp4_dequantize against the oracle for the four main scale formats (through the C ABI).

"NVFP4 vs MXFP" post (quant_prune_distill #486), section "Метод": a stored
element is an E2M1 value times its block scale, under the per-tensor global
scale; the oracle's dequantization is f32(f32(e2m1 * s_b) / s_enc).

For E4M3, UE5M3, E8M0 and E1M6, with float32 and bf16 output and both scale
layouts (plain row-major and the GEMM's tiled layout):
  * codes and scales the oracle made from a config-2-like tensor (per-column
    sigma log-uniform in [0.1, 10]) under a fresh and a stale global amax;
  * an exhaustive case: every E2M1 code against every finite non-negative
    scale code of the format.
Float32 output is compared bit for bit; bf16 output must equal the oracle's
float32 rounded to bf16 (nearest even).
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import quantize as Q
from gpu_util import dev, f32, lib, to_mma

pytestmark = pytest.mark.gpu

FORMATS = ["E4M3", "UE5M3", "E8M0", "E1M6"]
# largest finite non-negative code of each scale format (c-1 .. c-4 readings)
MAX_CODE = {"E4M3": 0x7E, "UE5M3": 0xFE, "E8M0": 0xFE, "E1M6": 0x7F}


def _gpu_dequant(codes, scales, fmt, g, bf16, mma):
    fp4 = lib()
    M, half = codes.shape
    K = 2 * half
    sc = to_mma(scales) if mma else scales.reshape(-1)
    out = torch.empty((M, K), dtype=torch.bfloat16 if bf16 else torch.float32, device="cuda")
    gt = torch.tensor([g], dtype=torch.float32, device="cuda")
    fp4.fp4_dequantize(dev(codes), dev(sc), fp4.FP4_SFLAYOUT_MMA if mma else fp4.FP4_SFLAYOUT_PLAIN, M, K, fmt, gt,
                       fp4.FP4_OUT_BF16 if bf16 else fp4.FP4_OUT_F32, out)
    torch.cuda.synchronize()
    return out.cpu()


def _check(got, ref_f32, bf16, what):
    if bf16:
        want = torch.from_numpy(np.ascontiguousarray(ref_f32)).to(torch.bfloat16)
        assert torch.equal(got.view(torch.int16), want.view(torch.int16)), what
    else:
        g = got.numpy().view(np.uint32)
        w = np.ascontiguousarray(ref_f32, dtype=np.float32).view(np.uint32)
        bad = np.argwhere(g != w)
        assert bad.size == 0, f"{what}: {len(bad)} differ, first at {bad[0].tolist()}"


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("mma", [False, True], ids=["plain", "mma"])
def test_dequantize_oracle_codes(fmt, bf16, mma):
    d = synth.config2(scale=16)  # X 512 x 256
    x = f32(d["X"])[:384]
    g_fresh = np.float32(np.max(np.abs(x)))
    for g in (g_fresh, np.float32(g_fresh / 64)):  # fresh, and a stale amax 64x below the data
        q = Q.quantize(x, fmt, "rne", 0, global_amax=g)
        ref = Q.dequantize(q["codes"], q["scales"], fmt, g)
        got = _gpu_dequant(q["codes"], q["scales"], fmt, float(g), bf16, mma)
        _check(got, ref, bf16, f"{fmt} g={g}")


@pytest.mark.parametrize("fmt", FORMATS)
@pytest.mark.parametrize("bf16", [False, True], ids=["f32", "bf16"])
@pytest.mark.parametrize("mma", [False, True], ids=["plain", "mma"])
def test_dequantize_every_code(fmt, bf16, mma):
    G = Q.group_size(fmt)
    ncodes = MAX_CODE[fmt] + 1
    rows = 128 * ((ncodes + 127) // 128)  # one scale code per row (tiled layout: rows % 128)
    nb = 4                                # blocks per row (tiled layout: nb % 4)
    K = nb * G
    scale_codes = np.zeros((rows, nb), dtype=np.uint8)
    scale_codes[:ncodes, :] = np.arange(ncodes, dtype=np.uint8)[:, None]
    # every E2M1 code (both signs) in every block: nibble i of a block is code i % 16
    nib = (np.arange(K) % 16).astype(np.uint8)
    codes = np.broadcast_to((nib[0::2] | (nib[1::2] << 4))[None, :], (rows, K // 2)).copy()
    for g in (np.float32(1.0), np.float32(37.25), np.float32(3.0e-3)):
        ref = Q.dequantize(codes, scale_codes, fmt, g)
        got = _gpu_dequant(codes, scale_codes, fmt, float(g), bf16, mma)
        _check(got, ref, bf16, f"{fmt} g={g}")


def test_dequantize_zero_amax_and_empty():
    # g == 0 means s_enc = 1 (reading R5); an empty tensor is a no-op
    fp4 = lib()
    codes = np.full((128, 8), 0x71, dtype=np.uint8)  # nibbles 1 (0.5) and 7 (6)
    scales = np.full((128, 1), 0x38, dtype=np.uint8)  # E4M3 code of 1.0
    ref = Q.dequantize(codes, scales, "E4M3", np.float32(0.0))
    assert ref[0, 0] == np.float32(0.5 / 1.0) and ref[0, 1] == np.float32(6.0)
    got = _gpu_dequant(codes, scales, "E4M3", 0.0, False, False)
    _check(got, ref, False, "g = 0")
    gt = torch.zeros(1, dtype=torch.float32, device="cuda")
    fp4.fp4_dequantize(None, None, fp4.FP4_SFLAYOUT_PLAIN, 0, 32, "E4M3", gt, fp4.FP4_OUT_F32, None)
    torch.cuda.synchronize()
