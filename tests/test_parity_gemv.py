"""GPU weight-only NVFP4 GEMV vs the oracle (through the C ABI)."""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import dev, f32, host, lib

pytestmark = pytest.mark.gpu


def run(W_bf16, x_bf16, out="f32"):
    fp4 = lib()
    qw = Q.quantize(f32(W_bf16), "E4M3")
    N, K = W_bf16.shape
    b = x_bf16.shape[0]
    y = torch.empty((b, N), dtype=torch.float32 if out == "f32" else torch.bfloat16, device="cuda")
    gw = torch.tensor([qw["amax"]], dtype=torch.float32, device="cuda")
    fp4.fp4_gemv_w4a16(dev(qw["codes"]), dev(qw["scales"]), gw, dev(x_bf16), b, N, K,
                       fp4.FP4_OUT_F32 if out == "f32" else fp4.FP4_OUT_BF16, y)
    yr, S = Gm.gemv_ref(qw["codes"], qw["scales"], qw["amax"], f32(x_bf16))
    yg = host(y.float())
    bound = Gm.gemm_bound(S) + (np.abs(yr) * 2.0 ** -8 if out == "bf16" else 0)
    err = np.abs(yg - yr)
    assert (err <= bound).all(), f"worst ratio {np.max(err / bound):.3g}"


@pytest.mark.parametrize("batch", [1, 3, 8, 13, 64])
def test_gemv_scaled_shapes(batch):
    d = synth.config5(batch, scale=4)  # W_up 4608 x 768, W_down 768 x 4608
    run(d["W_up"], d["x_up"])
    run(d["W_down"], d["x_down"], "bf16")


def test_gemv_ragged_rows_and_k():
    W = synth.normal((1000, 1056), 30, 0, std=0.02)  # N not a multiple of 16, K % 128 = 32
    x = synth.normal((5, 1056), 30, 1)
    run(W, x)


def test_gemv_ragged_rows_tma_form():
    # batch <= 8 and K % 256 == 0 take the shared-memory (TMA) form; N = 1000
    # leaves the last CTA's tiles partly past the end of W
    W = synth.normal((1000, 1024), 31, 0, std=0.02)
    for b in (1, 5, 8):
        run(W, synth.normal((b, 1024), 31, b))


def test_gemv_wide_scale_range():
    # block amaxes spread over 2^-20 .. 1 of the tensor amax: E4M3 block scales
    # down to the subnormal codes, and every E2M1 code, including +-0.5
    rng = np.random.default_rng(32)
    N, K = 512, 2048
    mag = 2.0 ** rng.uniform(-20, 0, (N, K // 16))
    W = rng.standard_normal((N, K)) * np.repeat(mag, 16, axis=1)
    W = torch.from_numpy(W.astype(np.float32)).to(torch.bfloat16)
    qw = Q.quantize(f32(W), "E4M3")
    assert (qw["scales"] < 8).any() and (qw["scales"] > 0).any()  # subnormal scale codes occur
    nib = np.concatenate([qw["codes"] & 15, qw["codes"] >> 4])
    assert np.isin(np.arange(16), nib).all()
    for b in (2, 8, 13, 64):
        run(W, synth.normal((b, K), 32, b), "bf16")


def test_gemv_ragged_rows_tensor_core_form():
    # batches 9..64 with K % 256 == 0 take the tcgen05 form (128 weight rows per
    # CTA, batch padded to 64 with zeros); N = 1000 leaves the last tile partly
    # past the end of W; K = 4096 splits K over a cluster of CTAs
    for K in (1024, 4096):
        W = synth.normal((1000, K), 34, K, std=0.02)
        for b in (9, 40, 64):
            run(W, synth.normal((b, K), 34, K + b), "f32" if b != 40 else "bf16")


@pytest.mark.parametrize("batch", [1, 8, 40])
def test_gemv_dependent_chain_reads_the_previous_output(batch):
    # each launch takes the previous launch's output as its activations; the
    # launches overlap (programmatic dependent launch), so a launch that read
    # its activations before the previous one finished would fail here
    fp4 = lib()
    K = 2048
    W = synth.normal((K, K), 38, 0, std=0.04)
    qw = Q.quantize(f32(W), "E4M3")
    codes, scales = dev(qw["codes"]), dev(qw["scales"])
    gw = torch.tensor([qw["amax"]], dtype=torch.float32, device="cuda")
    xs = [synth.normal((batch, K), 38, batch).cuda()]
    for _ in range(6):
        y = torch.empty((batch, K), dtype=torch.bfloat16, device="cuda")
        fp4.fp4_gemv_w4a16(codes, scales, gw, xs[-1], batch, K, K, fp4.FP4_OUT_BF16, y)
        xs.append(y)
    torch.cuda.synchronize()
    for i in range(6):
        yr, S = Gm.gemv_ref(qw["codes"], qw["scales"], qw["amax"], f32(xs[i].cpu()))
        yg = host(xs[i + 1].float())
        bound = Gm.gemm_bound(S) + np.abs(yr) * 2.0 ** -8
        assert (np.abs(yg - yr) <= bound).all(), f"link {i}"


def test_gemv_tensor_core_form_falls_back_for_k_not_multiple_of_256():
    W = synth.normal((384, 1056), 35, 0, std=0.02)
    run(W, synth.normal((33, 1056), 35, 1))


@pytest.mark.parametrize("batch", [8, 64])
def test_gemv_status_word_stays_clear(batch):
    fp4 = lib()
    W = synth.normal((4608, 768), 33, 0, std=0.02)
    x = synth.normal((batch, 768), 33, 1)
    qw = Q.quantize(f32(W), "E4M3")
    y = torch.empty((batch, 4608), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gw = torch.tensor([qw["amax"]], dtype=torch.float32, device="cuda")
    for _ in range(3):
        fp4.fp4_gemv_w4a16(dev(qw["codes"]), dev(qw["scales"]), gw, dev(x), batch, 4608, 768, fp4.FP4_OUT_F32, y,
                           dev_status=st)
    assert int(host(st)[0]) == 0
    yr, S = Gm.gemv_ref(qw["codes"], qw["scales"], qw["amax"], f32(x))
    assert (np.abs(host(y) - yr) <= Gm.gemm_bound(S)).all()
