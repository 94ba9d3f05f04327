"""UE5M3 two-linear stack with a stale global amax (through the C ABI).

"UE5M3 FP4 Block Scaling ..." blog, section "Что сделали": UE5M3 block scales,
the tensor maximum refreshed once every 50 steps with the stored value used in
between, stochastic rounding only on backward gradients, every linear in FP4.
The workload is the Nemotron-H-8B-like stack of two linears (H = X W1^T,
Y = H W2^T) over a sequence whose inputs drift by 1.02x per step, shrunk 32x
per dimension (M = 1024, hidden 256, FFN 512) so the oracle finishes quickly.

Per tested step every quantized operand (row and transposed, RNE forward, SR
for the gradients dY and dH) is compared bit-exactly, the UE5M3 -> E4M3
re-encode and its shift are compared exactly, and the six GEMMs (forward,
dgrad, wgrad of both layers) are checked against the oracle's float64 GEMM.
The layer-2 input H and the layer-1 gradient dH are the oracle's own bf16
GEMM outputs, fed identically to both sides.
"""

import numpy as np
import pytest
import torch

from fp4_block_scaled_amax_gb300 import synth
from oracle import gemm as Gm
from oracle import quantize as Q
from oracle.amax import AmaxState
from gpu_util import dev, f32, from_mma, host, lib, to_mma

pytestmark = pytest.mark.gpu

SCALE = 32
STEPS = (0, 1, 49, 50, 51, 99)


def bf16_of(a):
    return synth.to_bf16(np.asarray(a, dtype=np.float32))


def oracle_gemm(a, b):
    C, _ = Gm.gemm_ref(a["codes"], a["scales"], a["amax_used"], b["codes"], b["scales"], b["amax_used"], "UE5M3")
    return C


def oq(x_bf16, rounding, seed, g, transpose=False):
    q = Q.quantize(f32(x_bf16), "UE5M3", rounding, seed, global_amax=g, transpose=transpose)
    q["amax_used"] = np.float32(g)
    return q


def gpu_q(x_bf16, rounding, seed, g, transpose):
    fp4 = lib()
    x = dev(x_bf16)
    M, K = x.shape
    rows, cols = (K, M) if transpose else (M, K)
    codes = torch.empty((rows, cols // 2), dtype=torch.uint8, device="cuda")
    scales = torch.empty(rows * cols // 16, dtype=torch.uint8, device="cuda")
    gt = torch.tensor([g], dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp4.fp4_quantize(x, "UE5M3", fp4.FP4_ROUND_STOCHASTIC if rounding == "sr" else fp4.FP4_ROUND_RNE, seed, gt,
                     transpose, fp4.FP4_SFLAYOUT_MMA, codes, scales, None, st)
    assert int(host(st)[0]) == 0
    return codes, scales, gt


def gpu_gemm_ue5m3(a, b, M, N, K):
    """a, b: (codes, mma scales, g) on the device; returns (C float32 host, tA, tB)."""
    fp4 = lib()
    out = []
    for codes, scales, g in (a, b):
        t = torch.zeros(1, dtype=torch.int32, device="cuda")
        e4 = torch.empty_like(scales)
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp4.fp4_ue5m3_to_e4m3(scales, t, e4, st)
        assert int(host(st)[0]) == 0, "UE5M3 re-encode not exact"
        out.append((codes, e4, g, t))
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    (ac, ae, ag, at), (bc, be, bg, bt) = out
    fp4.fp4_gemm(ac, ae, bc, be, ag, bg, at, bt, M, N, K, "UE5M3", fp4.FP4_OUT_F32, C, dev_status=st)
    assert int(host(st)[0]) == 0
    return host(C), int(host(at)[0]), int(host(bt)[0])


def check_q(gq, ref, rows, cols, what):
    codes, scales, _ = gq
    assert np.array_equal(host(codes), ref["codes"]), what + " codes"
    assert np.array_equal(from_mma(host(scales), rows, cols // 16), ref["scales"]), what + " scales"


def check_gemm(Cg, a, b, what):
    C, S = Gm.gemm_ref(a["codes"], a["scales"], a["amax_used"], b["codes"], b["scales"], b["amax_used"], "UE5M3")
    err = np.abs(Cg - C)
    bound = Gm.gemm_bound(S)
    assert (err <= bound).all(), f"{what}: worst ratio {np.max(err / bound):.3g}"


def test_stack_over_steps():
    w = synth.config4_weights(SCALE)
    W1, W2 = w["W1"], w["W2"]  # [F, H], [H, F]
    F_, H_ = W1.shape
    state = {k: AmaxState(period=50) for k in ("X", "W1", "H", "W2", "dY", "dH")}
    for t in range(max(STEPS) + 1):
        refresh = t % 50 == 0
        if not refresh and t not in STEPS:
            continue  # nothing changes in between except the inputs, which are step-indexed
        d = synth.config4_step(t, SCALE)
        X, dY = d["X"], d["dY"]
        M = X.shape[0]
        g = {}
        for name, x in (("X", X), ("W1", W1), ("W2", W2), ("dY", dY)):
            g[name] = state[name].amax_for_step(t, f32(x))
        # oracle forward of layer 1 gives H; layer-2 dgrad gives dH (both bf16)
        qX = oq(X, "rne", 0, g["X"])
        qW1 = oq(W1, "rne", 0, g["W1"])
        H = bf16_of(oracle_gemm(qX, qW1))
        g["H"] = state["H"].amax_for_step(t, f32(H))
        qW2t = oq(W2, "rne", 0, g["W2"], transpose=True)
        seed = 1234 + 8 * t
        qdY = oq(dY, "sr", seed + 0, g["dY"])
        dH = bf16_of(oracle_gemm(qdY, qW2t))
        g["dH"] = state["dH"].amax_for_step(t, f32(dH))
        if t not in STEPS:
            continue
        # 40+ steps after a refresh the drift (1.02^t) has outgrown the stored amax
        if t % 50 >= 40:
            assert g["X"] < np.max(np.abs(f32(X)))
        qH = oq(H, "rne", 0, g["H"])
        qW2 = oq(W2, "rne", 0, g["W2"])
        qdYt = oq(dY, "sr", seed + 1, g["dY"], transpose=True)
        qHt = oq(H, "rne", 0, g["H"], transpose=True)
        qdH = oq(dH, "sr", seed + 2, g["dH"])
        qdHt = oq(dH, "sr", seed + 3, g["dH"], transpose=True)
        qW1t = oq(W1, "rne", 0, g["W1"], transpose=True)
        qXt = oq(X, "rne", 0, g["X"], transpose=True)

        G = {}
        specs = {
            "X": (X, "rne", 0, "X", False), "W1": (W1, "rne", 0, "W1", False), "H": (H, "rne", 0, "H", False),
            "W2": (W2, "rne", 0, "W2", False), "dY": (dY, "sr", seed + 0, "dY", False),
            "dH": (dH, "sr", seed + 2, "dH", False), "W2t": (W2, "rne", 0, "W2", True),
            "dYt": (dY, "sr", seed + 1, "dY", True), "Ht": (H, "rne", 0, "H", True),
            "dHt": (dH, "sr", seed + 3, "dH", True), "W1t": (W1, "rne", 0, "W1", True),
            "Xt": (X, "rne", 0, "X", True)}
        refs = {"X": qX, "W1": qW1, "H": qH, "W2": qW2, "dY": qdY, "dH": qdH, "W2t": qW2t, "dYt": qdYt,
                "Ht": qHt, "dHt": qdHt, "W1t": qW1t, "Xt": qXt}
        for key, (x, rnd, sd, gname, tr) in specs.items():
            G[key] = gpu_q(x, rnd, sd, float(g[gname]), tr)
            rows, cols = (x.shape[1], x.shape[0]) if tr else tuple(x.shape)
            check_q(G[key], refs[key], rows, cols, f"step {t} {key}")
            # UE5M3 re-encode shift equals the oracle's
            tref = Q.ue5m3_shift(refs[key]["scales"])
            _, exact = Q.ue5m3_reencode_e4m3(refs[key]["scales"], tref)
            assert exact, f"step {t} {key}: UE5M3 scales outside the E4M3 window"

        gemms = [("L1 fwd", "X", "W1", M, F_, H_), ("L2 fwd", "H", "W2", M, H_, F_),
                 ("L2 dgrad", "dY", "W2t", M, F_, H_), ("L2 wgrad", "dYt", "Ht", H_, F_, M),
                 ("L1 dgrad", "dH", "W1t", M, H_, F_), ("L1 wgrad", "dHt", "Xt", F_, H_, M)]
        for what, a, b, m, n, k in gemms:
            Cg, tA, tB = gpu_gemm_ue5m3(G[a], G[b], m, n, k)
            assert tA == Q.ue5m3_shift(refs[a]["scales"]) and tB == Q.ue5m3_shift(refs[b]["scales"])
            check_gemm(Cg, refs[a], refs[b], f"step {t} {what}")
