#!/usr/bin/env python3
"""Benchmark of the FP4 block-scaled linear layer at Llama-2-7B MLP shapes.

One step is one pass of the whole hot path over the seeded synthetic workload
"Llama-2 7B MLP linear, forward and backward" (tokens M = 16384, K = 4096,
N = 11008; X N(0,1) with 0.5 % outliers x100, W N(0,0.02), dY Laplace(0,1e-4)):

  fresh global amax of dY                            (amax kernel)
  dual quantization of dY (E4M3 scales, 16-element blocks, as below):
      rows stochastic (seed 1234), dY^T stochastic (seed 1235)
                                                     (TMA dual quantizer)
  fresh global amax of X and W                       (amax kernel)
      on a second stream, beside dY's quantizer
  dual quantization of X: rows RNE, X^T stochastic (seed 1236)
                    of W: rows RNE, W^T RNE
  forward  Y  = X W^T    16384 x 11008 x 4096  bf16 out (tcgen05 FP4 GEMM)
  dgrad    dX = dY W     16384 x  4096 x 11008 bf16 out
  wgrad    dW = dY^T X   11008 x  4096 x 16384 bf16 out
      dgrad and wgrad on their own streams, each launched after the previous
      GEMM and taking the SMs that its last, partial round of tiles leaves idle
  weight-only decode GEMV with the same layer's weight (quantized once,
      batch 8): y = x W^T                                (GEMV kernel)
      on another stream after dgrad, beside wgrad's last round of tiles

metric: FP4 GEMM TFLOP/s of the whole step (3 * 2*M*N*K / step time), the
step captured once as a CUDA graph and replayed once per timed step;
per-kernel rooflines from CUDA events between the kernels of as many more
steps launched kernel by kernel on one stream.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

--impl reference times the CPU oracle (plain numpy, test infrastructure) on
a bounded slice of the same step.  With N > 1 (torchrun) every rank runs its
own independent batch (weak scaling, no collective on the data path).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

M_TOK, K_HID, N_FFN = 16384, 4096, 11008
GEMV_BATCH = 8
CPU_SAMPLE_TOKENS, CPU_SAMPLE_FEATURES = 4096, 4096  # oracle slice timed for cpu_baseline (~10-20 s of CPU work)
STEP_FLOPS = 3 * 2 * M_TOK * N_FFN * K_HID
WORKLOAD = "llama2-7b-mlp-linear-fwd-bwd"
METRIC = "NVFP4 GEMM TFLOPS & quantize GB/s at 7B shapes, % of FP4-MMA/HBM peak"
FP4_PER_BF16 = 6.0  # nominal dense FP4 / bf16 tensor ratio on GB300 (13.5 / 2.25 PFLOP/s)
# DRAM bytes (read + write) per launch of the full-size step, from ncu
# captures of one kernel at a time (`ncu --metrics dram__bytes_read.sum,
# dram__bytes_write.sum,gpu__time_duration.sum -k <kernel> -c 3`, one pass),
# valid only while the kernel sources still hash to the recorded value.
# gemm: mean over the fwd, dgrad and wgrad launches; quant_dual: the step's
# three dual quantizations together; amax: the step's two launches together;
# gemv: one launch.  Writes still
# held in L2 when a kernel ends do not appear in its DRAM bytes.
NCU_TRAFFIC = {"gemm": {"bytes": 292.44e6, "src": "ff8a151e85c2daa4",
                        "files": ["gemm_sm103.cu", "async_sm103.cuh", "fp4_device.cuh", "device_cache.h"]},
               "quant_dual": {"bytes": 803.50e6, "src": "c7678099edfacfa1",
                              "files": ["quantize.cu", "async_sm103.cuh", "fp4_device.cuh", "device_cache.h"]},
               "gemv": {"bytes": 25.46e6, "src": "fe1ed2b164c87513",
                        "files": ["gemv.cu", "async_sm103.cuh", "fp4_device.cuh", "device_cache.h"]},
               "amax": {"bytes": 586.87e6, "src": "c7678099edfacfa1",
                        "files": ["quantize.cu", "async_sm103.cuh", "fp4_device.cuh", "device_cache.h"]}}


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=10)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--studies", default="all",
                   help="comma-separated side studies to run (default: all), e.g. formats,stack")
    p.add_argument("--no-studies", action="store_true",
                   help="skip the side measurements after the timed steps (for ncu launch lists)")
    p.add_argument("--tokens", type=int, default=16384,
                   help="token count M (default: the workload's 16384; smaller only for ncu captures)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU)
# ---------------------------------------------------------------------------

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    if world > 1 and not torch.distributed.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        torch.distributed.init_process_group(backend)


def barrier(world):
    if world > 1:
        torch.distributed.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest rank sets the time)."""
    if world == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# peaks, clocks, cpu baseline
# ---------------------------------------------------------------------------

def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons every 200 ms during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        # address the GPU by UUID: CUDA_VISIBLE_DEVICES may renumber devices
        try:
            u = str(torch.cuda.get_device_properties(device).uuid)
            self.gpu = u if u.startswith("GPU-") else "GPU-" + u
        except Exception:  # noqa: BLE001
            self.gpu = str(device.index or 0)
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in getattr(self, "lines", []):
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": smax, "reasons": sorted(reasons),
                "samples": len(sm)}


def oracle_slice_step(d, Ms=1024, Ns=1024):
    """The oracle's version of one step restricted to Ms tokens x Ns output
    features at full K (quantizations of the needed operands, then the three
    float64 GEMMs).  Returns (flops, seconds)."""
    from oracle import gemm as Gm
    from oracle import quantize as Q
    X = d["X"][:Ms].float().numpy()
    W = d["W"][:Ns].float().numpy()
    dY = d["dY"][:Ms, :Ns].float().numpy()
    t0 = time.perf_counter()
    qX = Q.quantize(X, "E4M3", "rne", 0)
    qXt = Q.quantize(X, "E4M3", "sr", 1236, transpose=True)
    qW = Q.quantize(W, "E4M3", "rne", 0)
    qWt = Q.quantize(W, "E4M3", "rne", 0, transpose=True)
    qd = Q.quantize(dY, "E4M3", "sr", 1234)
    qdt = Q.quantize(dY, "E4M3", "sr", 1235, transpose=True)
    for a, b in [(qX, qW), (qd, qWt), (qdt, qXt)]:
        Gm.gemm_ref(a["codes"], a["scales"], a["amax"], b["codes"], b["scales"], b["amax"], "E4M3")
    dt = time.perf_counter() - t0
    return 3 * 2 * Ms * Ns * K_HID, dt


def cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# ---------------------------------------------------------------------------
# the GPU step
# ---------------------------------------------------------------------------

STEP_EVENTS = 10  # start, after amax(dY), quantize dY, amax(X, W) joined, quantize X, W, fwd, dgrad, wgrad joined,
                  # GEMV joined


class LinearStep:
    """Device buffers of one step and the sequence of library calls."""

    def __init__(self, d, device):
        from fp4_block_scaled_amax_gb300 import fp4
        self.fp4 = fp4
        self.dev = device
        M, K, N = M_TOK, K_HID, N_FFN
        u8 = dict(dtype=torch.uint8, device=device)
        self.X = d["X"].to(device)
        self.W = d["W"].to(device)
        self.dY = d["dY"].to(device)
        self.amax = torch.zeros(3, dtype=torch.float32, device=device)
        self.q = {}
        for name, (R, C) in {"X": (M, K), "W": (N, K), "dY": (M, N)}.items():
            self.q[name] = (torch.empty((R, C // 2), **u8), torch.empty(R * C // 16, **u8),
                            torch.empty((C, R // 2), **u8), torch.empty(R * C // 16, **u8))
        self.Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.dW = torch.empty((N, K), dtype=torch.bfloat16, device=device)
        # weight-only decode operand: W quantized once (plain scale layout)
        self.Wg_codes = torch.empty((N, K // 2), **u8)
        self.Wg_scales = torch.empty(N * K // 16, **u8)
        self.Wg_amax = torch.zeros(1, dtype=torch.float32, device=device)
        fp4.fp4_quantize(self.W, "E4M3", fp4.FP4_ROUND_RNE, 0, None, False, fp4.FP4_SFLAYOUT_PLAIN,
                         self.Wg_codes, self.Wg_scales, self.Wg_amax)
        self.xg = d["x_dec"].to(device)
        self.yg = torch.empty((GEMV_BATCH, N), dtype=torch.bfloat16, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.launches_per_step = 9  # 2 amax launches (dY; X and W), 3 dual quantizers, 3 GEMMs, 1 GEMV
        # streams of the overlapped step (see run); the decode GEMV depends on
        # none of the GEMMs and fills the SMs that wgrad's last round leaves idle
        self.s_amax = torch.cuda.Stream(device=device)
        self.s_dgrad = torch.cuda.Stream(device=device)
        self.s_wgrad = torch.cuda.Stream(device=device)
        self.s_gemv = torch.cuda.Stream(device=device)
        self.ev_amax_dy = torch.cuda.Event()
        self.ev_amax_xw = torch.cuda.Event()
        self.ev_quant = torch.cuda.Event()
        self.ev_dgrad = torch.cuda.Event()
        self.ev_wgrad = torch.cuda.Event()
        self.ev_gemv = torch.cuda.Event()

    def run(self, ev=None, serial=False):
        """One step; ev: optional list of STEP_EVENTS CUDA events recorded
        between kernels.  serial: every kernel on the current stream, one after
        another (the form in which each kernel's own time is measured);
        otherwise wgrad and the GEMV overlap as described above."""
        fp4 = self.fp4
        RNE, SR, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA
        M, K, N = M_TOK, K_HID, N_FFN
        st = torch.cuda.current_stream()

        def mark(i):
            if ev is not None:
                ev[i].record(st)

        def quant(j, name, rr, sr, rc, sc):
            cr, srs, cc, scs = self.q[name]
            fp4.fp4_quantize_dual(getattr(self, name), "E4M3", rr, sr, rc, sc, self.amax[j:j + 1], MMA, cr, srs,
                                  cc, scs, None, self.status)

        mark(0)
        # dY's fresh amax first, so that its dual quantizer, the longest, can start
        fp4.fp4_amax_n([self.dY], self.amax[2:3])
        mark(1)
        self.ev_amax_dy.record(st)
        quant(2, "dY", SR, 1234, SR, 1235)
        mark(2)
        # the fresh amaxes of X and W (one memory-bound launch) on their own
        # stream, launched after dY's quantizer: its CTAs run in the registers
        # and threads that the quantizer's leave free on each SM
        s_amax = st if serial else self.s_amax
        s_amax.wait_event(self.ev_amax_dy)
        with torch.cuda.stream(s_amax):
            fp4.fp4_amax_n([self.X, self.W], self.amax[0:2])
        self.ev_amax_xw.record(s_amax)
        st.wait_event(self.ev_amax_xw)
        mark(3)
        quant(0, "X", RNE, 0, SR, 1236)
        mark(4)
        quant(1, "W", RNE, 0, RNE, 0)
        mark(5)
        qX, qW, qd = self.q["X"], self.q["W"], self.q["dY"]
        aX, aW, ad = self.amax[0:1], self.amax[1:2], self.amax[2:3]
        BF = fp4.FP4_OUT_BF16
        # The three GEMMs read only the quantized operands: dgrad and wgrad wait
        # for nothing else, each on its own stream. Launched in the order fwd,
        # dgrad, wgrad, each takes the SMs that the previous one's last, partial
        # round of tiles leaves idle.
        s_dgrad, s_wgrad, s_gemv = (st, st, st) if serial else (self.s_dgrad, self.s_wgrad, self.s_gemv)
        self.ev_quant.record(st)
        fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", BF, self.Y,
                     dev_status=self.status)
        mark(6)
        s_dgrad.wait_event(self.ev_quant)
        with torch.cuda.stream(s_dgrad):
            fp4.fp4_gemm(qd[0], qd[1], qW[2], qW[3], ad, aW, None, None, M, K, N, "E4M3", BF, self.dX,
                         dev_status=self.status)
        self.ev_dgrad.record(s_dgrad)
        mark(7)
        s_wgrad.wait_event(self.ev_quant)
        with torch.cuda.stream(s_wgrad):
            fp4.fp4_gemm(qd[2], qd[3], qX[2], qX[3], ad, aX, None, None, N, K, M, "E4M3", BF, self.dW,
                         dev_status=self.status)
        self.ev_wgrad.record(s_wgrad)
        st.wait_event(self.ev_dgrad)
        st.wait_event(self.ev_wgrad)
        mark(8)
        # launched after wgrad, so wgrad's tiles take the SMs first
        s_gemv.wait_event(self.ev_dgrad)
        with torch.cuda.stream(s_gemv):
            fp4.fp4_gemv_w4a16(self.Wg_codes, self.Wg_scales, self.Wg_amax, self.xg, GEMV_BATCH, N, K, BF, self.yg)
        self.ev_gemv.record(s_gemv)
        st.wait_event(self.ev_gemv)
        mark(9)


# ---------------------------------------------------------------------------
# Nemotron-H-8B-like linear stack with UE5M3 scales (the UE5M3 recipe)
# ---------------------------------------------------------------------------
C4_M, C4_H, C4_F = 32768, 4096, 21504
C4_STEPS, C4_PERIOD = 100, 50
C4_NAMES = ("X", "W1", "H", "W2", "dY", "dH")


class StackStep:
    """One training step of the two-linear stack H = X W1^T, Y = H W2^T with
    UE5M3 block scales ("UE5M3 FP4 Block Scaling ..." blog, "Что сделали"):
    every tensor keeps a stored global amax refreshed every 50 steps (fresh
    amax passes on refresh steps only), forward operands nearest-rounded,
    the gradients dY and dH stochastically rounded (Philox seeds
    1234 + 8 t + role, roles 0/1 dY rows/columns, 2/3 dH rows/columns), each
    tensor quantized once in both layouts; the UE5M3 scales reach the E4M3
    tensor-core path by the per-tensor shift the quantizer reports and one
    re-encode pass; six FP4 GEMMs with bf16 outputs:
      L1 fwd   H   = X W1^T     M x F x H      L2 fwd   Y   = H W2^T     M x H x F
      L2 dgrad dH  = dY W2      M x F x H      L2 wgrad dW2 = dY^T H     H x F x M
      L1 dgrad dX  = dH W1      M x H x F      L1 wgrad dW1 = dH^T X     F x H x M
    """

    def __init__(self, device, M=C4_M, Hd=C4_H, F=C4_F, weights=None):
        from fp4_block_scaled_amax_gb300 import fp4, synth
        self.fp4 = fp4
        self.dev = device
        self.M, self.Hd, self.F = M, Hd, F
        u8 = dict(dtype=torch.uint8, device=device)
        bf = dict(dtype=torch.bfloat16, device=device)
        if weights is None:
            scale = C4_M // M
            weights = synth.config4_weights(scale)
        self.W1 = weights["W1"].to(device)
        self.W2 = weights["W2"].to(device)
        self.H = torch.empty((M, F), **bf)
        self.dH = torch.empty((M, F), **bf)
        self.Y = torch.empty((M, Hd), **bf)
        self.dX = torch.empty((M, Hd), **bf)
        self.dW2 = torch.empty((Hd, F), **bf)
        self.dW1 = torch.empty((F, Hd), **bf)
        shapes = {"X": (M, Hd), "W1": (F, Hd), "H": (M, F), "W2": (Hd, F), "dY": (M, Hd), "dH": (M, F)}
        # per tensor: row codes, row scales (UE5M3, tiled), transposed codes and
        # scales, their E4M3 re-encodes, and the two shifts
        self.q = {}
        for n, (R, C) in shapes.items():
            self.q[n] = {"cr": torch.empty((R, C // 2), **u8), "sr": torch.empty(R * C // 16, **u8),
                         "cc": torch.empty((C, R // 2), **u8), "sc": torch.empty(R * C // 16, **u8),
                         "er": torch.empty(R * C // 16, **u8), "ec": torch.empty(R * C // 16, **u8),
                         "t": torch.zeros(2, dtype=torch.int32, device=device)}
        self.stored = torch.zeros(len(C4_NAMES), dtype=torch.float32, device=device)  # stored amaxes
        self.current = torch.zeros(len(C4_NAMES), dtype=torch.float32, device=device)  # max|x| by-products
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.flops = 6 * 2 * M * Hd * F

    def _g(self, name):
        j = C4_NAMES.index(name)
        return self.stored[j:j + 1], self.current[j:j + 1]

    def _quant(self, name, x, refresh, r_row, seed_row, r_col, seed_col):
        fp4 = self.fp4
        q = self.q[name]
        g, cur = self._g(name)
        if refresh:
            fp4.fp4_amax(x, g)  # the refresh: this step's max |x| becomes the stored amax
        fp4.fp4_quantize_dual(x, "UE5M3", r_row, seed_row, r_col, seed_col, g, fp4.FP4_SFLAYOUT_MMA, q["cr"], q["sr"],
                              q["cc"], q["sc"], None if refresh else cur, self.status, ue5m3_shift_out=q["t"])
        fp4.fp4_ue5m3_reencode(q["sr"], q["t"][0:1], q["er"], self.status)
        fp4.fp4_ue5m3_reencode(q["sc"], q["t"][1:2], q["ec"], self.status)

    def _gemm(self, a, a_col, b, b_col, M, N, K, out):
        fp4 = self.fp4
        qa, qb = self.q[a], self.q[b]
        ga, gb = self._g(a)[0], self._g(b)[0]
        ca, ea, ta = (qa["cc"], qa["ec"], qa["t"][1:2]) if a_col else (qa["cr"], qa["er"], qa["t"][0:1])
        cb, eb, tb = (qb["cc"], qb["ec"], qb["t"][1:2]) if b_col else (qb["cr"], qb["er"], qb["t"][0:1])
        fp4.fp4_gemm(ca, ea, cb, eb, ga, gb, ta, tb, M, N, K, "UE5M3", fp4.FP4_OUT_BF16, out, dev_status=self.status)

    def run(self, t, X, dY, ev=None):
        """Step t on inputs X [M, H], dY [M, H]; ev: optional list of 13 CUDA
        events (quantization and GEMM phases alternate)."""
        fp4 = self.fp4
        RNE, SR = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC
        M, Hd, F = self.M, self.Hd, self.F
        refresh = t % C4_PERIOD == 0
        seed = 1234 + 8 * t
        st = torch.cuda.current_stream()

        def mark(i):
            if ev is not None:
                ev[i].record(st)

        mark(0)
        self._quant("X", X, refresh, RNE, 0, RNE, 0)
        self._quant("W1", self.W1, refresh, RNE, 0, RNE, 0)
        mark(1)
        self._gemm("X", False, "W1", False, M, F, Hd, self.H)                 # L1 fwd
        mark(2)
        self._quant("H", self.H, refresh, RNE, 0, RNE, 0)
        self._quant("W2", self.W2, refresh, RNE, 0, RNE, 0)
        mark(3)
        self._gemm("H", False, "W2", False, M, Hd, F, self.Y)                 # L2 fwd
        mark(4)
        self._quant("dY", dY, refresh, SR, seed + 0, SR, seed + 1)
        mark(5)
        self._gemm("dY", False, "W2", True, M, F, Hd, self.dH)                # L2 dgrad
        mark(6)
        self._gemm("dY", True, "H", True, Hd, F, M, self.dW2)                 # L2 wgrad
        mark(7)
        self._quant("dH", self.dH, refresh, SR, seed + 2, SR, seed + 3)
        mark(8)
        self._gemm("dH", False, "W1", True, M, Hd, F, self.dX)                # L1 dgrad
        mark(9)
        self._gemm("dH", True, "X", True, F, Hd, M, self.dW1)                 # L1 wgrad
        mark(10)

    def launches(self, refresh):
        # 6 x (dual quantizer + shift finalize + 2 re-encodes) + 6 GEMMs (+ 6 amax on refresh steps)
        return 6 * 4 + 6 + (6 if refresh else 0)


def stack_study(device, reps=3):
    """The UE5M3 stack at full size: per step (a refresh step and a stale one,
    each timed alone after an L2 flush) and the whole 100-step sequence with
    refreshes at t = 0 and 50 (inputs drawn on the device between steps,
    outside the events; every step's kernels inside)."""
    from fp4_block_scaled_amax_gb300 import synth
    s = StackStep(device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(11)]
    per_phase = {"quant": 0.0, "gemm": 0.0}
    step_ms = []
    seq_ms = []
    for t in range(C4_STEPS):
        d = synth.config4_step_device(t, device)
        flush.zero_()
        torch.cuda.synchronize()
        s.run(t, d["X"], d["dY"], ev)
        torch.cuda.synchronize()
        ms = ev[0].elapsed_time(ev[10])
        seq_ms.append(ms)
        if t in (1, 2, 3):  # stale steps: the breakdown of the usual step
            step_ms.append(ms)
            for i in range(10):
                per_phase["gemm" if i in (1, 3, 5, 6, 8, 9) else "quant"] += ev[i].elapsed_time(ev[i + 1])
    if int(s.status.item()) != 0:
        raise RuntimeError(f"stack: device status {int(s.status.item())}")
    stale = statistics.median(seq_ms[1:C4_PERIOD])
    refresh = statistics.mean([seq_ms[0], seq_ms[C4_PERIOD]])
    total = sum(seq_ms)
    gemm_ms = per_phase["gemm"] / len(step_ms)
    return {"workload": f"nemotron-h-8b-like stack {C4_M} tokens x {C4_H} -> {C4_F} -> {C4_H}, UE5M3 g16, "
                        "fwd RNE, dY/dH SR, amax refreshed at t % 50 == 0",
            "unit": "ms", "step_refresh_ms": round(refresh, 4), "step_stale_ms": round(stale, 4),
            "step_stale_tflops": round(s.flops / (stale * 1e-3) / 1e12, 1),
            "gemm_ms_per_step": round(gemm_ms, 4),
            "gemm_tflops": round(s.flops / (gemm_ms * 1e-3) / 1e12, 1),
            "quant_reencode_amax_ms_per_step": round(per_phase["quant"] / len(step_ms), 4),
            "sequence_100_steps_ms": round(total, 2),
            "sequence_tflops": round(C4_STEPS * s.flops / (total * 1e-3) / 1e12, 1),
            "launches_per_step": {"refresh": s.launches(True), "stale": s.launches(False)}}


def quantizer_modes(step, flush, reps=5):
    """Given-amax quantizer of dY (the step's largest tensor) in each mode, timed
    alone with CUDA events after an L2 flush: row or transposed layout at
    2.5625 B/elem, both at once at 3.125 B/elem.  Outside the timed step."""
    fp4 = step.fp4
    RNE, SR, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA
    x, g = step.dY, step.amax[2:3]
    cr, srs, cc, scs = step.q["dY"]
    R, C = x.shape
    n = R * C
    hbm = peaks()[0]
    modes = {
        "rne_row": (2.5625, lambda: fp4.fp4_quantize(x, "E4M3", RNE, 0, g, False, MMA, cr, srs, None)),
        "rne_col": (2.5625, lambda: fp4.fp4_quantize(x, "E4M3", RNE, 0, g, True, MMA, cc, scs, None)),
        "sr_row": (2.5625, lambda: fp4.fp4_quantize(x, "E4M3", SR, 1234, g, False, MMA, cr, srs, None)),
        "sr_col": (2.5625, lambda: fp4.fp4_quantize(x, "E4M3", SR, 1235, g, True, MMA, cc, scs, None)),
        "dual_rne": (3.125, lambda: fp4.fp4_quantize_dual(x, "E4M3", RNE, 0, RNE, 0, g, MMA, cr, srs, cc, scs)),
        "dual_sr": (3.125, lambda: fp4.fp4_quantize_dual(x, "E4M3", SR, 1234, SR, 1235, g, MMA, cr, srs, cc, scs)),
    }
    out = {"tensor": f"dY {R}x{C} bf16, E4M3 g16, given amax", "unit": "GB/s", "peak": hbm}
    st = torch.cuda.current_stream()
    for name, (bpe, fn) in modes.items():
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        gbs = n * bpe / (statistics.median(ts) * 1e-3) / 1e9
        out[name] = {"us": round(statistics.median(ts) * 1e3, 2), "achieved": round(gbs, 1),
                     "frac": round(gbs / hbm, 4), "bytes_per_elem": bpe}
    return out


SWEEP_FORMATS = ["E4M3", "UE5M3", "E8M0", "E1M6", "E2M5", "E3M4", "E5M2", "E6M1", "E7M0", "NVINT4", "MXINT4"]


def scale_format_sweep(fp4, flush, device, reps=5):
    """Row quantizer (RNE, fresh amax given) on the 350M-parameter MLP input
    X 8192x1024 (per-column sigma log-uniform in [0.1, 10]) for every scale
    format and both INT4 grids: GB/s at 2 + 0.5 + 1/G B/elem, and the relative
    RMS error of the dequantized tensor.  Outside the timed step."""
    from fp4_block_scaled_amax_gb300 import synth
    x = synth.config2()["X"].to(device)
    M, K = x.shape
    g = x.float().abs().max().reshape(1)
    xf = x.float()
    ref_norm = float(xf.pow(2).mean().sqrt())
    hbm = peaks()[0]
    out = {"tensor": f"X {M}x{K} bf16 (350M MLP input), RNE rows, fresh amax", "unit": "GB/s", "peak": hbm}
    st = torch.cuda.current_stream()
    deq = torch.empty((M, K), dtype=torch.float32, device=device)
    for f in SWEEP_FORMATS:
        G = 32 if f in ("E8M0", "MXINT4") else 16
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        scales = torch.empty(M * K // G, dtype=torch.uint8, device=device)
        def run():
            fp4.fp4_quantize(x, f, fp4.FP4_ROUND_RNE, 0, g, False, fp4.FP4_SFLAYOUT_PLAIN, codes, scales, None)
        run()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            run()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        us = statistics.median(ts) * 1e3
        gbs = M * K * (2 + 0.5 + 1 / G) / us / 1e3
        fp4.fp4_dequantize(codes, scales, fp4.FP4_SFLAYOUT_PLAIN, M, K, f, g, fp4.FP4_OUT_F32, deq)
        rel_rmse = float((deq - xf).pow(2).mean().sqrt()) / ref_norm
        out[f] = {"us": round(us, 2), "achieved": round(gbs, 1), "frac": round(gbs / hbm, 4),
                  "rel_rmse": round(rel_rmse, 5)}
    return out


def _time_ms(fn, flush, reps):
    """Median of reps CUDA-event timings of fn(), each after an L2 flush."""
    st = torch.cuda.current_stream()
    fn()
    ts = []
    for _ in range(reps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(st)
        fn()
        e1.record(st)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    return statistics.median(ts)


def _ue5m3_operand(fp4, x, sr, seed, device):
    """Dual UE5M3 quantization of x with the shifts and E4M3 re-encodes the
    GEMM takes: ((row codes, row E4M3 scales, t_row), (col codes, col scales,
    t_col), amax)."""
    R, C = x.shape
    u8 = dict(dtype=torch.uint8, device=device)
    cr, srs, cc, scs = (torch.empty((R, C // 2), **u8), torch.empty(R * C // 16, **u8),
                        torch.empty((C, R // 2), **u8), torch.empty(R * C // 16, **u8))
    er, ec = torch.empty_like(srs), torch.empty_like(scs)
    t = torch.zeros(2, dtype=torch.int32, device=device)
    g = torch.zeros(1, dtype=torch.float32, device=device)
    rnd = fp4.FP4_ROUND_STOCHASTIC if sr else fp4.FP4_ROUND_RNE
    fp4.fp4_quantize_dual(x, "UE5M3", rnd, seed, rnd, seed + 1, None, fp4.FP4_SFLAYOUT_MMA, cr, srs, cc, scs, g,
                          ue5m3_shift_out=t)
    fp4.fp4_ue5m3_reencode(srs, t[0:1], er)
    fp4.fp4_ue5m3_reencode(scs, t[1:2], ec)
    return (cr, er, t[0:1]), (cc, ec, t[1:2]), g


def formats_7b_study(step, flush, reps=5):
    """Forward, dgrad and wgrad FP4 GEMMs of the 7B step (bf16 out) in each
    tensor-core scale format: NVFP4 (E4M3, group 16, scale_vec::4X), UE5M3
    (group 16, shifted onto the E4M3 path) and MXFP4 (E8M0, group 32,
    scale_vec::2X); operands quantized by the library once, outside the
    events."""
    fp4 = step.fp4
    dev = step.dev
    M, K, N = M_TOK, K_HID, N_FFN
    RNE, SR, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA
    out = {"shapes": {"fwd": [M, N, K], "dgrad": [M, K, N], "wgrad": [N, K, M]}, "unit": "ms", "out": "bf16"}
    C = {"fwd": step.Y, "dgrad": step.dX, "wgrad": step.dW}
    for fmt in ("E4M3", "UE5M3", "E8M0"):
        if fmt == "UE5M3":
            xr, xc, gx = _ue5m3_operand(fp4, step.X, False, 0, dev)
            wr, wc, gw = _ue5m3_operand(fp4, step.W, False, 0, dev)
            dr, dc, gd = _ue5m3_operand(fp4, step.dY, True, 1234, dev)
        else:
            G = 32 if fmt == "E8M0" else 16
            ops = []
            for x, sr in ((step.X, False), (step.W, False), (step.dY, True)):
                R, Cc = x.shape
                cr = torch.empty((R, Cc // 2), dtype=torch.uint8, device=dev)
                srs = torch.empty(R * Cc // G, dtype=torch.uint8, device=dev)
                cc = torch.empty((Cc, R // 2), dtype=torch.uint8, device=dev)
                scs = torch.empty(R * Cc // G, dtype=torch.uint8, device=dev)
                g = torch.zeros(1, dtype=torch.float32, device=dev)
                rnd = SR if sr else RNE
                fp4.fp4_quantize_dual(x, fmt, rnd, 1234, rnd, 1235, None, MMA, cr, srs, cc, scs, g)
                ops.append(((cr, srs, None), (cc, scs, None), g))
            (xr, xc, gx), (wr, wc, gw), (dr, dc, gd) = ops
        calls = {"fwd": (xr, gx, wr, gw, M, N, K), "dgrad": (dr, gd, wc, gw, M, K, N),
                 "wgrad": (dc, gd, xc, gx, N, K, M)}
        res = {}
        for name, (a, ga, b, gb, m, n, k) in calls.items():
            def run(a=a, ga=ga, b=b, gb=gb, m=m, n=n, k=k, c=C[name]):
                fp4.fp4_gemm(a[0], a[1], b[0], b[1], ga, gb, a[2], b[2], m, n, k, fmt, fp4.FP4_OUT_BF16, c,
                             dev_status=step.status)
            ms = _time_ms(run, flush, reps)
            res[name] = {"ms": round(ms, 4), "tflops": round(2 * m * n * k / (ms * 1e-3) / 1e12, 1)}
        res["mean_tflops"] = round(statistics.mean(v["tflops"] for v in res.values()), 1)
        out[fmt] = res
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"formats_7b: device status {int(step.status.item())}")
    return out


def cublaslt_nvfp4_study(step, flush, reps=5):
    """cuBLASLt's NVFP4 GEMM (torch._scaled_mm on the library's own E4M3
    codes and tiled scales, the blocked layout cuBLASLt reads; bf16 out,
    without the per-tensor alpha) on the step's three shapes, timed like the
    library's kernel: the vendor GEMM beside ours, outside the timed step."""
    fp4_dt = getattr(torch, "float4_e2m1fn_x2", None)
    if fp4_dt is None or not hasattr(torch, "_scaled_mm"):
        return {"unavailable": "this torch has no float4_e2m1fn_x2 / _scaled_mm"}
    M, K, N = M_TOK, K_HID, N_FFN
    qX, qW, qd = step.q["X"], step.q["W"], step.q["dY"]
    e4 = torch.float8_e4m3fn
    calls = {"fwd": (qX[0], qX[1], qW[0], qW[1], M, N, K), "dgrad": (qd[0], qd[1], qW[2], qW[3], M, K, N),
             "wgrad": (qd[2], qd[3], qX[2], qX[3], N, K, M)}
    out = {"unit": "ms", "out": "bf16", "api": "torch._scaled_mm (NVFP4, 1x16 E4M3 block scales)"}
    try:
        for name, (a, sa, b, sb, m, n, k) in calls.items():
            A = a.view(fp4_dt)
            B = b.view(fp4_dt).t()
            SA = sa.view(e4).reshape(m, k // 16)
            SB = sb.view(e4).reshape(n, k // 16)
            ms = _time_ms(lambda: torch._scaled_mm(A, B, SA, SB, out_dtype=torch.bfloat16), flush, reps)
            out[name] = {"ms": round(ms, 4), "tflops": round(2 * m * n * k / (ms * 1e-3) / 1e12, 1)}
        out["mean_tflops"] = round(statistics.mean(out[n]["tflops"] for n in calls), 1)
    except Exception as exc:  # noqa: BLE001 - reported, not fatal
        out["unavailable"] = f"{type(exc).__name__}: {str(exc).splitlines()[0][:200]}"
    return out


def config2_study(fp4, flush, device, reps=5):
    """The 350M-parameter MLP linear Y = X W^T, 8192 x 4096 x 1024, with X's
    per-channel sigma log-uniform in [0.1, 10]: the forward FP4 GEMM (bf16
    out) in E4M3, UE5M3 and E8M0; and the range study of the review of Intel's
    FP4 paper ("Форматы FP4": only E1M6, the narrowest scale format, fails):
    per format the fraction of nonzero blocks whose scale flushes to zero or
    saturates, along rows (the forward operand) and along columns (the wgrad
    operand X^T), and the relative Frobenius error of the product of the
    dequantized operands (X_q W_q^T against X W^T, float64 on 512 sampled
    rows; E1M6 has no tensor-core path, so its product uses the library's
    codes dequantized by the library)."""
    from fp4_block_scaled_amax_gb300 import synth
    d = synth.config2()
    X, W = d["X"].to(device), d["W"].to(device)
    M, K = X.shape
    N = W.shape[0]
    MMA = fp4.FP4_SFLAYOUT_MMA
    out = {"shape": [M, N, K], "unit": "ms", "out": "bf16"}
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
    rows = torch.arange(0, M, M // 512, device=device)
    ref = (X[rows].double() @ W.double().t())
    ref_norm = float(ref.norm())
    for fmt in ("E4M3", "UE5M3", "E8M0", "E1M6"):
        G = 32 if fmt == "E8M0" else 16
        res = {}
        ops = []
        for x in (X, W):
            R, C = x.shape
            cr = torch.empty((R, C // 2), dtype=torch.uint8, device=device)
            srs = torch.empty(R * C // G, dtype=torch.uint8, device=device)
            cc = torch.empty((C, R // 2), dtype=torch.uint8, device=device)
            scs = torch.empty(R * C // G, dtype=torch.uint8, device=device)
            g = torch.zeros(1, dtype=torch.float32, device=device)
            t = torch.zeros(2, dtype=torch.int32, device=device) if fmt == "UE5M3" else None
            fp4.fp4_quantize_dual(x, fmt, fp4.FP4_ROUND_RNE, 0, fp4.FP4_ROUND_RNE, 0, None, MMA, cr, srs, cc, scs, g,
                                  ue5m3_shift_out=t)
            ops.append((cr, srs, cc, scs, g, t))
        # blocks of X holding a nonzero element whose scale code is 0 (E4M3, UE5M3, E1M6: the
        # scale and every element flush to zero; E8M0 has no zero, code 0 is 2^-127), along rows
        # and along columns
        (cr, srs, cc, scs, g, _), _ = ops
        for tag, scales, R, C in (("rows", srs, M, K), ("cols", scs, K, M)):
            sc = scales.view(R // 128, (C // G) // 4, 32, 4, 4).permute(0, 3, 2, 1, 4).reshape(-1)  # tiled -> plain
            xr = X if tag == "rows" else X.t()
            blk_nz = xr.reshape(R, C // G, G).ne(0).any(dim=2).reshape(-1)
            res[f"flushed_{tag}"] = round(float((blk_nz & (sc == 0)).sum()) / float(blk_nz.sum()), 6)
        # error of the product of the dequantized operands
        dq = []
        for (cr, srs, cc, scs, g, t), x in zip(ops, (X, W)):
            R, C = x.shape
            o = torch.empty((R, C), dtype=torch.float32, device=device)
            fp4.fp4_dequantize(cr, srs, MMA, R, C, fmt, g, fp4.FP4_OUT_F32, o)
            dq.append(o)
        prod = dq[0][rows].double() @ dq[1].double().t()
        res["product_rel_err"] = round(float((prod - ref).norm()) / ref_norm, 6)
        if fmt != "E1M6":
            (ac, as_, _, _, ga, ta), (bc, bs, _, _, gb, tb) = ops
            if fmt == "UE5M3":
                ea, eb = torch.empty_like(as_), torch.empty_like(bs)
                fp4.fp4_ue5m3_reencode(as_, ta[0:1], ea)
                fp4.fp4_ue5m3_reencode(bs, tb[0:1], eb)
                as_, bs, ta, tb = ea, eb, ta[0:1], tb[0:1]
            ms = _time_ms(lambda: fp4.fp4_gemm(ac, as_, bc, bs, ga, gb, ta, tb, M, N, K, fmt, fp4.FP4_OUT_BF16, Y),
                          flush, reps)
            res["gemm_ms"] = round(ms, 4)
            res["gemm_tflops"] = round(2 * M * N * K / (ms * 1e-3) / 1e12, 1)
            res["gemm_rel_err"] = round(float((Y[rows].double() - prod).norm()) / float(prod.norm()), 6)
        out[fmt] = res
    return out


RHT_MASK = 0xB38D  # sign mask of the 16 x 16 random Hadamard transform (any 16-bit value)


def hadamard_study(step, fp4, flush, device, reps=5):
    """16 x 16 random Hadamard transform before quantization, outside the timed
    step: (1) its cost on the given-amax E4M3 quantizers of dY (GB/s with and
    without the transform: the row quantizer, 2.5625 B/elem, and the dual
    row + transposed SR quantizer, 3.125 B/elem); (2) relative RMS error of NVFP4 /
    NVINT4 / MXFP4 / MXINT4 on the 350M MLP input X 8192x1024 with and without
    the transform (fresh amax; with it, measured against the transformed
    tensor, whose norm the orthogonal transform keeps)."""
    from fp4_block_scaled_amax_gb300 import synth
    hbm = peaks()[0]
    st = torch.cuda.current_stream()

    def timed(fn):
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return statistics.median(ts) * 1e3

    x, g = step.dY, step.amax[2:3]
    cr, srs, _, _ = step.q["dY"]
    n = x.numel()
    RNE, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_SFLAYOUT_MMA
    us_plain = timed(lambda: fp4.fp4_quantize(x, "E4M3", RNE, 0, g, False, MMA, cr, srs, None))
    us_rht = timed(lambda: fp4.fp4_quantize_rht(x, "E4M3", RNE, 0, RHT_MASK, g, MMA, cr, srs, None))
    _, _, cc, scs = step.q["dY"]
    SR = fp4.FP4_ROUND_STOCHASTIC
    us_dual = timed(lambda: fp4.fp4_quantize_dual(x, "E4M3", SR, 1234, SR, 1235, g, MMA, cr, srs, cc, scs))
    us_dual_rht = timed(lambda: fp4.fp4_quantize_dual_rht(x, "E4M3", SR, 1234, SR, 1235, RHT_MASK, g, g, MMA,
                                                           cr, srs, cc, scs))
    out = {"cost": {"tensor": f"dY {x.shape[0]}x{x.shape[1]}, E4M3 RNE rows, given amax", "unit": "GB/s",
                    "plain": round(n * 2.5625 / us_plain / 1e3, 1), "with_rht": round(n * 2.5625 / us_rht / 1e3, 1),
                    "us_plain": round(us_plain, 2), "us_rht": round(us_rht, 2), "peak": hbm},
           "cost_dual": {"tensor": f"dY {x.shape[0]}x{x.shape[1]}, E4M3 SR rows + SR transposed, given amax",
                         "unit": "GB/s", "plain": round(n * 3.125 / us_dual / 1e3, 1),
                         "with_rht": round(n * 3.125 / us_dual_rht / 1e3, 1), "us_plain": round(us_dual, 2),
                         "us_rht": round(us_dual_rht, 2), "peak": hbm}}
    X = synth.config2()["X"].to(device)
    M, K = X.shape
    Xf = X.float()
    i = torch.arange(16, device=device)
    par = torch.zeros((16, 16), dtype=torch.int64, device=device)
    for b in range(4):
        par += ((i[:, None] & i[None, :]) >> b) & 1
    H = 1.0 - 2.0 * (par % 2).double()
    sgn = torch.tensor([-1.0 if (RHT_MASK >> j) & 1 else 1.0 for j in range(16)], dtype=torch.float64, device=device)
    T = 0.25 * H * sgn[None, :]
    Xt = (Xf.double().reshape(-1, 16) @ T.T).reshape(M, K)  # reference only (float64)
    deq = torch.empty((M, K), dtype=torch.float32, device=device)
    amax = torch.zeros(1, dtype=torch.float32, device=device)
    errs = {}
    for f in ("E4M3", "NVINT4", "E8M0", "MXINT4"):
        G = 32 if f in ("E8M0", "MXINT4") else 16
        codes = torch.empty((M, K // 2), dtype=torch.uint8, device=device)
        scales = torch.empty(M * K // G, dtype=torch.uint8, device=device)
        e = {}
        for name, use in (("plain", False), ("rht", True)):
            if use:
                fp4.fp4_quantize_rht(X, f, RNE, 0, RHT_MASK, None, fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax)
                ref = Xt
            else:
                fp4.fp4_quantize(X, f, RNE, 0, None, False, fp4.FP4_SFLAYOUT_PLAIN, codes, scales, amax)
                ref = Xf.double()
            fp4.fp4_dequantize(codes, scales, fp4.FP4_SFLAYOUT_PLAIN, M, K, f, amax, fp4.FP4_OUT_F32, deq)
            e[name] = round(float((deq.double() - ref).norm() / ref.norm()), 5)
        errs[{"E4M3": "NVFP4", "E8M0": "MXFP4"}.get(f, f)] = e
    out["rel_rmse"] = {"tensor": f"X {M}x{K} (350M MLP input), RNE rows, fresh amax", **errs}
    return out


def step_variants_study(step, flush, reps=5):
    """The linear layer's forward + backward (three quantizations, three
    GEMMs; no GEMV) in four forms, each timed end to end with CUDA events
    after an L2 flush: bf16 cuBLAS GEMMs (torch.matmul, the BF16 baseline the
    UE5M3 blog compares against), FP4 with a fresh amax per tensor (the timed
    step), FP4 with the stored amax (the UE5M3 recipe between refreshes, no
    amax pass), and FP4 with the 16 x 16 random Hadamard transform and fresh
    amaxes of the transformed tensors (the variant the recipe removes).
    Outside the timed step."""
    fp4 = step.fp4
    M, K, N = M_TOK, K_HID, N_FFN
    RNE, SR, MMA, BF = fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA, fp4.FP4_OUT_BF16
    dev = step.Y.device
    plan = [("X", RNE, 0, SR, 1236), ("W", RNE, 0, RNE, 0), ("dY", SR, 1234, SR, 1235)]
    rht_amax = torch.zeros(6, dtype=torch.float32, device=dev)
    qX, qW, qd = step.q["X"], step.q["W"], step.q["dY"]
    st = torch.cuda.current_stream()

    def gemms(a):
        aX, aW, ad = a[0:1], a[1:2], a[2:3]
        fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", BF, step.Y)
        fp4.fp4_gemm(qd[0], qd[1], qW[2], qW[3], ad, aW, None, None, M, K, N, "E4M3", BF, step.dX)
        fp4.fp4_gemm(qd[2], qd[3], qX[2], qX[3], ad, aX, None, None, N, K, M, "E4M3", BF, step.dW)

    def bf16_step():
        torch.matmul(step.X, step.W.t(), out=step.Y)
        torch.matmul(step.dY, step.W, out=step.dX)
        torch.matmul(step.dY.t(), step.X, out=step.dW)

    def fp4_step(fresh):
        if fresh:
            fp4.fp4_amax_n([step.X, step.W, step.dY], step.amax)
        for j, (name, rr, sr, rc, sc) in enumerate(plan):
            x, a = getattr(step, name), step.amax[j:j + 1]
            cr, srs, cc, scs = step.q[name]
            fp4.fp4_quantize_dual(x, "E4M3", rr, sr, rc, sc, a, MMA, cr, srs, cc, scs)
        gemms(step.amax)

    def rht_step():
        for j, (name, rr, sr, rc, sc) in enumerate(plan):
            cr, srs, cc, scs = step.q[name]
            fp4.fp4_quantize_dual_rht(getattr(step, name), "E4M3", rr, sr, rc, sc, RHT_MASK, None, None, MMA,
                                      cr, srs, cc, scs, rht_amax[2 * j:2 * j + 1], rht_amax[2 * j + 1:2 * j + 2])
        # rows of X, W, dY carry their row-transform amax; the transposed operands their column one
        fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], rht_amax[0:1], rht_amax[2:3], None, None, M, N, K, "E4M3", BF,
                     step.Y)
        fp4.fp4_gemm(qd[0], qd[1], qW[2], qW[3], rht_amax[4:5], rht_amax[3:4], None, None, M, K, N, "E4M3", BF,
                     step.dX)
        fp4.fp4_gemm(qd[2], qd[3], qX[2], qX[3], rht_amax[5:6], rht_amax[1:2], None, None, N, K, M, "E4M3", BF,
                     step.dW)

    variants = [("bf16_cublas", bf16_step), ("fp4_fresh_amax", lambda: fp4_step(True)),
                ("fp4_stored_amax", lambda: fp4_step(False)), ("fp4_rht16_fresh_amax", rht_step)]
    flops = 3 * 2 * M * N * K
    res = {"linear": f"fwd + dgrad + wgrad, {M} tokens x {K} -> {N}", "unit": "ms"}
    for name, fn in variants:
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        res[name] = {"ms": round(ms, 4), "TFLOP/s": round(flops / (ms * 1e-3) / 1e12, 1)}
    base = res["bf16_cublas"]["ms"]
    for name in ("fp4_fresh_amax", "fp4_stored_amax", "fp4_rht16_fresh_amax"):
        res[name]["speedup_vs_bf16"] = round(base / res[name]["ms"], 3)
    res["rht_removal_gain"] = round(res["fp4_rht16_fresh_amax"]["ms"] / res["fp4_fresh_amax"]["ms"] - 1, 4)
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    return res


def ue5m3_windows_study(step, flush, reps=3):
    """The forward GEMM 16384 x 11008 x 4096 on UE5M3 operands (float32 out):
    the single-shift path (fp4_ue5m3_to_e4m3 + fp4_gemm) against the
    window path (fp4_ue5m3_windows + fp4_gemm_ue5m3_windows), A = X with a
    fresh amax (one window: the window path only adds launches), and A = a
    seeded 16384 x 4096 tensor whose 16-element blocks are scaled by
    2^U(-30, 0), with a stored amax 256x below its maximum (scales from
    UE5M3's top to its bottom: three windows, where the single shift is not
    exact).  B = W, fresh amax.  Scale preparation included in both.
    Outside the timed step."""
    fp4 = step.fp4
    M, N, K = M_TOK, N_FFN, K_HID
    dev = step.Y.device
    RNE, MMA = fp4.FP4_ROUND_RNE, fp4.FP4_SFLAYOUT_MMA
    u8 = dict(dtype=torch.uint8, device=dev)
    i32 = dict(dtype=torch.int32, device=dev)
    C = torch.empty((M, N), dtype=torch.float32, device=dev)
    st = torch.cuda.current_stream()
    res = {"gemm": f"fwd {M}x{N}x{K}, UE5M3 scales, float32 out", "unit": "ms"}
    gen = torch.Generator(device=dev)
    gen.manual_seed(60)
    wide = torch.randn(M, K, device=dev, generator=gen)
    wide = (wide * torch.exp2(-30.0 * torch.rand(M, K // 16, device=dev, generator=gen)).repeat_interleave(16, 1))
    wide = wide.to(torch.bfloat16)
    wide_amax = (wide.float().abs().max() / 256.0).reshape(1)
    for label, a_in, a_amax in (("X_fresh_amax", step.X, step.amax[0:1]),
                                ("wide_blocks_stored_amax", wide, wide_amax)):
        ops = {}
        for name, x, amax in (("X", a_in, a_amax), ("W", step.W, step.amax[1:2])):
            R = x.shape[0]
            codes, scales = torch.empty((R, K // 2), **u8), torch.empty(R * K // 16, **u8)
            amax = amax.contiguous().clone()
            fp4.fp4_quantize(x, "UE5M3", RNE, 0, amax, False, MMA, codes, scales, None)
            ops[name] = (codes, scales, amax, torch.empty_like(scales), torch.zeros(1, **i32),
                         torch.empty(3 * scales.numel(), **u8), torch.zeros(3, **i32), torch.zeros(1, **i32))
        (xc, xs, xa, xe, xt, xw, xwt, xn), (wc, ws, wa, we, wt, ww, wwt, wn) = ops["X"], ops["W"]

        def single():
            fp4.fp4_ue5m3_to_e4m3(xs, xt, xe)
            fp4.fp4_ue5m3_to_e4m3(ws, wt, we)
            fp4.fp4_gemm(xc, xe, wc, we, xa, wa, xt, wt, M, N, K, "UE5M3", fp4.FP4_OUT_F32, C)

        def windows():
            fp4.fp4_ue5m3_windows(xs, xwt, xn, xw)
            fp4.fp4_ue5m3_windows(ws, wwt, wn, ww)
            fp4.fp4_gemm_ue5m3_windows(xc, xw, xwt, xn, wc, ww, wwt, wn, xa, wa, M, N, K, C)

        out = {}
        for name, fn in (("single_shift", single), ("windows", windows)):
            fn()
            ts = []
            for _ in range(reps):
                flush.zero_()
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(st)
                fn()
                e1.record(st)
                torch.cuda.synchronize()
                ts.append(e0.elapsed_time(e1))
            out[name] = round(statistics.median(ts), 4)
        out["windows_in_use"] = [int(xn.item()), int(wn.item())]
        # how far the single shift's result (inexact scales rounded) is from the exact window sum
        windows()
        ref = C.clone()
        single()
        out["single_shift_rel_err"] = float((C - ref).norm() / ref.norm())
        del ref
        res[label] = out
    del wide
    return res


def gemv_graph_study(step, reps=5, launches=64, copies=8):
    """Weight-only GEMV as a decode loop would issue it: `launches` launches
    back to back over `copies` copies of the 11008 x 4096 NVFP4 weight
    (8 x 25.6 MB > L2, so each launch streams its weights from HBM), issued
    one by one on the stream against replayed from one captured CUDA graph.
    Per-launch time, outside the timed step."""
    fp4 = step.fp4
    N, K = N_FFN, K_HID
    dev = step.Y.device
    BF = fp4.FP4_OUT_BF16
    ws = [(step.Wg_codes, step.Wg_scales, step.Wg_amax)]
    for _ in range(copies - 1):
        ws.append((step.Wg_codes.clone(), step.Wg_scales.clone(), step.Wg_amax.clone()))
    y = torch.empty((GEMV_BATCH, N), dtype=torch.bfloat16, device=dev)

    def loop():
        for i in range(launches):
            c, sc, a = ws[i % copies]
            fp4.fp4_gemv_w4a16(c, sc, a, step.xg, GEMV_BATCH, N, K, BF, y)

    loop()
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            loop()
    torch.cuda.current_stream().wait_stream(side)
    st = torch.cuda.current_stream()
    res = {"gemv": f"batch {GEMV_BATCH}, {N}x{K}, {launches} launches over {copies} weight copies", "unit": "us/launch"}
    gv_bytes = N * K * (0.5 + 1 / 16) + 2 * GEMV_BATCH * (N + K)
    for name, fn in (("stream", loop), ("cuda_graph", graph.replay)):
        fn()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3 / launches)
        us = statistics.median(ts)
        res[name] = {"us": round(us, 2), "GB/s": round(gv_bytes / us / 1e3, 1)}
    del graph
    return res


def capture_step(step):
    """step.run() captured as one CUDA graph (on a side stream, as capture
    requires; its fork to the wgrad and GEMV streams joins back inside)."""
    st = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    side.wait_stream(st)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            step.run()
    st.wait_stream(side)
    return graph


def step_graph_study(step, flush, reps=5):
    """The timed step (10 launches) replayed from one captured CUDA graph
    against the same step launched one kernel at a time, each timed with
    CUDA events after an L2 flush.  Outside the timed step."""
    st = torch.cuda.current_stream()
    step.run()
    torch.cuda.synchronize()
    graph = capture_step(step)
    res = {"step": "the timed step: 3 amax, 3 dual quantizations, 3 GEMMs, GEMV", "unit": "ms"}
    for name, fn in (("eager", step.run), ("cuda_graph", graph.replay)):
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms = statistics.median(ts)
        res[name] = {"ms": round(ms, 4), "TFLOP/s": round(STEP_FLOPS / (ms * 1e-3) / 1e12, 1)}
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    del graph
    return res


def gemv_shapes_study(step, reps=5, launches=32):
    """The weight-only GEMV on the Qwen2.5-7B-like MLP shapes, W_up 18944 x
    3584 and W_down 3584 x 18944 (NVFP4, quantized once), at batch 1, 8 and
    64: per-launch time over `launches` back-to-back launches that rotate over
    enough weight copies to exceed L2 (each launch streams its weights from
    HBM), issued one by one and replayed from a CUDA graph.  K is a multiple
    of 256 on both shapes, so batches 1 and 8 run the TMA-fed mma.sync kernel
    (k_gemv_w4a16_tma) and batch 64 the tcgen05 one (k_gemv_w4a16_umma); the
    long K of W_down splits over clusters of CTAs in both.  Outside the
    timed step."""
    from fp4_block_scaled_amax_gb300 import synth
    fp4 = step.fp4
    dev = step.Y.device
    BF, RNE, PLAIN = fp4.FP4_OUT_BF16, fp4.FP4_ROUND_RNE, fp4.FP4_SFLAYOUT_PLAIN
    st = torch.cuda.current_stream()
    res = {"unit": "us/launch"}
    for wname, xname in (("W_up", "x_up"), ("W_down", "x_down")):
        W = synth.config5(1)[wname].to(dev)
        N, K = W.shape
        codes = torch.empty((N, K // 2), dtype=torch.uint8, device=dev)
        scales = torch.empty(N * K // 16, dtype=torch.uint8, device=dev)
        amax = torch.zeros(1, dtype=torch.float32, device=dev)
        fp4.fp4_quantize(W, "E4M3", RNE, 0, None, False, PLAIN, codes, scales, amax)
        del W
        wbytes = N * K * (0.5 + 1 / 16)
        copies = max(2, int(300e6 // wbytes) + 1)
        ws = [(codes, scales)] + [(codes.clone(), scales.clone()) for _ in range(copies - 1)]
        out = {}
        for b in (1, 8, 64):
            x = synth.config5(b)[xname].to(dev)
            y = torch.empty((b, N), dtype=torch.bfloat16, device=dev)

            def loop():
                for i in range(launches):
                    c, sc = ws[i % copies]
                    fp4.fp4_gemv_w4a16(c, sc, amax, x, b, N, K, BF, y)

            loop()
            # the same launches replayed from one CUDA graph (no host launch cost between them)
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph):
                loop()
            graph.replay()

            def timed(fn):
                ts = []
                for _ in range(reps):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(st)
                    fn()
                    e1.record(st)
                    torch.cuda.synchronize()
                    ts.append(e0.elapsed_time(e1) * 1e3 / launches)
                return statistics.median(ts)

            us, gus = timed(loop), timed(graph.replay)
            nbytes = wbytes + 2 * b * (N + K)
            out[f"batch_{b}"] = {"us": round(us, 2), "GB/s": round(nbytes / us / 1e3, 1),
                                 "graph_us": round(gus, 2), "graph_GB/s": round(nbytes / gus / 1e3, 1),
                                 "graph_frac": round(nbytes / gus / 1e3 / peaks()[0], 4)}
            del graph
        res[f"{wname} {N}x{K}"] = out
        del ws
    return res


def fused_epilogue_study(step, flush, reps=5):
    """The forward GEMM Y = X W^T with Y quantized for the next layer (NVFP4,
    the stored amax of Y), outside the timed step:
      * rows only (RNE): the GEMM writing bf16 Y followed by the row
        quantizer, against the GEMM quantizing Y in its epilogue
        (fp4_gemm_quantize);
      * rows (RNE) and columns (SR, the layout of Y^T the backward pass
        takes): the GEMM, then the one-read dual quantizer, against the dual
        quantizing epilogue (fp4_gemm_quantize_dual)."""
    fp4 = step.fp4
    M, N, K = M_TOK, N_FFN, K_HID
    qX, qW = step.q["X"], step.q["W"]
    aX, aW = step.amax[0:1], step.amax[1:2]
    BF, RNE, SR, MMA = fp4.FP4_OUT_BF16, fp4.FP4_ROUND_RNE, fp4.FP4_ROUND_STOCHASTIC, fp4.FP4_SFLAYOUT_MMA
    dev = step.Y.device
    codes = torch.empty((M, N // 2), dtype=torch.uint8, device=dev)
    scales = torch.empty(M * N // 16, dtype=torch.uint8, device=dev)
    tcodes = torch.empty((N, M // 2), dtype=torch.uint8, device=dev)
    tscales = torch.empty(M * N // 16, dtype=torch.uint8, device=dev)
    fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", BF, step.Y)
    gY = step.Y.float().abs().max().reshape(1)  # the stored amax of Y
    st = torch.cuda.current_stream()

    def two_calls():
        fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", BF, step.Y)
        fp4.fp4_quantize(step.Y, "E4M3", RNE, 0, gY, False, MMA, codes, scales, None)

    def one_call():
        fp4.fp4_gemm_quantize(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", gY, RNE, 0, MMA,
                              codes, scales)

    def two_calls_dual():
        fp4.fp4_gemm(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", BF, step.Y)
        fp4.fp4_quantize_dual(step.Y, "E4M3", RNE, 0, SR, 9, gY, MMA, codes, scales, tcodes, tscales, None)

    def one_call_dual():
        fp4.fp4_gemm_quantize_dual(qX[0], qX[1], qW[0], qW[1], aX, aW, None, None, M, N, K, "E4M3", gY, RNE, 0, SR,
                                   9, MMA, codes, scales, tcodes, tscales)

    res = {}
    for name, fn in (("gemm_then_quantize", two_calls), ("gemm_quantize_epilogue", one_call),
                     ("gemm_then_quantize_dual", two_calls_dual), ("gemm_quantize_dual_epilogue", one_call_dual)):
        fn()
        ts = []
        for _ in range(reps):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            fn()
            e1.record(st)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        res[name] = round(statistics.median(ts), 4)
    return {"gemm": f"fwd {M}x{N}x{K} E4M3, Y -> NVFP4 rows (RNE) [+ columns (SR)], stored amax", "unit": "ms", **res,
            "fused_tflops": round(2 * M * N * K / (res["gemm_quantize_epilogue"] * 1e-3) / 1e12, 1),
            "fused_dual_tflops": round(2 * M * N * K / (res["gemm_quantize_dual_epilogue"] * 1e-3) / 1e12, 1)}


def make_inputs():
    from fp4_block_scaled_amax_gb300 import synth
    d = synth.config3()
    if M_TOK != d["X"].shape[0]:
        d["X"], d["dY"] = d["X"][:M_TOK].contiguous(), d["dY"][:M_TOK].contiguous()
    d["x_dec"] = synth.normal((GEMV_BATCH, K_HID), 3, 50)
    return d


def src_hash(names):
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "fp4_block_scaled_amax_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


STUDIES = ("formats", "cublaslt", "config2", "stack", "gemv_shapes", "step_graph", "gemv_graph", "variants",
           "windows", "qmodes", "sweep", "hadamard", "fused", "ceiling")


def tensor_ceiling_study():
    """The tensor cores' FLOP per clock per SM on this GPU, from the package's
    tc_ceiling program (each SM streams 2048 MMAs of one form from one warp,
    no waits between them): kind::f16 bf16 (M 128, N 256, K 16), the FP4
    GEMM's own form (kind::mxf4nvf4 scale_vec::4X, CTA pair, M 256, N 256,
    K 64) and MXFP4 (scale_vec::2X, M 128).  Runs as its own process, outside
    the timed step."""
    from fp4_block_scaled_amax_gb300 import build as b
    try:
        exe = b.build_ceiling()
        r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    except (OSError, RuntimeError, subprocess.SubprocessError) as e:
        return {"error": str(e)[-300:]}
    if r.returncode != 0:
        return {"error": (r.stdout + r.stderr).strip()[-300:]}
    d = json.loads(r.stdout.strip().splitlines()[-1])
    d["fp4_to_bf16_per_clock"] = round(d["nvf4_pair_flop_per_clk_sm"] / d["bf16_flop_per_clk_sm"], 3)
    return d


def run_ours(args, rank, world, local):
    from fp4_block_scaled_amax_gb300 import build as b
    if rank == 0:
        b.build()
    barrier(world)
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    d = make_inputs()
    step = LinearStep(d, device)
    flush = torch.empty(512 * 1024 * 1024, dtype=torch.uint8, device=device)  # > 129 MB L2

    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())} during warm-up")

    # The timed step runs as production would run it: step.run() (its eight
    # launches on three streams) captured once as a CUDA graph and replayed
    # once per step, with an L2 flush between steps outside the events.
    graph = capture_step(step)
    graph.replay()
    torch.cuda.synchronize()
    st = torch.cuda.current_stream()
    t0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(device) as clk:
        for i in range(args.steps):
            flush.zero_()  # L2 flush between timed steps, outside the events
            t0[i].record(st)
            graph.replay()
            t1[i].record(st)
        torch.cuda.synchronize()
    barrier(world)
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())}")
    del graph

    def span(e, a, z):
        return e[a].elapsed_time(e[z])

    step_ms = [t0[i].elapsed_time(t1[i]) for i in range(args.steps)]
    ms = statistics.mean(step_ms)
    ms_max = max_over_ranks(ms, world, device)
    # Each kernel's own time comes from as many more steps launched one kernel
    # at a time, every kernel on one stream (the same launches and inputs, the
    # same L2 flush before each step), with CUDA events between the kernels.
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(STEP_EVENTS)] for _ in range(args.steps)]
    for i in range(args.steps):
        flush.zero_()
        step.run(sevs[i], serial=True)
    torch.cuda.synchronize()
    if int(step.status.item()) != 0:
        raise RuntimeError(f"device status {int(step.status.item())}")
    quant_ms = [span(e, a, a + 1) for e in sevs for a in (1, 3, 4)]
    amax_ms = [span(e, a, a + 1) for e in sevs for a in (0, 2)]
    gemm_ms = [span(e, i, i + 1) for e in sevs for i in (5, 6, 7)]
    fwd_ms = [span(e, 5, 6) for e in sevs]
    gemv_ms = [span(e, 8, 9) for e in sevs]
    serial_ms = statistics.mean(span(e, 0, 9) for e in sevs)

    hbm, bf16, src = peaks()
    fp4_peak = bf16 * FP4_PER_BF16
    gemm_tflops = 2 * M_TOK * N_FFN * K_HID / (statistics.mean(gemm_ms) * 1e-3) / 1e12
    elems = [M_TOK * K_HID, N_FFN * K_HID, M_TOK * N_FFN]
    q_bytes = sum(e * 3.125 for e in elems)          # per step, three dual quantizations
    q_gbs = q_bytes / (sum(quant_ms) / args.steps * 1e-3) / 1e9
    a_gbs = sum(e * 2 for e in elems) / (sum(amax_ms) / args.steps * 1e-3) / 1e9
    gv_bytes = N_FFN * K_HID * (0.5 + 1 / 16) + 2 * GEMV_BATCH * (N_FFN + K_HID)
    gv_gbs = gv_bytes / (statistics.mean(gemv_ms) * 1e-3) / 1e9
    def traffic_of(key):
        t = NCU_TRAFFIC.get(key)
        return t["bytes"] if t and t["src"] == src_hash(t["files"]) and M_TOK == 16384 else None
    traffic_v = traffic_of("gemm")
    qtraffic_v = traffic_of("quant_dual")
    gvtraffic_v = traffic_of("gemv")

    qmodes = sweep = hadamard = fused_ep = variants = windows = gv_graph = step_graph = gv_shapes = ceiling = None
    formats = cublas = cfg2 = stack = None
    chosen = set() if args.no_studies else (
        set(STUDIES) if args.studies == "all" else set(x.strip() for x in args.studies.split(",")))
    unknown = chosen - set(STUDIES)
    if unknown:
        raise SystemExit(f"unknown studies {sorted(unknown)}; known: {', '.join(STUDIES)}")
    if "formats" in chosen:
        formats = formats_7b_study(step, flush)
    if "cublaslt" in chosen:
        cublas = cublaslt_nvfp4_study(step, flush)
    if "config2" in chosen:
        cfg2 = config2_study(step.fp4, flush, device)
    if "stack" in chosen and M_TOK == 16384:
        stack = stack_study(device)
    if "gemv_shapes" in chosen:
        gv_shapes = gemv_shapes_study(step)
    if "step_graph" in chosen:
        step_graph = step_graph_study(step, flush)
    if "gemv_graph" in chosen:
        gv_graph = gemv_graph_study(step)
    if "variants" in chosen:
        variants = step_variants_study(step, flush)
    if "windows" in chosen:
        windows = ue5m3_windows_study(step, flush)
    if "qmodes" in chosen:
        qmodes = quantizer_modes(step, flush)
    if "sweep" in chosen:
        sweep = scale_format_sweep(step.fp4, flush, device)
    if "hadamard" in chosen:
        hadamard = hadamard_study(step, step.fp4, flush, device)
    if "fused" in chosen:
        fused_ep = fused_epilogue_study(step, flush)
    if "ceiling" in chosen:
        ceiling = tensor_ceiling_study()
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(step, d, args, world, device)

    line = {
        "metric": METRIC,
        "value": round(world * STEP_FLOPS / (ms_max * 1e-3) / 1e12, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_max, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e2m1xe2m1->f32 (tcgen05 kind::mxf4nvf4), bf16 in/out",
        "data": "synthetic (seeded; shapes and distributions of the Llama-2-7B MLP workload)",
        "config": {"workload": WORKLOAD if M_TOK == 16384 else WORKLOAD + "-reduced-tokens",
                   "tokens": M_TOK, "hidden": K_HID, "ffn": N_FFN, "scale_fmt": "E4M3",
                   "group": 16, "amax": "fresh per step", "gemm_out": "bf16", "gemv_batch": GEMV_BATCH,
                   "l2": "512 MB buffer written between timed steps (outside the events); X and dY also exceed L2",
                   "launch": "step captured as one CUDA graph (8 kernels on 3 streams), replayed per step",
                   "parallelism": f"dp{world} (independent batches)"},
        "roofline": {"kernel": "k_gemm_fp4 (mean of fwd, dgrad, wgrad)", "bound": "tensor",
                     "achieved": round(gemm_tflops, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                     "frac": round(gemm_tflops / fp4_peak, 4), "traffic": traffic_v,
                     "peak_source": f"{src}: bf16 burst {bf16} x {FP4_PER_BF16} (nominal FP4/bf16)",
                     "measured": f"each GEMM with CUDA events in {args.steps} steps launched kernel by kernel on one "
                                 "stream after the timed steps (graph replays, wgrad beside dgrad)"},
        "roofline_quantize": {"kernel": "k_quant_dual_tma (dual, 3.125 B/elem; X, W, dY per step)", "bound": "hbm",
                              "achieved": round(q_gbs, 1), "peak": hbm, "unit": "GB/s",
                              "frac": round(q_gbs / hbm, 4), "traffic": qtraffic_v, "peak_source": src,
                              "measured": "as the GEMMs'"},
        "quantize_modes": qmodes,
        "formats_7b_gemm": formats,
        "cublaslt_nvfp4": cublas,
        "config2_350m_mlp": cfg2,
        "stack_ue5m3": stack,
        "scale_format_sweep": sweep,
        "hadamard_16x16": hadamard,
        "fused_epilogue_quantize": fused_ep,
        "step_variants": variants,
        "ue5m3_windows": windows,
        "gemv_decode_loop": gv_graph,
        "gemv_qwen_mlp_shapes": gv_shapes,
        "step_cuda_graph": step_graph,
        "amax_gbs": round(a_gbs, 1),
        "roofline_amax": {"kernel": "k_amax_n (dY; X and W: two launches, 2 B/elem read)", "bound": "hbm",
                          "achieved": round(a_gbs, 1), "peak": hbm, "unit": "GB/s", "frac": round(a_gbs / hbm, 4),
                          "traffic": traffic_of("amax"), "peak_source": src,
                          "note": "the first launch after the L2 flush also writes back the flush's dirty lines",
                          "measured": "as the GEMMs'"},
        "gemv_w4a16": {"batch": GEMV_BATCH, "N": N_FFN, "K": K_HID, "us": round(statistics.mean(gemv_ms) * 1e3, 2),
                       "GB/s": round(gv_gbs, 1), "frac": round(gv_gbs / hbm, 4), "traffic": gvtraffic_v,
                       "measured": "after wgrad in the serial form of the step"},
        "kernel_ms": {"fwd_gemm": round(statistics.mean(fwd_ms), 4),
                      "gemm_mean": round(statistics.mean(gemm_ms), 4),
                      "quant_dual_total": round(sum(quant_ms) / args.steps, 4),
                      "amax_total": round(sum(amax_ms) / args.steps, 4),
                      "serial_step": round(serial_ms, 4)},
        "gpu_launches": step.launches_per_step * args.steps,
        "clocks": clk.summary(),
    }
    if ceiling is not None:
        line["tensor_ceiling"] = ceiling
        mhz = line["clocks"].get("sm_mhz")
        if "nvf4_pair_flop_per_clk_sm" in ceiling and mhz:
            # the FP4 MMA's own ceiling at the SM clock sampled during the timed steps
            c = ceiling["nvf4_pair_flop_per_clk_sm"] * ceiling["sms"] * mhz * 1e6 / 1e12
            line["roofline"]["mma_ceiling"] = {
                "tflops": round(c, 1), "frac": round(gemm_tflops / c, 4), "sm_mhz": mhz,
                "basis": "tc_ceiling: kind::mxf4nvf4 4X pair FLOP/clk/SM x SMs x median SM clock of the timed steps"}
    if e2e is not None:
        line["e2e"] = e2e
    if rank == 0 and not args.no_cpu_baseline:
        flops, dt = oracle_slice_step(d, CPU_SAMPLE_TOKENS, CPU_SAMPLE_FEATURES)
        line["cpu_baseline"] = {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": cores(),
                                "kind": "oracle",
                                "sample": f"oracle step on {CPU_SAMPLE_TOKENS} tokens x {CPU_SAMPLE_FEATURES} output "
                                          f"features at K=4096 (quantize 6 operands + 3 float64 GEMMs), {dt:.1f} s"}
    return line


# Each direction's copies split by rows over this many streams.  One stream per
# direction measured fastest on GB300 (3.79 ms per step; four: 4.42 ms).
E2E_COPY_STREAMS = 1
# Timed steps of the end-to-end loop (at least): the host link bounds it (about
# 170 GB/s each way at once on GB300), and the unoverlapped first H2D and last
# D2H add a whole step's copies to the total.
E2E_MIN_STEPS = 40


def run_e2e(step, d, args, world, device):
    """Same metric through the C ABI with host buffers: every step copies X, W
    and dY in from pinned host memory and Y, dX, dW back out, inside the timed
    region.  Pipelined as a serving or training loop would run it: two device
    buffer slots, so that the H2D of step i+1 and the D2H of step i-1 overlap
    step i's kernels, each direction's copies split by rows over
    E2E_COPY_STREAMS streams; events order every reuse of a slot."""
    hX, hW, hdY = (d[k].pin_memory() for k in ("X", "W", "dY"))
    hY = torch.empty(step.Y.shape, dtype=torch.bfloat16).pin_memory()
    hdX = torch.empty(step.dX.shape, dtype=torch.bfloat16).pin_memory()
    hdW = torch.empty(step.dW.shape, dtype=torch.bfloat16).pin_memory()
    host_in, host_out = {"X": hX, "W": hW, "dY": hdY}, {"Y": hY, "dX": hdX, "dW": hdW}
    names_in, names_out = tuple(host_in), tuple(host_out)
    slots = [{n: getattr(step, n) for n in names_in + names_out}]
    slots.append({n: torch.empty_like(getattr(step, n)) for n in names_in + names_out})
    compute = torch.cuda.current_stream()
    C = E2E_COPY_STREAMS
    h2d = [torch.cuda.Stream() for _ in range(C)]
    d2h = [torch.cuda.Stream() for _ in range(C)]
    in_ready = [[torch.cuda.Event() for _ in range(C)] for _ in range(2)]
    out_done = [[torch.cuda.Event() for _ in range(C)] for _ in range(2)]
    computed = [torch.cuda.Event(), torch.cuda.Event()]
    started = [False, False]

    def rows(t, c):
        r = t.shape[0]
        return slice(r * c // C, r * (c + 1) // C)

    def one(i):
        k = i % 2
        sl = slots[k]
        for c in range(C):
            with torch.cuda.stream(h2d[c]):
                if started[k]:
                    h2d[c].wait_event(computed[k])      # slot k's inputs are free again
                for n in names_in:
                    sl[n][rows(sl[n], c)].copy_(host_in[n][rows(sl[n], c)], non_blocking=True)
                in_ready[k][c].record(h2d[c])
            compute.wait_event(in_ready[k][c])
            if started[k]:
                compute.wait_event(out_done[k][c])      # slot k's outputs have been read back
        for n in names_in + names_out:
            setattr(step, n, sl[n])
        step.run()
        computed[k].record(compute)
        for c in range(C):
            with torch.cuda.stream(d2h[c]):
                d2h[c].wait_event(computed[k])
                for n in names_out:
                    host_out[n][rows(sl[n], c)].copy_(sl[n][rows(sl[n], c)], non_blocking=True)
                out_done[k][c].record(d2h[c])
        started[k] = True

    for i in range(max(2, args.warmup)):
        one(i)
    torch.cuda.synchronize()
    barrier(world)
    # the pipeline's fill (the first H2D) and drain (the last D2H) overlap
    # nothing; over at least E2E_MIN_STEPS steps they weigh little
    steps = max(args.steps, E2E_MIN_STEPS)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(compute)
    for st in h2d:
        st.wait_stream(compute)
    for i in range(steps):
        one(i)
    for st in d2h:
        compute.wait_stream(st)
    e.record(compute)
    torch.cuda.synchronize()
    for n in names_in + names_out:
        setattr(step, n, slots[0][n])
    ms = max_over_ranks(s.elapsed_time(e) / steps, world, device)
    h2d_b = sum(t.numel() * t.element_size() for t in (hX, hW, hdY))
    d2h_b = sum(t.numel() * t.element_size() for t in (hY, hdX, hdW))
    return {"value": round(world * STEP_FLOPS / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
            "ms_per_step": round(ms, 4), "steps": steps, "h2d_bytes_per_step": h2d_b, "d2h_bytes_per_step": d2h_b,
            "pipeline": f"2 buffer slots; H2D and D2H over {C} streams each, overlapping the kernels of the "
                        "neighbouring steps",
            "h2d_gbs": round(h2d_b / (ms * 1e-3) / 1e9, 1)}


def run_reference(args, rank, world):
    """The CPU oracle, timed as it stands, on a bounded slice of the step."""
    if rank != 0:
        return None
    d = make_inputs()
    for _ in range(args.warmup):
        oracle_slice_step(d, 512, 512)
    times = []
    flops = 0
    for _ in range(args.steps):
        flops, dt = oracle_slice_step(d, 512, 512)
        times.append(dt)
    sec = statistics.mean(times)
    v = round(flops / sec / 1e12, 6)
    return {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sec * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": WORKLOAD, "tokens": M_TOK, "hidden": K_HID, "ffn": N_FFN, "scale_fmt": "E4M3",
                   "group": 16, "parallelism": "cpu"},
        "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": cores(), "kind": "oracle",
                         "sample": "each step: oracle step on 512 tokens x 512 output features at K=4096 "
                                   "(quantize 6 operands + 3 float64 GEMMs)"},
        "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    global M_TOK, STEP_FLOPS
    args = parse()
    if args.tokens != M_TOK:
        if args.tokens % 256 or args.tokens <= 0:
            raise SystemExit("--tokens must be a positive multiple of 256")
        M_TOK = args.tokens
        STEP_FLOPS = 3 * 2 * M_TOK * N_FFN * K_HID
    rank, world, local = dist_env()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
        if line is not None:
            print(json.dumps(line), flush=True)
        return
    dist_init(world, "nccl")
    line = run_ours(args, rank, world, local)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
