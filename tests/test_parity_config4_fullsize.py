"""Config 4 at full size: the UE5M3 stack step as bench.py runs it (through the C ABI).

"UE5M3 FP4 Block Scaling ..." blog, section "Что сделали": UE5M3 scales per
16 elements, the tensor maximum refreshed once every 50 steps and the stored
value used in between, stochastic rounding on the backward gradients, every
linear in FP4.  The Nemotron-H-8B-like stack at its stated size: 32768 tokens,
4096 -> 21504 -> 4096, six GEMMs of 5.77 TFLOP per step.

bench.StackStep runs step 0 (a refresh: fresh amaxes) and then step 49 (the
amaxes stored at step 0, by then 1.02^49 = 2.6x below the inputs).  After
each step, against the oracle:
  * stored amaxes (step 0) and max|x| by-products (step 49): exact;
  * every quantized operand (rows and transposed layout of X, W1, H, W2, dY,
    dH): sampled rows and columns, codes and UE5M3 scales bit-exact;
  * the UE5M3 shift by-product of every operand equals the oracle's t, and the
    E4M3 re-encodes of the sampled rows equal the oracle's (all exact: the
    device status stays 0);
  * the six GEMMs on 8 sampled 128 x 128 output tiles each, within
    1e-5 * sum|a||b| + 1e-6 plus one bf16 rounding (bf16 outputs).
H and dH are the GPU's bf16 GEMM outputs; the oracle reads the same bytes.
"""

import numpy as np
import pytest
import torch

from oracle import gemm as Gm
from oracle import quantize as Q
from gpu_util import from_mma, lib

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

FMT = "UE5M3"


def _pick(n, k, seed):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([[0, n - 1], rng.integers(0, n, k)]))


def _blocks(n, k, seed):
    """k distinct 128-aligned starts in [0, n), the last block among them."""
    rng = np.random.default_rng(seed)
    starts = rng.choice(n // 128 - 1, size=k - 1, replace=False) * 128
    return sorted([int(v) for v in starts] + [n - 128])


class Sources:
    """Host copies (bf16 torch) of the step's tensors, sliced to float32 on demand."""

    def __init__(self, s, X, dY):
        self.t = {"X": X.cpu(), "W1": s.W1.cpu(), "H": s.H.cpu(), "W2": s.W2.cpu(), "dY": dY.cpu(),
                  "dH": s.dH.cpu()}

    def rows(self, name, r0, r1):
        return self.t[name][r0:r1].float().numpy()

    def cols(self, name, c0, c1):
        # columns c0..c1 of the tensor as rows of its transpose
        return self.t[name][:, c0:c1].float().numpy().T.copy()

    def amax(self, name):
        return np.float32(self.t[name].abs().max().float().item())


def _oracle_rows(src, name, col, start, count, seed, rounding, g):
    x = src.cols(name, start, start + count) if col else src.rows(name, start, start + count)
    return Q.quantize_rows(x, FMT, rounding, seed, g, row0=start)


def _check_step(s, src, t, g_used):
    """g_used: the global amax each tensor was quantized with (numpy float32)."""
    seed = 1234 + 8 * t
    rnd = {"X": ("rne", 0, "rne", 0), "W1": ("rne", 0, "rne", 0), "H": ("rne", 0, "rne", 0),
           "W2": ("rne", 0, "rne", 0), "dY": ("sr", seed, "sr", seed + 1), "dH": ("sr", seed + 2, "sr", seed + 3)}
    for name, (rr, sr_, rc, sc_) in rnd.items():
        q = {k: v.cpu().numpy() for k, v in s.q[name].items()}
        R, C = src.t[name].shape
        g = g_used[name]
        # the shift by-product: the largest scale code belongs to the block holding max|x|
        code_max, _ = Q.block_scales(np.array([[src.amax(name)]], dtype=np.float32),
                                     Q.global_encode_scale(g, FMT), FMT)
        t_ref = Q.ue5m3_shift(code_max)
        assert q["t"].tolist() == [t_ref, t_ref], (t, name)
        srow = from_mma(q["sr"], R, C // 16)
        erow = from_mma(q["er"], R, C // 16)
        for r in _pick(R, 4, 10 + t):
            codes, scales = Q.quantize_rows(src.rows(name, r, r + 1), FMT, rr, sr_, g, row0=int(r))
            assert np.array_equal(q["cr"][r], codes[0]) and np.array_equal(srow[r], scales[0]), (t, name, "row", r)
            e4, exact = Q.ue5m3_reencode_e4m3(scales[0], t_ref)
            assert exact and np.array_equal(erow[r], e4), (t, name, "re-encode", r)
        scol = from_mma(q["sc"], C, R // 16)
        for c in _pick(C, 4, 20 + t):
            codes, scales = Q.quantize_rows(src.cols(name, c, c + 1), FMT, rc, sc_, g, row0=int(c))
            assert np.array_equal(q["cc"][c], codes[0]) and np.array_equal(scol[c], scales[0]), (t, name, "col", c)

    M, Hd, F = s.M, s.Hd, s.F
    # (what, A tensor, A transposed?, B tensor, B transposed?, output, out rows, out cols)
    gemms = [("L1 fwd", "X", False, "W1", False, s.H, M, F), ("L2 fwd", "H", False, "W2", False, s.Y, M, Hd),
             ("L2 dgrad", "dY", False, "W2", True, s.dH, M, F), ("L2 wgrad", "dY", True, "H", True, s.dW2, Hd, F),
             ("L1 dgrad", "dH", False, "W1", True, s.dX, M, Hd), ("L1 wgrad", "dH", True, "X", True, s.dW1, F, Hd)]
    for gi, (what, a, a_col, b, b_col, out, Mo, No) in enumerate(gemms):
        ra, sa_, ca, sca = rnd[a]
        rb, sb_, cb, scb = rnd[b]
        a_round, a_seed = (ca, sca) if a_col else (ra, sa_)
        b_round, b_seed = (cb, scb) if b_col else (rb, sb_)
        mb = _blocks(Mo, 4, 100 * t + gi)
        nb = _blocks(No, 4, 100 * t + gi + 50)
        qa = {m: _oracle_rows(src, a, a_col, m, 128, a_seed, a_round, g_used[a]) for m in mb}
        qb = {n: _oracle_rows(src, b, b_col, n, 128, b_seed, b_round, g_used[b]) for n in nb}
        got_all = out.cpu()
        for k in range(8):  # tiles (m_i, n_i) and (m_i, n_{i+1}): 8 tiles from 4 + 4 row blocks
            m0, n0 = mb[k % 4], nb[(k % 4 + k // 4) % 4]
            (ac, as_), (bc, bs) = qa[m0], qb[n0]
            Cr, S = Gm.gemm_ref(ac, as_, g_used[a], bc, bs, g_used[b], FMT)
            got = got_all[m0:m0 + 128, n0:n0 + 128].float().numpy()
            bound = Gm.gemm_bound(S) + np.abs(Cr) * 2.0 ** -8
            err = np.abs(got - Cr)
            assert (err <= bound).all(), f"step {t} {what} tile ({m0}, {n0}): worst {np.max(err / bound):.3g}"


def test_stack_full_size_refresh_and_stale():
    lib()
    import bench
    from fp4_block_scaled_amax_gb300 import synth
    dev = torch.device("cuda", 0)
    s = bench.StackStep(dev)
    stored = {}
    for t in (0, 49):
        d = synth.config4_step_device(t, dev)
        s.run(t, d["X"], d["dY"])
        torch.cuda.synchronize()
        assert int(s.status.item()) == 0, f"device status {int(s.status.item())} at step {t}"
        src = Sources(s, d["X"], d["dY"])
        amax_now = {n: src.amax(n) for n in bench.C4_NAMES}
        st = s.stored.cpu().numpy()
        if t == 0:
            for j, n in enumerate(bench.C4_NAMES):
                assert st[j] == amax_now[n], n  # fresh amaxes stored at the refresh
                stored[n] = np.float32(st[j])
        else:
            cur = s.current.cpu().numpy()
            for j, n in enumerate(bench.C4_NAMES):
                assert st[j] == stored[n], n   # nothing refreshed between refreshes
                assert cur[j] == amax_now[n], n  # the by-product: this step's max |x|
            assert amax_now["X"] > 2 * stored["X"]  # the drift has outgrown the stored amax
        _check_step(s, src, t, stored)
        del src
