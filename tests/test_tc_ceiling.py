"""The tensor-core ceiling program (csrc/tc_ceiling.cu) on the GPU.

It streams tcgen05.mma instructions of the bf16 and the block-scaled FP4 forms
and reports FLOP per clock per SM.  Checked here: it runs to completion (every
commit landed), the bf16 form is within the tensor pipe's architectural rate of
8192 FLOP per clock per SM (a streaming loop cannot exceed it), and the FP4 forms
run faster than bf16 and no faster than the 6x the nominal dense figures imply.
"""

import json
import subprocess

import pytest

from fp4_block_scaled_amax_gb300 import build

pytestmark = pytest.mark.gpu


def test_ceiling_program_runs_and_orders_the_forms():
    exe = build.build_ceiling()
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    d = json.loads(r.stdout.strip().splitlines()[-1])
    assert d["ok"] is True
    bf16 = d["bf16_flop_per_clk_sm"]
    assert 4096 < bf16 <= 8192 * 1.02
    for key in ("nvf4_pair_flop_per_clk_sm", "mxf4_flop_per_clk_sm"):
        assert 2.0 * bf16 < d[key] <= 6.0 * 8192 * 1.02, key
