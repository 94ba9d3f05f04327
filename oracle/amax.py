"""Stale per-tensor global amax (oracle; test infrastructure only).

"UE5M3 FP4 Block Scaling ..." blog, section "Что сделали": the maximum of the
whole tensor is updated once every 50 steps and the stored value is used in
between.  Reading fixed here: the stored amax is refreshed to max|x_t| at every
step t with t % period == 0 (t = 0, 50, ...); other steps quantize with the
stored value.  Blocks whose amax exceeds the stored value get a larger scale
(E4M3 saturates at 448; UE5M3 has room up to 114688).
"""

from __future__ import annotations

import dataclasses

import numpy as np


@dataclasses.dataclass
class AmaxState:
    period: int = 50
    amax: float = 0.0
    last_refresh_step: int = -1

    def amax_for_step(self, step: int, x: np.ndarray) -> np.float32:
        """The global amax to quantize step `step`'s tensor x with."""
        if self.last_refresh_step < 0 or step % self.period == 0:
            self.amax = float(np.max(np.abs(np.asarray(x, dtype=np.float32))))
            self.last_refresh_step = step
        return np.float32(self.amax)
