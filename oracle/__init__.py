"""CPU oracle for the FP4 block-scaled linear-layer hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library and
its Python binding) may import, call or link anything in this package; only the
test suite, the smoke check and the benchmark's CPU-baseline leg use it.  It
shares no code, table or constant generator with the CUDA path.

It is a plain, slow, step-by-step restatement of what the source pages describe:

* "NVFP4 vs MXFP" post (quant_prune_distill #486, section "Метод"): NVFP4 is
  E2M1 with a group of 16 and an E4M3 block scale (4.5 bits per parameter);
  MXFP4 uses a group of 32 and an E8M0 (power-of-two) scale (4.25 bits).
* Review of Intel's FP4 training paper (gonzo_ML #3986, sections
  "Форматы FP4" and "Стохастическая квантизация"): group 16, a sweep of scale
  formats E1M6..E8M0, nearest rounding for forward weights and activations,
  stochastic rounding (up or down with a probability set by the distance to the
  neighbour) for the backward pass.
* "UE5M3 FP4 Block Scaling for Stable Language Model Pretraining" (rit.work
  blog, sections "Что сделали" and "Ограничения"): an unsigned 8-bit block
  scale with 5 exponent and 3 fraction bits, one per 16 elements; the
  whole-tensor maximum refreshed once every 50 steps; stochastic rounding on
  backward gradients only; UE5M3 run through software emulation.
* Weight-only NVFP4 post (quant_prune_distill #574, section "Эксперименты"):
  NVFP4 weights, activations untouched, a memory-bound kernel.

Every floating-point step that the method performs in single precision is done
here as one numpy float32 operation (IEEE round-to-nearest-even, no fused
multiply-add); GEMM values are float64.  Where the pages leave a bit-level
detail open the oracle takes one fixed reading, named at the function.

Modules: ``formats`` (element and scale codecs), ``philox`` (counter-based
RNG), ``quantize`` (global/block scaling, rounding, packing, dequantization),
``gemm`` (float64 reference GEMM/GEMV and the tolerance bound), ``amax``
(stale global-amax state).
"""

from . import formats, philox, quantize, gemm, amax  # noqa: F401
