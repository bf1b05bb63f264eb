"""CPU oracle for the 6Bit-Diffusion hot path.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only the tests, the smoke check and the bench's CPU-baseline / reference arm
may call it.  It shares no code with the CUDA library (no kernels, headers,
tables or helpers); the two meet only in the seeded inputs of `synthetic`.

Source: "6Bit-Diffusion: Inference-Time Mixed-Precision Quantization for Video
Diffusion Models" (arXiv 2603.18742), as described on three web pages:
  * mlsanity.com/paper/2603.18742, "Abstract" -- NVFP4 for temporally stable
    layers, INT8 for volatile ones, a lightweight linear predictor, Temporal
    Delta Cache (TDC) skipping invariant blocks;
  * thelatestinai.com/papers/2603.18742, Figure 1-4 captions -- relative L2
    quantization error per layer, Gamma = block relative L1 input/output
    distance at the preceding step, per-layer line E_rel = alpha*Gamma + beta,
    TDC on the updates Delta of the preceding two steps, measured by cosine
    similarity / relative L2 difference;
  * "Table 2" / "Table 3" of the same page -- W4A6 mixed, uniform W4A4 / W4A8.

The pages print no equations, formats or kernels.  Every step that they leave
open is a stated reading (module docstrings say which); the NVFP4 and E4M3
number formats follow the OCP 8-bit floating point and microscaling format
definitions.

Precision: decisions that produce integers (codes, scale bytes, Delta's bf16
bits, flags) are taken in float32 with round-to-nearest-even, the precision
the kernels use.  Sums, matrix products and norms are float64.

Parity status per function is listed in each module's header.
"""
from . import codecs, nvfp4, int8, gemm, gamma, dmpq, tdc, block, calib, mxcache  # noqa: F401
