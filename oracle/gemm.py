"""W4A4 and W4A8 quantized linear layers with their epilogue.

Pages: a linear layer runs with 4-bit weights and NVFP4 or INT8 activations
("W4A6" mixed in "Table 2"; "Uniform W4A4" / "Uniform W4A8" in "Table 3" of
the thelatestinai.com page; the choice per layer from the mlsanity.com
"Abstract").  The pages print no GEMM; this is the plain definition:

  W4A4:  y[m,n] = g_a g_w  sum_k (E2M1(a)*S_a)[m,k] (E2M1(w)*S_w)[n,k]
  W4A8:  y[m,n] = s_a[m] g_w sum_k q[m,k] (E2M1(w)*S_w)[n,k]
  then   y += bias[n];  y = GELU_tanh(y) if asked;  y += residual[m,n]
and the result is stored as float32 or bf16 (round to nearest even).

Everything is float64 here (every product of decoded values is exact in
float64 and the sums are as good as float64 gets); the kernels accumulate
in float32, so parity is a tolerance, not bit equality.

Parity: pinned (pure-Python float64 triple loop on tiny shapes; unit scales
reduce to an exact integer matmul; GELU against torch's tanh GELU).
"""
from __future__ import annotations

import numpy as np

from . import nvfp4
from .codecs import bf16_to_f32, f64_to_bf16

SQRT_2_OVER_PI = np.sqrt(2.0 / np.pi)


def gelu_tanh(x):
    """0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))), float64."""
    x = np.asarray(x, dtype=np.float64)
    return 0.5 * x * (1.0 + np.tanh(SQRT_2_OVER_PI * (x + 0.044715 * x * x * x)))


def epilogue(acc, bias=None, gelu=False, residual=None, out_dtype="f32"):
    """acc float64 [M,N] already scaled; bias bf16 bits [N]; residual bf16 bits [M,N]."""
    y = np.asarray(acc, dtype=np.float64)
    if bias is not None:
        y = y + bf16_to_f32(bias).astype(np.float64)[None, :]
    if gelu:
        y = gelu_tanh(y)
    if residual is not None:
        y = y + bf16_to_f32(residual).astype(np.float64)
    if out_dtype == "f32":
        return y.astype(np.float32)
    if out_dtype == "bf16":
        return f64_to_bf16(y)
    raise ValueError(out_dtype)


def w4a4(a_codes, a_sf, g_a, w_codes, w_sf, g_w, bias=None, gelu=False, residual=None, out_dtype="f32",
         w_deq=None):
    """a_codes [M,K/2], a_sf [M,K/16] (plain layout), w likewise with N rows.
    w_deq (optional): nvfp4.dequantize(w_codes, w_sf) computed once by the
    caller, for repeated products with one weight."""
    A = nvfp4.dequantize(a_codes, a_sf)             # float64, without g
    W = nvfp4.dequantize(w_codes, w_sf) if w_deq is None else w_deq
    acc = (A @ W.T) * (float(g_a) * float(g_w))
    return epilogue(acc, bias, gelu, residual, out_dtype)


def w4a8(q, s_a, w_codes, w_sf, g_w, bias=None, gelu=False, residual=None, out_dtype="f32", w_deq=None):
    """q int8 [M,K], s_a float32 [M]; w codes/scales (and w_deq) as in w4a4."""
    A = np.asarray(q, dtype=np.float64)
    W = nvfp4.dequantize(w_codes, w_sf) if w_deq is None else w_deq
    acc = (A @ W.T) * (np.asarray(s_a, dtype=np.float64)[:, None] * float(g_w))
    return epilogue(acc, bias, gelu, residual, out_dtype)


def w4a4_rows(rows, a_codes, a_sf, g_a, w_codes, w_sf, g_w, **kw):
    """Same as w4a4 on a subset of rows (for sampled checks at full size)."""
    rows = np.asarray(rows)
    res = kw.pop("residual", None)
    return w4a4(a_codes[rows], a_sf[rows], g_a, w_codes, w_sf, g_w,
                residual=None if res is None else res[rows], **kw)


def w4a8_rows(rows, q, s_a, w_codes, w_sf, g_w, **kw):
    rows = np.asarray(rows)
    res = kw.pop("residual", None)
    return w4a8(q[rows], s_a[rows], w_codes, w_sf, g_w,
                residual=None if res is None else res[rows], **kw)
