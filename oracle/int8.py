"""INT8 per-token dynamic quant and the W8A8 linear, written from definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[W8A8] section 1 ("how to compare the quantization gain with the extra
cost") gives the chain  BF16 X -> npu_dynamic_quant -> INT8 X + per-token
scale -> npu_quant_matmul -> BF16 Y, and its "reuse already-quantized
activations" paragraph lets a linear take a ready (int8, scale) tuple.
The pages do not print the arithmetic, so these readings are used:
  * per-token scale s = absmax / 127 in fp32 (IEEE division);
  * q = clamp(round_half_even(x / s), -127, 127), x / s an fp32 division;
    a zero row gives s = 0 and q = 0 (0/0 is read as 0);
  * the GEMM accumulates exactly in integers (int32 range is checked);
  * dequant Y = bf16_RN((fp32(acc) * s[m]) * sw[n]), each product an fp32
    rounding, left to right.
"""
import numpy as np

from .codecs import bf16_to_f32, f32_to_bf16

INT8_QMAX = np.float32(127.0)


def dynamic_quant_int8(x_bf16):
    """Per-token (per-row) INT8 quant of X[M, K] (bf16 bits).

    Returns (q int8 [M, K], s float32 [M]).
    [W8A8] section 1 (npu_dynamic_quant: INT8 X + per-token scale) and
    section 2 (one row = the last dimension, one token per row).
    """
    return quant_int8_rows(bf16_to_f32(np.asarray(x_bf16, dtype=np.uint16)))


def quant_int8_rows(x):
    """The per-token INT8 rule on fp32 values x[M, K] (bf16 inputs widen
    exactly; the RMSNorm producer feeds its fp32 rows here)."""
    x = np.asarray(x, dtype=np.float32)
    if x.ndim != 2:
        raise ValueError("X must be [M, K]")
    M, K = x.shape
    if M == 0:
        return np.zeros((0, K), np.int8), np.zeros((0,), np.float32)
    amax = np.max(np.abs(x), axis=1)                     # exact
    s = (amax / INT8_QMAX).astype(np.float32)            # fp32 division
    with np.errstate(divide="ignore", invalid="ignore"):
        r = (x / s[:, None]).astype(np.float32)          # fp32 division per element
    r = np.where(np.isnan(r), np.float32(0), r)          # 0/0 of an all-zero row
    q = np.clip(np.rint(r), -127, 127)                   # rint: ties to even
    return q.astype(np.int8), s


def int_gemm_nt(q, w_nk):
    """acc[m, n] = sum_k q[m, k] * w_nk[n, k], exact.

    The products are integers of magnitude <= 127*127 and K is small enough
    that every partial sum is an integer below 2**53, so a float64 matrix
    product (a library primitive) returns the exact integer sum.
    """
    q = np.asarray(q)
    w = np.asarray(w_nk)
    K = q.shape[1]
    if K * 127 * 127 >= 2 ** 53:
        raise ValueError("K too large for an exact float64 integer sum")
    acc = q.astype(np.float64) @ w.astype(np.float64).T
    return acc.astype(np.int64)


def dequant_bf16(acc, s, sw):
    """Y = bf16_RN((fp32(acc) * s[m]) * sw[n]), fp32 rounding at each step."""
    acc = np.asarray(acc, dtype=np.int64)
    if acc.size and np.abs(acc).max() >= 2 ** 31:
        raise ValueError("accumulator leaves the int32 range")
    a32 = acc.astype(np.float32)                          # int -> fp32, nearest
    t = (a32 * np.asarray(s, np.float32)[:, None]).astype(np.float32)
    y = (t * np.asarray(sw, np.float32)[None, :]).astype(np.float32)
    return f32_to_bf16(y)


def w8a8_linear(q, s, w_nk, sw):
    """W8A8 linear on pre-quantized activations.

    q int8 [M, K], s fp32 [M], w_nk int8 [N, K] (logical W[k, n] = w_nk[n, k]),
    sw fp32 [N]  ->  Y bf16 bits [M, N].
    [W8A8] section 1 (npu_quant_matmul -> BF16 Y; a linear may consume the
    upstream (int8, scale) tuple directly).
    """
    acc = int_gemm_nt(q, w_nk)
    return dequant_bf16(acc, s, sw)


def w8a8_quant_linear(x_bf16, w_nk, sw):
    """BF16 X -> dynamic quant -> W8A8 linear.  Returns (Y, q, s).

    [W8A8] section 1: T_W8A8_linear = T_dynamic_quant + T_quant_matmul + ...;
    the fused call must give exactly what the two steps give.
    """
    q, s = dynamic_quant_int8(x_bf16)
    return w8a8_linear(q, s, w_nk, sw), q, s

