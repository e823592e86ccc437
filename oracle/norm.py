"""RMSNorm fused with the per-token INT8 quant or the per-128-group FP8
quant: the producer of the quantized activation a linear consumes.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[DF] section 2.3 ("operator fusion: removing quant/dequant nodes"), first
fusion: the unfused RMSNorm wrote an FP32 output that a separate op then
quantized for the next linear; fused, the normalisation stays in registers
and only the quantized activation is written.  [W8A8] section 1 lets that
linear consume a ready (int8, per-token scale) tuple.

RMSNorm is y_k = x_k / sqrt(mean_k(x_k^2) + eps) * gamma_k.  The pages
print no arithmetic, so these readings are used:
  * the row statistic is exact: ss = sum_k x_k^2 summed without rounding and
    rounded once to float64 (math.fsum), then t = ss / K, u = t + eps,
    r = fp32(1 / sqrt(u)), each step one IEEE float64 rounding and a final
    rounding to fp32; u == 0 (an all-zero row with eps == 0) gives r = 0;
  * y_k = fp32(fp32(x_k * r) * gamma_k): the normalised row stays fp32 (the
    page's unfused RMSNorm wrote FP32) and is quantized directly;
  * x and gamma are bf16, eps an fp32 value;
  * INT8: the per-token rule of int8.quant_int8_rows on y;
    FP8: the per-128-group rule of fp8.quant_fp8_group_values on y with one
    outer group (G = 1, D = K) and packed UE8M0 scales [1, P, Ta].
"""
import math

import numpy as np

from .codecs import bf16_to_f32
from .fp8 import packed_dims, pack_exponents, quant_fp8_group_values
from .int8 import quant_int8_rows


def rms_scale(x_row_f32, eps):
    """r = fp32(1 / sqrt(fsum(x^2) / K + eps)) for one row (fp32 values)."""
    K = len(x_row_f32)
    ss = math.fsum(float(v) * float(v) for v in x_row_f32)   # exact sum, one rounding
    u = ss / K + float(np.float32(eps))
    if u == 0.0:
        return np.float32(0.0)
    return np.float32(1.0 / math.sqrt(u))


def rmsnorm_f32(x_bf16, gamma_bf16, eps):
    """y[M, K] fp32 = fp32(fp32(x * r_row) * gamma)."""
    x = bf16_to_f32(np.asarray(x_bf16, np.uint16))
    g = bf16_to_f32(np.asarray(gamma_bf16, np.uint16))
    if x.ndim != 2 or g.shape != (x.shape[1],):
        raise ValueError("x must be [M, K] and gamma [K]")
    y = np.empty_like(x)
    for m in range(x.shape[0]):
        r = rms_scale(x[m], eps)
        y[m] = ((x[m] * r).astype(np.float32) * g).astype(np.float32)
    return y


def rmsnorm_quant_int8(x_bf16, gamma_bf16, eps):
    """(q int8 [M, K], s fp32 [M]) of the RMSNorm output."""
    return quant_int8_rows(rmsnorm_f32(x_bf16, gamma_bf16, eps))


def rmsnorm_quant_fp8_ue8m0_packed(x_bf16, gamma_bf16, eps):
    """(E4M3 codes uint8 [T, K], packed UE8M0 storage int32 [1, P, Ta])."""
    y = rmsnorm_f32(x_bf16, gamma_bf16, eps).astype(np.float64)
    T, K = y.shape
    NG, _, _ = packed_dims(T, K)
    xq, e = quant_fp8_group_values(y.reshape(T, 1, K))
    return xq.reshape(T, K), pack_exponents(e, T, 1, NG)
