"""MXFP8-like block-scaled FP8: 32 consecutive elements share one UE8M0
scale, payloads E4M3; and the linear that consumes it.  Written from
definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[DF] section 2.1 ("why block scaling"): the chosen format gives every 32
elements one shared 8-bit scale with E4M3 mantissas.  The page prints no
rounding rule, so the per-128-group reading of [PR] is carried over to
32-element blocks:
  * scale 2^e, e = clamp(ceil(log2(absmax / 448)), -127, 127), absmax == 0
    -> e = -127; the byte is u = e + 127;
  * payload E4M3_RN_satfinite(x * 2^-e) (an exact scaling).
Blocks run along the last (K) dimension of a row-major [R, K] tensor, K a
multiple of 32; scales are stored [R, K/32] as bytes.  The same rule makes
both operands of the linear (activations per token, weights per output row).

Scale storage read by the linear (the consumer's native layout, as [PR]
has the producer write its consumer's layout): for every 128 rows and every
128-element K block, one 512-byte chunk; byte
    (r % 32) * 16 + ((r % 128) // 32) * 4 + (k // 32) % 4
of chunk (r // 128, k // 128) holds row r's scale for K block k // 32.  Rows
past R in the last chunk row are zero bytes.

Linear: Y[m, n] = bf16_RN( sum_b 2^(ex[m,b] + ew[n,b]) * sum_{k in b} qx[m,k] qw[n,k] ),
the exact value rounded once (the GPU accumulates in fp32 inside the tensor
core and is held to 1e-2 relative + 1e-3 absolute).
"""
from fractions import Fraction
import math

import numpy as np

from .codecs import bf16_to_f32, e4m3_decode, e4m3_encode, f64_to_bf16
from .fp8 import ue8m0_exponent

BLOCK = 32


def quant_mx_values(x):
    """x float64 [R, K] holding exact (bf16 / fp32) values -> (codes uint8 [R, K], e int32 [R, K/32])."""
    x = np.asarray(x, np.float64)
    R, K = x.shape
    if K % BLOCK:
        raise ValueError("K must be a multiple of 32")
    xb = x.reshape(R, K // BLOCK, BLOCK)
    amax = np.max(np.abs(xb), axis=2) if R else np.zeros((0, K // BLOCK))
    e = np.vectorize(ue8m0_exponent, otypes=[np.int64])(amax) if amax.size else np.zeros(amax.shape, np.int64)
    codes = e4m3_encode(xb * np.ldexp(1.0, -e)[..., None]).reshape(R, K)
    return codes, e.astype(np.int32)


def quant_mxfp8(x_bf16):
    """bf16 bits [R, K] -> (E4M3 codes uint8 [R, K], UE8M0 bytes uint8 [R, K/32])."""
    codes, e = quant_mx_values(bf16_to_f32(np.asarray(x_bf16, np.uint16)).astype(np.float64))
    return codes, (e + 127).astype(np.uint8)


def mxfp8_linear(qx, sx, qw, sw):
    """qx [M, K] E4M3 codes, sx [M, K/32] UE8M0 bytes, qw [N, K], sw [N, K/32] -> bf16 bits [M, N].

    Block sums are exact integers times 2^-18 (E4M3 values are multiples of
    2^-9) and are added with their power-of-two scales in exact rational
    arithmetic, then rounded once."""
    ax = e4m3_decode(np.asarray(qx)).astype(np.float64)
    aw = e4m3_decode(np.asarray(qw)).astype(np.float64)
    M, K = ax.shape
    N = aw.shape[0]
    nb = K // BLOCK
    ex = np.asarray(sx, np.int64) - 127
    ew = np.asarray(sw, np.int64) - 127
    # per-block dot products: exact in float64 (32 products of 4-bit-mantissa values)
    blk = np.einsum("mbk,nbk->mnb", ax.reshape(M, nb, BLOCK), aw.reshape(N, nb, BLOCK))
    out = np.empty((M, N), np.float64)
    for m in range(M):
        for n in range(N):
            tot = Fraction(0)
            for b in range(nb):
                if blk[m, n, b] != 0.0:
                    tot += Fraction(blk[m, n, b]) * Fraction(2) ** int(ex[m, b] + ew[n, b])
            out[m, n] = float(tot)  # correctly rounded to float64; bf16 rounding below is from the exact value
            # a float64 result can round differently from the exact value only at a bf16 tie, which the
            # single rounding below resolves from the float64; exact ties are re-checked here:
            f = Fraction(out[m, n])
            if f != tot and _is_bf16_tie(out[m, n]):
                out[m, n] = math.nextafter(out[m, n], math.inf if tot > f else -math.inf)
    return f64_to_bf16(out)


def _is_bf16_tie(v):
    """True if float64 v sits exactly halfway between two bf16 values."""
    b = np.asarray([v], np.float64).view(np.uint64)[0]
    mant = int(b) & ((1 << 52) - 1)
    return (mant & ((1 << 45) - 1)) == (1 << 44)


def pack_sf_blocked(sf):
    """UE8M0 bytes [R, K/32] -> blocked storage uint8 [ceil(R/128), K/128, 512]."""
    sf = np.asarray(sf, np.uint8)
    R, NB = sf.shape
    if NB % 4:
        raise ValueError("K must be a multiple of 128")
    RB = (R + 127) // 128
    out = np.zeros((RB, NB // 4, 512), np.uint8)
    for r in range(R):
        for b in range(NB):
            out[r // 128, b // 4, (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4] = sf[r, b]
    return out


def unpack_sf_blocked(blocked, R):
    """Inverse of pack_sf_blocked."""
    blocked = np.asarray(blocked, np.uint8)
    RB, KB, _ = blocked.shape
    sf = np.zeros((R, KB * 4), np.uint8)
    for r in range(R):
        for b in range(KB * 4):
            sf[r, b] = blocked[r // 128, b // 4, (r % 32) * 16 + ((r % 128) // 32) * 4 + b % 4]
    return sf
