"""Number formats used on the path, written from their definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

* bf16: the upper 16 bits of an IEEE binary32; conversion from binary32
  rounds to nearest, ties to even.
* E4M3 (OCP FP8, the ``float8_e4m3fn`` flavour): 1 sign bit, 4 exponent
  bits with bias 7, 3 mantissa bits; no infinities; S.1111.111 is NaN; the
  largest finite magnitude is 448; subnormals step by 2**-9.  Encoding here
  is round-to-nearest-even with saturation to +-448 ("satfinite").
* UE8M0: an unsigned byte u standing for the power of two 2**(u-127).

The E4M3 encoder is a nearest-value search over the decoded code table, so
it follows the definition rather than any bit trick.
"""
import numpy as np

# ---------------------------------------------------------------- bf16

def bf16_to_f32(bits):
    """bf16 bit patterns (uint16) -> float32, exactly (shift into the top half)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16(x):
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    Keeping the upper 16 bits of the binary32 pattern; the dropped half is
    compared with one half-unit (0x8000) and ties go to an even upper half.
    NaN does not occur on this path and is rejected.
    """
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    if np.isnan(f).any():
        raise ValueError("NaN is outside the path's contract")
    u = f.view(np.uint32).astype(np.uint64)
    upper = u >> np.uint64(16)
    lower = u & np.uint64(0xFFFF)
    round_up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & np.uint64(1)) == 1))
    return (upper + round_up.astype(np.uint64)).astype(np.uint16)


def f64_to_bf16(x):
    """float64 -> bf16 bit patterns with ONE rounding (nearest, ties to even).

    A value v = m * 2**ex (frexp, 0.5 <= |m| < 1) has its leading bit at
    2**(ex-1); bf16 keeps 8 significant bits, so the quantum is 2**(ex-8),
    floored at the smallest bf16 subnormal 2**-133.  v / quantum is exact in
    float64 and np.rint rounds it half-to-even, giving a value that is exactly
    representable in bf16 (the path never overflows bf16).
    """
    v = np.asarray(x, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN is outside the path's contract")
    _, ex = np.frexp(v)
    qexp = np.maximum(ex.astype(np.int64) - 8, -133)
    quantum = np.ldexp(1.0, qexp)
    r = np.rint(v / quantum) * quantum
    r32 = r.astype(np.float32)  # exact: r has <= 8 significant bits, in range
    if not np.array_equal(r32.astype(np.float64), r):
        raise ValueError("value outside the bf16 range")
    out = (np.ascontiguousarray(r32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)
    # keep the sign of values that round to zero
    neg0 = (r == 0) & np.signbit(v)
    return np.where(neg0, np.uint16(0x8000), out).astype(np.uint16)

# ---------------------------------------------------------------- E4M3

def e4m3_decode(codes):
    """E4M3 codes (uint8) -> float64 values; NaN codes (0x7F, 0xFF) -> NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.ldexp(1.0, e - 7)
    sub = (m / 8.0) * np.ldexp(1.0, -6)
    v = np.where(e == 0, sub, normal) * sign
    return np.where((c & 0x7F) == 0x7F, np.nan, v)


# magnitudes of the non-negative finite codes 0x00..0x7E, ascending in code order
_E4M3_POS = e4m3_decode(np.arange(0x7F, dtype=np.uint8))
E4M3_MAX = 448.0


def e4m3_encode(x):
    """Real values -> E4M3 codes, round to nearest (ties to even code), satfinite.

    Magnitudes at or above 448 become 448 (code 0x7E); otherwise the nearest
    entry of the decoded table is taken, and on an exact tie the entry with an
    even code (mantissa LSB 0).  The sign bit is copied from the input, so a
    negative value that rounds to zero gives 0x80.
    """
    v = np.asarray(x, dtype=np.float64)
    if np.isnan(v).any():
        raise ValueError("NaN is outside the path's contract")
    a = np.minimum(np.abs(v), E4M3_MAX)
    hi = np.searchsorted(_E4M3_POS, a, side="left")          # first table entry >= a
    hi = np.minimum(hi, 0x7E)
    lo = np.maximum(hi - 1, 0)
    d_hi = _E4M3_POS[hi] - a
    d_lo = a - _E4M3_POS[lo]
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    code = np.where(pick_lo, lo, hi).astype(np.uint8)
    return np.where(np.signbit(v), code | np.uint8(0x80), code).astype(np.uint8)

# ---------------------------------------------------------------- UE8M0

def ue8m0_decode(u):
    """UE8M0 bytes -> float64 powers of two 2**(u-127) (u=255 is NaN, never produced)."""
    b = np.asarray(u, dtype=np.uint8).astype(np.int64)
    return np.ldexp(1.0, b - 127)
