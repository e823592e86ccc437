"""Pins of the MXFP8-like (32-element block) oracle, CPU only."""
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs, fp8 as of8, mx
from fp8_dynamic_quant_gb300 import synth


def bf(vals):
    return codecs.f64_to_bf16(np.asarray(vals, np.float64))


def test_hand_blocks():
    # block 0: absmax 448 -> e = 0 (byte 127), 448 -> code 0x7E;
    # block 1: absmax 1 -> e = ceil(log2(1/448)) = -8 (byte 119), 1 * 2^8 = 256 -> code 0x78,
    #          -0.5 * 2^8 = -128 -> code 0xF0
    row = np.zeros(64)
    row[0], row[1] = 448.0, -3.0
    row[32], row[33] = 1.0, -0.5
    q, s = mx.quant_mxfp8(bf([row]))
    assert s.tolist() == [[127, 119]]
    assert q[0, 0] == 0x7E and q[0, 32] == 0x78 and q[0, 33] == 0xF0
    assert codecs.e4m3_decode(np.array([q[0, 1]]))[0] == -3.0
    assert (q[0, 2:32] == 0).all()


def test_agrees_with_128_groups_when_subblocks_share_the_exponent():
    # scale each 32-block so its absmax is exactly 300 * 2^k for the block's group:
    # all four sub-blocks of a 128-group then get the group's exponent
    r = synth.rng(3)
    x = r.uniform(-1, 1, (4, 512))
    for g in range(4):
        for b in range(4):
            blk = x[:, 128 * g + 32 * b:128 * g + 32 * b + 32]
            blk /= np.abs(blk).max(axis=1, keepdims=True)
            blk *= 300.0 * 2.0 ** (g - 2)
    xb = bf(x)
    q, s = mx.quant_mxfp8(xb)
    q128, e128 = of8.quant_fp8_group(xb.reshape(4, 1, 512))
    assert np.array_equal(q, q128.reshape(4, 512))
    assert np.array_equal(s.astype(np.int64) - 127, np.repeat(e128.reshape(4, 4), 4, axis=1))


def test_dequant_within_half_an_e4m3_step():
    x = synth.activations(5, 256, 4)
    q, s = mx.quant_mxfp8(x)
    xf = codecs.bf16_to_f32(x).astype(np.float64)
    deq = codecs.e4m3_decode(q).astype(np.float64) * np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
    step = np.repeat(np.ldexp(1.0, s.astype(np.int64) - 127), 32, axis=1)
    assert np.all(np.abs(deq - xf) <= np.maximum(np.abs(xf) * 2.0 ** -4, step * 2.0 ** -10))


def exact_linear(qx, sx, qw, sw):
    """Independent restatement: every product dequantized on its own, summed exactly."""
    ax = codecs.e4m3_decode(qx).astype(np.float64)
    aw = codecs.e4m3_decode(qw).astype(np.float64)
    M, K = ax.shape
    out = np.empty((M, aw.shape[0]), np.float64)
    for m in range(M):
        for n in range(aw.shape[0]):
            tot = Fraction(0)
            for k in range(K):
                if ax[m, k] and aw[n, k]:
                    tot += (Fraction(ax[m, k]) * Fraction(2) ** (int(sx[m, k // 32]) - 127) *
                            Fraction(aw[n, k]) * Fraction(2) ** (int(sw[n, k // 32]) - 127))
            out[m, n] = float(tot)
    return codecs.f64_to_bf16(out)


@pytest.mark.parametrize("M,N,K", [(1, 3, 32), (3, 5, 96), (2, 4, 256)])
def test_linear_matches_per_element_exact_sum(M, N, K):
    x = synth.activations(M, K, 10 + K)
    w = codecs.f64_to_bf16(synth.rng(11 + K).standard_normal((N, K)) * 0.05)
    qx, sx = mx.quant_mxfp8(x)
    qw, sw = mx.quant_mxfp8(w)
    assert np.array_equal(mx.mxfp8_linear(qx, sx, qw, sw), exact_linear(qx, sx, qw, sw))


def test_linear_integer_case_and_scale_doubling():
    r = synth.rng(12)
    xi = r.integers(-8, 9, (3, 64)).astype(np.float64)
    wi = r.integers(-8, 9, (4, 64)).astype(np.float64)
    qx, qw = codecs.e4m3_encode(xi), codecs.e4m3_encode(wi)
    sx = np.full((3, 2), 127, np.uint8)
    sw = np.full((4, 2), 127, np.uint8)
    y = mx.mxfp8_linear(qx, sx, qw, sw)
    assert np.array_equal(y, codecs.f64_to_bf16(xi @ wi.T))
    # +1 on every activation scale byte doubles Y exactly
    y2 = mx.mxfp8_linear(qx, sx + 1, qw, sw)
    assert np.array_equal(codecs.bf16_to_f32(y2), 2 * codecs.bf16_to_f32(y))


def test_blocked_scale_layout_by_hand():
    # R = 130 rows, K = 256: chunks [2, 2, 512]; row 33, K block 5 -> chunk (0, 1),
    # byte (33 % 32) * 16 + (33 // 32) * 4 + 5 % 4 = 16 + 4 + 1 = 21; row 129, block 2 ->
    # chunk (1, 0), byte 1 * 16 + 0 + 2 = 18
    sf = np.zeros((130, 8), np.uint8)
    sf[33, 5] = 200
    sf[129, 2] = 17
    b = mx.pack_sf_blocked(sf)
    assert b.shape == (2, 2, 512)
    assert b[0, 1, 21] == 200 and b[1, 0, 18] == 17
    assert int(b.astype(np.int64).sum()) == 217          # everything else zero, incl. rows 130..255
    assert np.array_equal(mx.unpack_sf_blocked(b, 130), sf)
