"""Pins for the FP8 group-quant / packed-scale / einsum oracle."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs, fp8
from fp8_dynamic_quant_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    return codecs.f32_to_bf16(np.asarray(x, np.float32))


def test_exponent_golden():
    d = json.load(open(os.path.join(GOLD, "ue8m0_layout.json")))
    for c in d["exponents"]:
        e = fp8.ue8m0_exponent(c["amax"])
        assert e == c["e"] and e + 127 == c["byte"], c


def test_exponent_exhaustive_against_definition():
    """Every positive finite bf16 amax: e is the smallest integer with amax <= 448 * 2**e (clamped)."""
    b = np.arange(1, 0x7F80, dtype=np.uint16)                       # positive finite
    a = codecs.bf16_to_f32(b).astype(np.float64)
    for amax in a[::3]:
        e = fp8.ue8m0_exponent(amax)
        # brute definition with exact rationals
        fa = Fraction(float(amax))
        k = -140
        while fa > 448 * Fraction(2) ** k:
            k += 1
        assert e == max(-127, min(127, k)), amax


def test_payload_golden():
    d = json.load(open(os.path.join(GOLD, "ue8m0_layout.json")))
    for c in d["payloads"]:
        x = np.zeros((1, 1, 128), np.float32)
        x[0, 0, 0] = c["x"]
        x[0, 0, 1] = c["amax"]
        xq, e = fp8.quant_fp8_group(bf(x))
        assert int(xq[0, 0, 0]) == c["code"], c


def test_layout_golden_bytes():
    d = json.load(open(os.path.join(GOLD, "ue8m0_layout.json")))["layout"]
    T, G, D = d["T"], d["G"], d["D"]
    x = np.zeros((T, G, D), np.float32)
    for g in range(G):
        for j in range(D // 128):
            x[0, g, j * 128 + 5] = 448.0 * 2.0 ** (j - 2 + 3 * g)
    _, st = fp8.quant_fp8_group_ue8m0_packed(bf(x))
    assert st.shape == (2, 2, 4) and st.dtype == np.int32
    assert st.astype("<i4").tobytes().hex() == d["storage_bytes_hex"]


@pytest.mark.parametrize("T", [0, 1, 3, 4, 17])
def test_storage_and_logical_view_shapes(T):
    G, D = 3, 384                                      # NG = 3, P = 1: byte 3 of each pack unused
    x = synth.group_activations(T, G, D, 100 + T)
    xq, st = fp8.quant_fp8_group_ue8m0_packed(x)
    Ta = (T + 3) // 4 * 4
    assert xq.shape == (T, G, D) and st.shape == (G, 1, Ta)
    by = st.view(np.uint8).reshape(G, 1, Ta, 4)
    assert np.all(by[..., 3] == 0)                     # tail byte of the last pack
    assert np.all(by[:, :, T:, :] == 0)                # token padding (reading: zeroed)
    v = fp8.logical_scale_view(st, T)
    assert v.shape == (T, G, 1)
    if T == 0:
        assert v.shape == (0, 3, 1)                    # the PR's empty-token case


def test_logical_view_strides():
    T, G, D = 5, 2, 1024
    st = np.arange(G * 2 * 8, dtype=np.int32).reshape(G, 2, 8)
    v = fp8.logical_scale_view(st, T)
    P, Ta = 2, 8
    assert v.shape == (T, G, P)
    assert tuple(s // 4 for s in v.strides) == (1, P * Ta, Ta)


def test_dequant_within_half_ulp():
    x = synth.group_activations(6, 2, 512, 8)
    xq, e = fp8.quant_fp8_group(x)
    xf = codecs.bf16_to_f32(x).astype(np.float64).reshape(6, 2, 4, 128)
    dq = codecs.e4m3_decode(xq).reshape(6, 2, 4, 128) * np.ldexp(1.0, e)[..., None]
    scale = np.ldexp(1.0, e)[..., None]
    # E4M3: relative half-ulp 2^-4 for normals; absolute 2^-10 * scale in the subnormal range
    bound = np.maximum(np.abs(xf) * 2.0 ** -4, 2.0 ** -10 * scale)
    assert np.all(np.abs(dq - xf) <= bound)
    # the scaled group maximum lies in (224, 448]; after E4M3 rounding in [224, 448]
    amax = np.max(np.abs(xf), axis=3)
    assert np.all((amax / np.ldexp(1.0, e) > 224) & (amax / np.ldexp(1.0, e) <= 448))
    top = np.max(np.abs(codecs.e4m3_decode(xq)).reshape(6, 2, 4, 128), axis=3)
    assert np.all((top >= 224) & (top <= 448))


def test_repack_matches_direct_packing():
    for T, G, D in [(1, 2, 640), (17, 8, 4096), (6, 3, 384)]:
        x = synth.group_activations(T, G, D, T + G)
        _, st = fp8.quant_fp8_group_ue8m0_packed(x)
        _, sf = fp8.quant_fp8_group_fp32_scales(x)
        assert np.array_equal(fp8.repack_fp32_scales_to_ue8m0(sf), st)
        assert np.array_equal(fp8.unpack_scales(st, T, D // 128), sf.astype(np.float64))


def test_weight_block_quant_properties():
    w = synth.fp8_einsum_weights(2, 256, 384, 4)
    wq, sw = fp8.quantize_weight_fp8_block(w)
    assert wq.shape == (2, 256, 384) and sw.shape == (2, 3, 2)
    deq = codecs.e4m3_decode(wq).reshape(2, 2, 128, 3, 128) * sw.transpose(0, 2, 1)[:, :, None, :, None]
    wf = w.astype(np.float64).reshape(2, 2, 128, 3, 128)
    rel = np.abs(deq - wf) / np.maximum(np.abs(wf), 1e-30)
    assert np.all((rel <= 2.0 ** -4 + 1e-6) | (np.abs(deq - wf) <= 2.0 ** -10 * sw.max()))
    # block amax maps to 448 (the fp32 quotient amax / (amax/448) may round to 448 exactly or a hair off)
    top = np.max(np.abs(codecs.e4m3_decode(wq)).reshape(2, 2, 128, 3, 128), axis=(2, 4))
    assert np.all(top == 448.0)


def test_einsum_integer_special_case_exact():
    """sx = 1 (byte 127), sw = 1, small-integer E4M3 values: Y is an exact integer sum."""
    r = np.random.default_rng(9)
    T, G, D, N = 3, 2, 256, 128
    xi = r.integers(-8, 9, (T, G, D))
    wi = r.integers(-8, 9, (G, N, D))
    xq = codecs.e4m3_encode(xi)
    wq = codecs.e4m3_encode(wi)
    sx = np.ones((T, G, 2))
    sw = np.ones((G, 2, 1), np.float32)
    y = codecs.bf16_to_f32(fp8.fp8_group_einsum(xq, sx, wq, sw))
    exact = np.einsum("tgd,gnd->tgn", xi, wi).astype(np.float64)
    assert np.array_equal(y.astype(np.float64), codecs.bf16_to_f32(codecs.f64_to_bf16(exact)).astype(np.float64))
    # with the range cut to |v| <= 2 every sum stays below 256 and is exact in bf16
    xs, ws = np.clip(xi, -2, 2), np.clip(wi, -2, 2)
    ys = codecs.bf16_to_f32(fp8.fp8_group_einsum(codecs.e4m3_encode(xs), sx, codecs.e4m3_encode(ws), sw))
    exs = np.einsum("tgd,gnd->tgn", xs, ws)
    assert np.all(np.abs(exs) < 256) and np.array_equal(ys, exs.astype(np.float32))


def test_einsum_brute_force_rational():
    T, G, D, N = 2, 1, 256, 128
    x = synth.group_activations(T, G, D, 31)
    xq, st = fp8.quant_fp8_group_ue8m0_packed(x)
    w = synth.fp8_einsum_weights(G, N, D, 32)
    wq, sw = fp8.quantize_weight_fp8_block(w)
    sx = fp8.unpack_scales(st, T, D // 128)
    y = fp8.fp8_group_einsum(xq, sx, wq, sw)
    xv = codecs.e4m3_decode(xq)
    wv = codecs.e4m3_decode(wq)
    for t in range(T):
        for n in range(0, N, 17):
            tot = Fraction(0)
            for kb in range(D // 128):
                blk = sum(Fraction(float(xv[t, 0, d])) * Fraction(float(wv[0, n, d]))
                          for d in range(kb * 128, kb * 128 + 128))
                tot += blk * Fraction(float(sx[t, 0, kb])) * Fraction(float(sw[0, kb, n // 128]))
            want = codecs.f64_to_bf16(np.array([float(tot)]))[0]
            # float(tot) is one rounding of the exact value; bf16 rounding of it
            # equals bf16 rounding of the exact value unless float(tot) sits on a tie
            assert int(y[t, 0, n]) == int(want)


def test_packed_and_fp32_scale_paths_identical():
    T, G, D, N = 4, 2, 512, 256
    x = synth.group_activations(T, G, D, 41)
    xq, st = fp8.quant_fp8_group_ue8m0_packed(x)
    _, sf = fp8.quant_fp8_group_fp32_scales(x)
    wq, sw = fp8.quantize_weight_fp8_block(synth.fp8_einsum_weights(G, N, D, 42))
    y1 = fp8.fp8_group_einsum(xq, fp8.unpack_scales(st, T, D // 128), wq, sw)
    y2 = fp8.fp8_group_einsum(xq, sf, wq, sw)
    assert np.array_equal(y1, y2)
