"""Pins for oracle.codecs against the format definitions and library routines."""
import json
import os
from fractions import Fraction

import numpy as np
import torch

from oracle import codecs

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def all_finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = codecs.bf16_to_f32(b)
    return b[np.isfinite(f)], f[np.isfinite(f)]


def test_bf16_roundtrip_all_patterns():
    b, f = all_finite_bf16()
    assert np.array_equal(codecs.f32_to_bf16(f), b)


def test_f32_to_bf16_matches_torch():
    r = np.random.default_rng(1)
    x = np.concatenate([
        r.standard_normal(200000).astype(np.float32) * np.float32(1e3),
        # exact ties: upper half + 0x8000 in the dropped half
        ((r.integers(0, 2 ** 15, 5000).astype(np.uint32) << 16) | 0x8000).view(np.float32),
        np.array([0.0, -0.0, 1e-40, -1e-40, 3.3e38], np.float32),
    ])
    x = x[np.isfinite(x)]
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(codecs.f32_to_bf16(x), ref)


def _nearest_bf16_exact(v):
    """Brute force: nearest finite bf16 to the rational v, ties to even pattern."""
    fv = Fraction(v)
    f = np.float32(v)
    c = int(codecs.f32_to_bf16(np.array([f]))[0])
    best = None
    for cand in range(max(0, (c & 0x7FFF) - 2), min(0x7F7F, (c & 0x7FFF) + 2) + 1):
        pat = cand | (c & 0x8000)
        val = Fraction(float(codecs.bf16_to_f32(np.array([pat], np.uint16))[0]))
        d = abs(val - fv)
        key = (d, pat & 1)
        if best is None or key < best[0]:
            best = (key, pat)
    return best[1]


def test_f64_to_bf16_single_rounding_brute_force():
    r = np.random.default_rng(2)
    v = np.concatenate([r.standard_normal(3000) * 10.0 ** r.uniform(-30, 30, 3000),
                        np.array([1.0 + 2 ** -8, 1.0 + 2 ** -8 + 2 ** -40, -(1.0 + 3 * 2 ** -8)])])
    got = codecs.f64_to_bf16(v)
    for i in range(v.size):
        assert int(got[i]) == _nearest_bf16_exact(float(v[i])), v[i]


def test_f64_to_bf16_avoids_double_rounding():
    # 1 + 2^-8 + 2^-40 lies just above the bf16 midpoint between 1 and 1 + 2^-7.
    # Rounding to fp32 first would land exactly on the midpoint and then tie to
    # even (1.0); the single rounding must give 1 + 2^-7 (0x3F81).
    # 1 + 2^-8 - 2^-40 lies just below it and must give 1.0 (0x3F80).
    v = np.array([1.0 + 2.0 ** -8 + 2.0 ** -40, 1.0 + 2.0 ** -8 - 2.0 ** -40])
    assert np.float32(v[0]) == np.float32(1.0 + 2.0 ** -8)
    got = codecs.f64_to_bf16(v)
    assert got[0] == 0x3F81 and got[1] == 0x3F80


def test_e4m3_decode_matches_torch_all_codes():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = codecs.e4m3_decode(codes)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(ref[~nan], got[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x08] == 2.0 ** -6


def test_e4m3_encode_golden():
    d = json.load(open(os.path.join(GOLD, "e4m3_values.json")))
    for c in d["cases"]:
        assert int(codecs.e4m3_encode(np.array([c["x"]]))[0]) == c["code"], c


def test_e4m3_encode_matches_torch_in_range():
    # torch's float -> float8_e4m3fn cast is round-to-nearest-even; it does not
    # saturate, so compare inside [-448, 448] only, on every finite bf16 value
    # there plus random fp32 values.
    b, f = all_finite_bf16()
    r = np.random.default_rng(3)
    f = np.concatenate([f, (r.standard_normal(500000) * 10.0 ** r.uniform(-4, 2.6, 500000)).astype(np.float32)])
    f = f[np.abs(f) <= 448]
    ref = torch.from_numpy(f).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codecs.e4m3_encode(f), ref)


def test_e4m3_satfinite():
    x = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e30, -1e30])
    assert list(codecs.e4m3_encode(x)) == [0x7E] * 5 + [0x7E, 0xFE]


def test_ue8m0_decode():
    assert codecs.ue8m0_decode(np.array([127]))[0] == 1.0
    assert codecs.ue8m0_decode(np.array([0]))[0] == 2.0 ** -127
    assert codecs.ue8m0_decode(np.array([254]))[0] == 2.0 ** 127
