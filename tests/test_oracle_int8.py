"""Pins for the INT8 oracle: hand-derived rows, brute force, closed forms."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import codecs, int8
from fp8_dynamic_quant_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def bf(x):
    return codecs.f32_to_bf16(np.asarray(x, np.float32))


def test_quant_golden_rows():
    d = json.load(open(os.path.join(GOLD, "int8_rows.json")))
    for c in d["cases"]:
        x = bf([c["x"]])
        q, s = int8.dynamic_quant_int8(x)
        assert float(s[0]) == c["s"], c
        assert q[0].tolist() == c["q"], c


def test_quant_empty_and_single_row():
    q, s = int8.dynamic_quant_int8(np.zeros((0, 64), np.uint16))
    assert q.shape == (0, 64) and s.shape == (0,)
    q, s = int8.dynamic_quant_int8(synth.activations(1, 4096, 7))
    assert q.shape == (1, 4096) and s.shape == (1,)


def test_quant_invariants_and_brute_force_rounding():
    x = synth.activations(9, 1024, 11)
    q, s = int8.dynamic_quant_int8(x)
    xf = codecs.bf16_to_f32(x)
    assert np.abs(q.astype(int)).max() <= 127
    for m in range(x.shape[0]):
        amax = np.abs(xf[m]).max()
        assert s[m] == np.float32(amax) / np.float32(127)
        k = int(np.argmax(np.abs(xf[m])))
        assert abs(int(q[m, k])) == 127 and np.sign(q[m, k]) == np.sign(xf[m, k])
        for k in range(0, x.shape[1], 7):
            # exact check: q is the integer nearest the fp32 quotient, ties to even
            r = Fraction(float(np.float32(xf[m, k]) / np.float32(s[m])))
            lo = r.numerator // r.denominator
            frac = r - lo
            if frac > Fraction(1, 2) or (frac == Fraction(1, 2) and lo % 2 == 1):
                want = lo + 1
            else:
                want = lo
            want = max(-127, min(127, want))
            assert int(q[m, k]) == want


def _brute_acc(q, w):
    M, K = q.shape
    N = w.shape[0]
    return [[sum(int(q[m, k]) * int(w[n, k]) for k in range(K)) for n in range(N)] for m in range(M)]


@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (3, 64, 48), (4, 16, 48), (7, 64, 16), (8, 16, 16), (9, 64, 48)])
def test_int_gemm_brute_force(M, K, N):
    r = np.random.default_rng(M * 100 + K + N)
    q = r.integers(-127, 128, (M, K), dtype=np.int8)
    w = r.integers(-127, 128, (N, K), dtype=np.int8)
    assert int8.int_gemm_nt(q, w).tolist() == _brute_acc(q, w)


@pytest.mark.parametrize("M,K,N", [(1, 16, 16), (4, 64, 48), (9, 64, 48)])
def test_linear_close_to_real_dequant(M, K, N):
    """Y is the real value sum_k (q*s)*(w*sw) rounded: within one bf16 ulp (+ fp32 slack)."""
    c = synth.int8_linear_case(M, K, N, 5)
    q, s = int8.dynamic_quant_int8(c["x"])
    y = codecs.bf16_to_f32(int8.w8a8_linear(q, s, c["w_nk"], c["sw"])).astype(np.float64)
    exact = (q.astype(np.float64) * s[:, None].astype(np.float64)) @ \
            (c["w_nk"].astype(np.float64) * c["sw"][:, None].astype(np.float64)).T
    assert np.all(np.abs(y - exact) <= np.abs(exact) * 2.0 ** -8 * 1.01 + 1e-30)


def test_linear_identity_weight():
    x = synth.activations(3, 64, 9)
    q, s = int8.dynamic_quant_int8(x)
    w = np.eye(64, dtype=np.int8)
    sw = np.full(64, 0.5, np.float32)
    y = int8.w8a8_linear(q, s, w, sw)
    want = codecs.f32_to_bf16((q.astype(np.float32) * s[:, None]).astype(np.float32) * np.float32(0.5))
    assert np.array_equal(y, want)
    y2 = int8.w8a8_linear(q, s, -w, sw)
    assert np.array_equal(codecs.bf16_to_f32(y2), -codecs.bf16_to_f32(want))


def test_accumulator_extreme_closed_form():
    K = 4096
    q = np.full((1, K), 127, np.int8)
    w = np.full((2, K), 127, np.int8)
    w[1] = -127
    acc = int8.int_gemm_nt(q, w)
    assert acc.tolist() == [[66064384, -66064384]]          # 127*127*4096
    s = np.array([0.25], np.float32)
    sw = np.array([2.0 ** -20, 2.0 ** -20], np.float32)
    y = codecs.bf16_to_f32(int8.w8a8_linear(q, s, w, sw))
    # 66064384 = 16129 * 2^12 exactly in fp32; * 2^-2 * 2^-20 = 16129 * 2^-10 = 15.7509765625
    # -> bf16 (step 2^-4 in [8, 16)) 252.015625/16 -> 252/16 = 15.75
    assert y.tolist() == [[15.75, -15.75]]


def test_fused_equals_two_steps():
    c = synth.int8_linear_case(4, 256, 64, 3)
    y, q, s = int8.w8a8_quant_linear(c["x"], c["w_nk"], c["sw"])
    q2, s2 = int8.dynamic_quant_int8(c["x"])
    assert np.array_equal(q, q2) and np.array_equal(s, s2)
    assert np.array_equal(y, int8.w8a8_linear(q2, s2, c["w_nk"], c["sw"]))
