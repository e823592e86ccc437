"""Pins of the RMSNorm + quant oracle (CPU only).

Each case fixes one step against a closed form, an invariance or an
already-pinned oracle: the 1/K mean, the eps term, the sqrt and reciprocal,
the order of the two fp32 products, the zero-row rule, and the hand-off to
the INT8 per-token and FP8 per-group rules.
"""
import numpy as np
import pytest

from oracle import codecs, int8 as oi8, fp8 as of8, norm
from fp8_dynamic_quant_gb300 import synth


def bf(vals):
    return codecs.f64_to_bf16(np.asarray(vals, np.float64))


def test_hand_row_int8():
    # x = [1,-1,1,-1]: mean(x^2) = 1, r = 1; y = gamma; s = 127/127 = 1 exactly,
    # so q = rint(y): 127, -63.5 -> -64 and -0.5 -> 0 (ties to even), -2.5 -> -2
    q, s = norm.rmsnorm_quant_int8(bf([[1, -1, 1, -1]]), bf([127, 63.5, -2.5, 0.5]), 0.0)
    assert s.tolist() == [1.0]
    assert q.tolist() == [[127, -64, -2, 0]]


def test_mean_divides_by_k_and_eps_adds():
    # [2, 0, 0, 0]: ss = 4, t = 4 / 4 = 1 -> r = 1 (a 1/(K-1) or nonzero-count mean would not give 1)
    y = norm.rmsnorm_f32(bf([[2, 0, 0, 0]]), bf([1, 1, 1, 1]), 0.0)
    assert y.tolist() == [[2.0, 0.0, 0.0, 0.0]]
    # [3, 4], eps = 3.5: ss = 25, t = 12.5, u = 16, r = 1/4 exactly
    y = norm.rmsnorm_f32(bf([[3, 4]]), bf([1, -2]), 3.5)
    assert y.tolist() == [[0.75, -2.0]]


def test_product_order_x_times_r_then_gamma():
    # x = 3: r = fp32(1/3); fp32(3 * r) = 1 exactly, then * 5 = 5.  The other
    # order, 3 * fp32(r * 5), gives 4.9999998807907104.
    y = norm.rmsnorm_f32(bf([[3, 3, 3, 3]]), bf([5, 5, 5, 5]), 0.0)
    assert y.tolist() == [[5.0, 5.0, 5.0, 5.0]]
    r = norm.rms_scale(np.full(4, 3.0, np.float32), 0.0)
    assert r == np.float32(1.0) / np.float32(3.0)


def test_power_of_two_scale_invariance():
    x = synth.activations(3, 256, 5)
    xf = codecs.bf16_to_f32(x).astype(np.float64)
    g = synth.activations(1, 256, 6)[0]
    y0 = norm.rmsnorm_f32(x, g, 0.0)
    for k in (-20, -3, 5, 40):
        yk = norm.rmsnorm_f32(codecs.f64_to_bf16(xf * 2.0 ** k), g, 0.0)
        assert np.array_equal(yk.view(np.uint32), y0.view(np.uint32)), k


def test_zero_rows():
    q, s = norm.rmsnorm_quant_int8(bf([[0, 0, 0, 0]]), bf([1, 2, 3, 4]), 0.0)   # u = 0 -> r = 0
    assert s.tolist() == [0.0] and q.tolist() == [[0, 0, 0, 0]]
    q, s = norm.rmsnorm_quant_int8(bf([[0, 0, 0, 0]]), bf([1, 2, 3, 4]), 1e-6)
    assert s.tolist() == [0.0] and q.tolist() == [[0, 0, 0, 0]]


def test_unit_rows_reduce_to_the_plain_quant_rules():
    # a constant row c = 3 normalises to exactly 1 (see the product-order pin),
    # so the output is gamma itself: the INT8 and FP8 results must equal the
    # pinned per-token and per-group rules applied to gamma
    K = 384
    g = synth.activations(1, K, 7)
    x = bf(np.full((2, K), 3.0))
    q, s = norm.rmsnorm_quant_int8(x, g[0], 0.0)
    q0, s0 = oi8.dynamic_quant_int8(np.repeat(g, 2, axis=0))
    assert np.array_equal(q, q0) and np.array_equal(s, s0)
    xq, st = norm.rmsnorm_quant_fp8_ue8m0_packed(x, g[0], 0.0)
    xq0, st0 = of8.quant_fp8_group_ue8m0_packed(np.repeat(g, 2, axis=0).reshape(2, 1, K))
    assert np.array_equal(xq, xq0.reshape(2, K)) and np.array_equal(st, st0)


def test_statistic_matches_a_float64_library_sum():
    # for data whose squares sum exactly in float64 the exact-sum reading and
    # numpy's own sum agree; r is then 1/sqrt in float64 rounded to fp32
    x = synth.activations(4, 512, 8)
    xf = codecs.bf16_to_f32(x).astype(np.float64)
    for m in range(4):
        want = np.float32(1.0 / np.sqrt(np.sum(xf[m] ** 2) / 512 + np.float64(np.float32(1e-6))))
        assert norm.rms_scale(xf[m].astype(np.float32), 1e-6) == want


@pytest.mark.parametrize("T,K", [(1, 128), (3, 384), (5, 4096)])
def test_fp8_layout_and_bounds(T, K):
    x = synth.activations(T, K, 9 + T)
    g = synth.activations(1, K, 10)[0]
    xq, st = norm.rmsnorm_quant_fp8_ue8m0_packed(x, g, 1e-6)
    NG, P, Ta = of8.packed_dims(T, K)
    assert xq.shape == (T, K) and st.shape == (1, P, Ta)
    y = norm.rmsnorm_f32(x, g, 1e-6).astype(np.float64).reshape(T, 1, NG, 128)
    e = of8.unpack_scales(st, T, NG).reshape(T, 1, NG)
    deq = codecs.e4m3_decode(xq).reshape(T, 1, NG, 128) * e[..., None]
    # every decoded payload is within half an E4M3 step (relative 2^-4) of y, or a subnormal step
    err = np.abs(deq - y)
    assert np.all(err <= np.maximum(np.abs(y) * 2.0 ** -4, e[..., None] * 2.0 ** -10))
