"""GPU parity of the RMSNorm + quant producer against the oracle.

Bar: bit-exact.  The row statistic is an exact sum of squares rounded once
and the rest are IEEE-rounded fp64/fp32 steps, so the fp32 row and every
quant decision on it have one correct value.
"""
import numpy as np
import pytest
import torch

from oracle import codecs, norm
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import bf16_to_dev, e4m3_to_np

pytestmark = pytest.mark.gpu

SHAPES = [(1, 4096), (4, 4096), (64, 4096), (3, 7168), (5, 384), (9, 128), (17, 16384), (130, 1024), (2, 2048)]


def case(M, K, seed):
    x = synth.activations(M, K, seed)
    g = codecs.f64_to_bf16(1.0 + 0.25 * synth.rng(seed + 1).standard_normal(K))
    return x, g


@pytest.mark.parametrize("eps", [1e-6, 0.0, 0.5])
@pytest.mark.parametrize("M,K", SHAPES + [(7, 16), (3, 48)])
def test_int8_bit_exact(M, K, eps):
    x, g = case(M, K, 6000 + M + K)
    q, s = fq.rmsnorm_quant_int8(bf16_to_dev(x), bf16_to_dev(g), eps)
    oq, os_ = norm.rmsnorm_quant_int8(x, g, eps)
    assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q.cpu().numpy(), oq)


@pytest.mark.parametrize("eps", [1e-6, 0.0])
@pytest.mark.parametrize("M,K", SHAPES)
def test_fp8_bit_exact(M, K, eps):
    x, g = case(M, K, 7000 + M + K)
    xq, st = fq.rmsnorm_quant_fp8_ue8m0_packed(bf16_to_dev(x), bf16_to_dev(g), eps)
    oxq, ost = norm.rmsnorm_quant_fp8_ue8m0_packed(x, g, eps)
    assert np.array_equal(st.cpu().numpy(), ost)
    assert np.array_equal(e4m3_to_np(xq), oxq)


def test_edge_rows():
    # zero row (eps 0 and > 0), a row of one huge outlier, a row of bf16
    # subnormals, a constant row, alternating signs
    K = 512
    rows = np.zeros((6, K))
    rows[1, 7] = 3.0e38
    rows[2] = 2.0 ** -130 * (1 + np.arange(K) % 7)
    rows[3] = 3.0
    rows[4] = np.where(np.arange(K) % 2, -1.5, 1.5)
    rows[5, :5] = [1e-30, -2e30, 5.0, -7.0, 1e-3]
    g = codecs.f64_to_bf16(np.linspace(-2, 2, K))
    for eps in (0.0, 1e-6):
        # with eps = 0 the all-subnormal row would make 1/rms overflow fp32
        # (outside the contract); it runs only with eps > 0
        x = codecs.f64_to_bf16(rows if eps > 0 else np.delete(rows, 2, axis=0))
        q, s = fq.rmsnorm_quant_int8(bf16_to_dev(x), bf16_to_dev(g), eps)
        oq, os_ = norm.rmsnorm_quant_int8(x, g, eps)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32)), eps
        assert np.array_equal(q.cpu().numpy(), oq), eps
        xq, st = fq.rmsnorm_quant_fp8_ue8m0_packed(bf16_to_dev(x), bf16_to_dev(g), eps)
        oxq, ost = norm.rmsnorm_quant_fp8_ue8m0_packed(x, g, eps)
        assert np.array_equal(st.cpu().numpy(), ost), eps
        assert np.array_equal(e4m3_to_np(xq), oxq), eps


def test_feeds_the_linear():
    # the (int8, scale) tuple goes straight into the W8A8 linear
    from oracle import int8 as oi8
    M, K, N = 4, 4096, 1024
    x, g = case(M, K, 8100)
    w = synth.uniform_int8((N, K), 8101)
    sw = synth.channel_scales(N, 8102)
    q, s = fq.rmsnorm_quant_int8(bf16_to_dev(x), bf16_to_dev(g), 1e-6)
    y = fq.w8a8_linear(q, s, torch.from_numpy(w).cuda(), torch.from_numpy(sw).cuda())
    oq, os_ = norm.rmsnorm_quant_int8(x, g, 1e-6)
    want = oi8.w8a8_linear(oq, os_, w, sw)
    assert np.array_equal(y.cpu().view(torch.int16).numpy().view(np.uint16), want)


@pytest.mark.parametrize("K", [16, 128, 4096])
def test_wide_exponent_rows_and_ties(K):
    """Rows whose values span ~2^250 (squares far below the largest one are
    summed through the sticky bit) and rows whose two large squares sum to an
    fp64 rounding tie that only the tiny terms break."""
    r = synth.rng(9000 + K)
    rows = []
    for _ in range(12):
        rows.append(r.standard_normal(K) * np.exp2(r.uniform(-125, 120, K)))
    for _ in range(4):
        t = np.zeros(K)
        t[0], t[1] = 1.5 * 2.0 ** 40, 1.25 * 2.0 ** 14
        t[2:] = 2.0 ** -100 * r.standard_normal(K - 2)
        rows.append(t)
    x = codecs.f64_to_bf16(np.clip(np.array(rows), -3e38, 3e38))
    g = codecs.f64_to_bf16(1.0 + 0.25 * r.standard_normal(K))
    for eps in (0.0, 1e-6):
        q, s = fq.rmsnorm_quant_int8(bf16_to_dev(x), bf16_to_dev(g), eps)
        oq, os_ = norm.rmsnorm_quant_int8(x, g, eps)
        assert np.array_equal(s.cpu().numpy().view(np.uint32), os_.view(np.uint32)), eps
        assert np.array_equal(q.cpu().numpy(), oq), eps
