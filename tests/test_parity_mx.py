"""GPU parity of the 32-element block-scaled FP8 path (MXFP8-like).

Producer: bit-exact (E4M3 codes and the blocked UE8M0 scale bytes).  Linear:
the tensor cores accumulate in fp32, so Y is held to 1e-2 relative + 1e-3
absolute against the exact block-scaled sum rounded once (the einsum's bar),
and repeated calls must give identical bits.
"""
import numpy as np
import pytest
import torch

from oracle import codecs, mx
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import assert_within_tol, bf16_to_dev, bf16_to_np, e4m3_to_np, within_tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("R,K", [(1, 128), (3, 256), (130, 384), (64, 4096), (300, 1024), (1024, 128)])
def test_quant_bit_exact(R, K):
    x = synth.activations(R, K, 500 + R + K)
    q, sf = fq.quant_mxfp8(bf16_to_dev(x))
    oq, os_ = mx.quant_mxfp8(x)
    assert np.array_equal(e4m3_to_np(q), oq)
    assert np.array_equal(sf.cpu().numpy(), mx.pack_sf_blocked(os_))


def weights(N, K, seed):
    w = codecs.f64_to_bf16(synth.rng(seed).standard_normal((N, K)) * 0.02)
    return w, mx.quant_mxfp8(w)


@pytest.mark.parametrize("M,K,N", [(1, 4096, 1024), (4, 4096, 1024), (16, 1024, 512), (17, 512, 384),
                                   (33, 256, 128), (64, 4096, 256), (100, 384, 272), (130, 256, 128)])
def test_linear_within_tolerance(M, K, N):
    x = synth.activations(M, K, 600 + M + K)
    _, (oqw, osw) = weights(N, K, 601 + N)
    qx, sx = fq.quant_mxfp8(bf16_to_dev(x))
    qw = torch.from_numpy(oqw).cuda().view(torch.float8_e4m3fn)
    wsf = torch.from_numpy(mx.pack_sf_blocked(osw)).cuda()
    y = fq.mxfp8_linear(qx, sx, qw, wsf)
    oqx, osx = mx.quant_mxfp8(x)
    want = mx.mxfp8_linear(oqx, osx, oqw, osw)
    assert_within_tol(bf16_to_np(y), want)
    assert fq.device_error() == (0, 0)


@pytest.mark.parametrize("M", [1, 4, 64, 200])
def test_linear_repeatable(M):
    K, N = 2048, 1024
    x = synth.activations(M, K, 700 + M)
    _, (oqw, osw) = weights(N, K, 701)
    qx, sx = fq.quant_mxfp8(bf16_to_dev(x))
    qw = torch.from_numpy(oqw).cuda().view(torch.float8_e4m3fn)
    wsf = torch.from_numpy(mx.pack_sf_blocked(osw)).cuda()
    ys = [fq.mxfp8_linear(qx, sx, qw, wsf).view(torch.int16).clone() for _ in range(8)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_integer_case_exact():
    # small integer codes with unit scales: every block sum is exact in fp32,
    # so the result is the integer product rounded once to bf16
    M, K, N = 8, 512, 256
    r = synth.rng(710)
    xi = r.integers(-6, 7, (M, K)).astype(np.float64)
    wi = r.integers(-6, 7, (N, K)).astype(np.float64)
    qx = torch.from_numpy(codecs.e4m3_encode(xi)).cuda().view(torch.float8_e4m3fn)
    qw = torch.from_numpy(codecs.e4m3_encode(wi)).cuda().view(torch.float8_e4m3fn)
    sx = torch.from_numpy(mx.pack_sf_blocked(np.full((M, K // 32), 127, np.uint8))).cuda()
    sw = torch.from_numpy(mx.pack_sf_blocked(np.full((N, K // 32), 127, np.uint8))).cuda()
    y = fq.mxfp8_linear(qx, sx, qw, sw)
    assert np.array_equal(bf16_to_np(y), codecs.f64_to_bf16(xi @ wi.T))


def test_many_iterations_per_cta_no_drain_stall():
    """K=1024, N=32768: ~13 k-blocks per CTA, more than the stage ring holds, so
    stages are reused and a CTA covers three segments.  Checks sampled columns
    against the oracle and that a warm call does not stall at exit."""
    import time
    M, K, N = 1, 1024, 32768
    x = synth.activations(M, K, 720)
    w = codecs.f64_to_bf16(synth.rng(721).standard_normal((N, K)) * 0.02)
    qx, sx = fq.quant_mxfp8(bf16_to_dev(x))
    qw, sw = fq.quant_mxfp8(bf16_to_dev(w))
    y = fq.mxfp8_linear(qx, sx, qw, sw)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    y = fq.mxfp8_linear(qx, sx, qw, sw)
    torch.cuda.synchronize()
    assert time.perf_counter() - t0 < 0.1
    assert fq.device_error() == (0, 0)
    cols = np.r_[0:256, 16384:16640, 32512:32768]
    oqx, osx = mx.quant_mxfp8(x)
    oqw, osw = mx.quant_mxfp8(w[cols])
    want = mx.mxfp8_linear(oqx, osx, oqw, osw)
    assert_within_tol(bf16_to_np(y)[:, cols], want)


def test_linear_right_after_weight_quant():
    """quant_mxfp8 of the weights launched right before mxfp8_linear with nothing else on the stream in
    between: the linear streams its weights and their scales before it waits on the previous kernel."""
    dev = torch.device("cuda")
    M, K, N = 4, 4096, 1024
    x = synth.activations(M, K, 95)
    qx, sx = fq.quant_mxfp8(bf16_to_dev(x))
    oqx, osx = mx.quant_mxfp8(x)
    qw = torch.empty(N, K, dtype=torch.float8_e4m3fn, device=dev)
    wsf = torch.empty((N // 128, K // 128, 512), dtype=torch.uint8, device=dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = fq.new_workspace(fq.workspace_bytes(fq.OP_MXFP8_LINEAR, M, K, N), dev)
    for i in range(3):
        w, (oqw, osw) = weights(N, K, 700 + i)
        wd = bf16_to_dev(w)
        torch.cuda.synchronize()
        fq.quant_mxfp8(wd, qw, wsf)
        fq.mxfp8_linear(qx, sx, qw, wsf, y=y, ws=ws)
        torch.cuda.synchronize()
        assert_within_tol(bf16_to_np(y), mx.mxfp8_linear(oqx, osx, oqw, osw))
    assert fq.device_error() == (0, 0)
