"""GPU parity of call chains captured into CUDA graphs.

In a captured graph the library's kernels run back to back with programmatic
dependent launch: a kernel may start while the previous one is finishing and
stream its weights before it waits on it.  These tests replay captured chains
(the decode sweep step, a weight quant right before its linear, the MXFP8 and
FP8 einsum paths) and compare every output with the oracle: bit-exact for the
INT8 path, the 1e-2 relative + 1e-3 absolute bar for the FP8 ones.
"""
import numpy as np
import pytest
import torch

from oracle import codecs, fp8 as of8, int8 as oi8, mx
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import assert_within_tol, bf16_to_dev, bf16_to_np, np_to_dev, within_tol

pytestmark = pytest.mark.gpu


def capture(fn):
    fn()  # eager first: host-side set-up (tensor maps, attributes) outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


def test_int8_decode_sweep_in_one_graph():
    """Quant, GEMM and fused calls over both decode linears and M in {1, 8, 16, 32, 64}, every call on
    its own weights, back to back in one graph (every schedule: one-launch fused, 224-row tiles,
    cluster split-K, tcgen05), replayed three times."""
    dev = torch.device("cuda")
    calls, checks = [], []
    for K, N in [(1024, 32768), (4096, 1024)]:
        ws = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_QUANT_LINEAR, 64, K, N), dev)
        for i, M in enumerate([1, 8, 16, 32, 64]):
            c = synth.int8_linear_case(M, K, N, 8100 + 10 * i + K)
            w2, sw2 = synth.int8_weights(N, K, 8200 + 10 * i + K), synth.channel_scales(N, 8300 + 10 * i + K)
            t = dict(x=bf16_to_dev(c["x"]), w=np_to_dev(c["w_nk"]), sw=np_to_dev(c["sw"]), w2=np_to_dev(w2),
                     sw2=np_to_dev(sw2), xq=torch.empty((M, K), dtype=torch.int8, device=dev),
                     sx=torch.empty((M,), dtype=torch.float32, device=dev),
                     y=torch.empty((M, N), dtype=torch.bfloat16, device=dev),
                     yf=torch.empty((M, N), dtype=torch.bfloat16, device=dev), ws=ws)
            calls.append(t)
            q, s = oi8.dynamic_quant_int8(c["x"])
            checks.append((t, q, s, oi8.w8a8_linear(q, s, c["w_nk"], c["sw"]), oi8.w8a8_linear(q, s, w2, sw2)))

    def step():
        for t in calls:
            fq.dynamic_quant_int8(t["x"], t["xq"], t["sx"])
            fq.w8a8_linear(t["xq"], t["sx"], t["w"], t["sw"], y=t["y"], ws=t["ws"])
            fq.w8a8_quant_linear(t["x"], t["w2"], t["sw2"], y=t["yf"], ws=t["ws"])

    g = capture(step)
    for _ in range(3):
        for t in calls:
            t["y"].zero_()
            t["yf"].zero_()
        g.replay()
        torch.cuda.synchronize()
        for t, q, s, want, want_f in checks:
            assert np.array_equal(t["xq"].cpu().numpy(), q)
            assert np.array_equal(t["sx"].cpu().numpy().view(np.uint32), s.view(np.uint32))
            assert np.array_equal(bf16_to_np(t["y"]), want)
            assert np.array_equal(bf16_to_np(t["yf"]), want_f)
    assert fq.device_error() == (0, 0)


@pytest.mark.parametrize("K,N", [(1024, 32768), (4096, 1024)])
def test_weight_quant_then_linear_in_graph(K, N):
    """A per-channel weight quant and the linear that reads its output, captured back to back; new
    weights are copied in before every replay, so a linear that read its weights before the quant had
    finished would give the previous replay's answer."""
    dev = torch.device("cuda")
    M = 4
    x = synth.activations(M, K, 93)
    q, s = oi8.dynamic_quant_int8(x)
    qd, sd = np_to_dev(q), np_to_dev(s)
    wf_dev = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    wq = torch.empty((N, K), dtype=torch.int8, device=dev)
    swq = torch.empty((N,), dtype=torch.float32, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_LINEAR, M, K, N), dev)
    wf_dev.copy_(bf16_to_dev(synth.activations(N, K, 9000)))
    g = capture(lambda: (fq.dynamic_quant_int8(wf_dev, wq, swq), fq.w8a8_linear(qd, sd, wq, swq, y=y, ws=ws)))
    for i in range(3):
        wf = synth.activations(N, K, 9100 + i)
        wf_dev.copy_(bf16_to_dev(wf))
        g.replay()
        torch.cuda.synchronize()
        oq, os_ = oi8.dynamic_quant_int8(wf)
        assert np.array_equal(bf16_to_np(y), oi8.w8a8_linear(q, s, oq, os_))
    assert fq.device_error() == (0, 0)


def test_mxfp8_chain_in_graph():
    """quant_mxfp8 of the weights, then of the activations, then the linear, captured back to back;
    new weights and activations before every replay."""
    dev = torch.device("cuda")
    M, K, N = 16, 4096, 1024
    w_dev = torch.empty((N, K), dtype=torch.bfloat16, device=dev)
    x_dev = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
    qw = torch.empty((N, K), dtype=torch.float8_e4m3fn, device=dev)
    wsf = torch.empty((N // 128, K // 128, 512), dtype=torch.uint8, device=dev)
    qx = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    xsf = torch.empty((1, K // 128, 512), dtype=torch.uint8, device=dev)
    y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    ws = fq.new_workspace(fq.workspace_bytes(fq.OP_MXFP8_LINEAR, M, K, N), dev)

    def load(i):
        w = codecs.f64_to_bf16(synth.rng(9300 + i).standard_normal((N, K)) * 0.02)
        x = synth.activations(M, K, 9400 + i)
        w_dev.copy_(bf16_to_dev(w))
        x_dev.copy_(bf16_to_dev(x))
        return w, x

    load(0)
    g = capture(lambda: (fq.quant_mxfp8(w_dev, qw, wsf), fq.quant_mxfp8(x_dev, qx, xsf),
                         fq.mxfp8_linear(qx, xsf, qw, wsf, y=y, ws=ws)))
    for i in range(1, 4):
        w, x = load(i)
        g.replay()
        torch.cuda.synchronize()
        oqw, osw = mx.quant_mxfp8(w)
        oqx, osx = mx.quant_mxfp8(x)
        assert_within_tol(bf16_to_np(y), mx.mxfp8_linear(oqx, osx, oqw, osw))
    assert fq.device_error() == (0, 0)


def test_group_quant_then_einsum_in_graph():
    """The FP8 group quant writing packed UE8M0 scales, then the grouped einsum reading them, captured
    back to back for T in {1, 16}; new activations before every replay."""
    dev = torch.device("cuda")
    G, D, N = 8, 4096, 1024
    w = synth.fp8_einsum_weights(G, N, D, 21)
    owq, osw = of8.quantize_weight_fp8_block(w)
    wq, sw = fq.quantize_weight_fp8_block(np_to_dev(w))
    for T in (1, 16):
        x_dev = torch.empty((T, G, D), dtype=torch.bfloat16, device=dev)
        x_dev.copy_(bf16_to_dev(synth.group_activations(T, G, D, 9500 + T)))
        xq, st = fq.quant_fp8_group_ue8m0_packed(x_dev)
        y = torch.empty((T, G, N), dtype=torch.bfloat16, device=dev)
        ws = fq.new_workspace(fq.workspace_bytes(fq.OP_FP8_GROUP_EINSUM, T, D, N, G), dev)
        g = capture(lambda: (fq.quant_fp8_group_ue8m0_packed(x_dev, xq, st),
                             fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw, y=y, ws=ws)))
        for i in range(3):
            x = synth.group_activations(T, G, D, 9600 + 10 * T + i)
            x_dev.copy_(bf16_to_dev(x))
            g.replay()
            torch.cuda.synchronize()
            oxq, ost = of8.quant_fp8_group_ue8m0_packed(x)
            want = of8.fp8_group_einsum(oxq, of8.unpack_scales(ost, T, D // 128), owq, osw)
            ok, info = within_tol(bf16_to_np(y), want)
            assert ok, info
    assert fq.device_error() == (0, 0)
