"""GPU parity of the FP8 path: group quant + packed UE8M0 layout (bit-exact),
fp32-scale control + repack (bit-exact), weight block quant (bit-exact) and the
block-scaled einsum (tolerance 1e-2 rel + 1e-3 abs; packed vs fp32 scales
bit-identical)."""
import json
import os

import numpy as np
import pytest
import torch

from oracle import codecs, fp8 as of8
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import assert_within_tol, bf16_to_dev, bf16_to_np, e4m3_to_np, e4m3_to_dev, np_to_dev, within_tol

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gpu_group_quant(x_bits):
    xq, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(x_bits))
    torch.cuda.synchronize()
    return e4m3_to_np(xq), st.cpu().numpy()


@pytest.mark.parametrize("T,G,D", [(1, 8, 4096), (3, 8, 4096), (4, 8, 4096), (17, 8, 4096), (128, 8, 4096),
                                   (5, 3, 384), (2, 2, 640), (6, 1, 128), (9, 4, 1152)])
def test_group_quant_bit_exact(T, G, D):
    x = synth.group_activations(T, G, D, 4000 + T * 3 + G + D)
    xq, st = gpu_group_quant(x)
    oxq, ost = of8.quant_fp8_group_ue8m0_packed(x)
    assert st.shape == ost.shape and st.dtype == np.int32
    assert np.array_equal(st, ost)
    assert np.array_equal(xq, oxq)


def test_group_quant_full_size_sampled_tokens():
    """T = 4096, G = 8, D = 4096 in one launch; tokens are independent, so the
    oracle is run on a sample of them and compared byte for byte."""
    T, G, D = 4096, 8, 4096
    x = synth.group_activations(T, G, D, 4242)
    xq, st = gpu_group_quant(x)
    NG, P, Ta = of8.packed_dims(T, D)
    assert st.shape == (G, P, Ta)
    sample = np.unique(np.concatenate([[0, 1, T - 1], np.random.default_rng(1).integers(0, T, 61)]))
    oxq, oe = of8.quant_fp8_group(x[sample])
    assert np.array_equal(xq[sample], oxq)
    by = st.view(np.uint8).reshape(G, P, Ta, 4)
    for i, t in enumerate(sample):
        for j in range(NG):
            assert by[:, j // 4, t, j % 4].tolist() == (oe[i, :, j] + 127).tolist()


def test_group_quant_token_padding_and_tail_zero():
    for T, D in [(1, 384), (3, 640), (5, 1152), (17, 384)]:
        x = synth.group_activations(T, 2, D, T + D)
        _, st = gpu_group_quant(x)
        NG, P, Ta = of8.packed_dims(T, D)
        by = st.view(np.uint8).reshape(2, P, Ta, 4)
        assert np.all(by[:, :, T:, :] == 0)
        for j in range(NG, 4 * P):
            assert np.all(by[:, j // 4, :, j % 4] == 0)


def test_group_quant_garbage_in_storage_is_overwritten():
    """The storage handed in may hold allocator garbage: every byte must be written."""
    T, G, D = 3, 2, 640
    x = synth.group_activations(T, G, D, 77)
    xg = bf16_to_dev(x)
    xq = torch.empty((T, G, D), dtype=torch.float8_e4m3fn, device="cuda")
    st = torch.full((G, 2, 4), -1, dtype=torch.int32, device="cuda")
    L = fq.lib()
    import ctypes
    rc = L.quant_fp8_group_ue8m0_packed(ctypes.c_void_p(xg.data_ptr()), T, G, D, ctypes.c_void_p(xq.data_ptr()),
                                        ctypes.c_void_p(st.data_ptr()), fq._stream())
    assert rc == 0
    _, ost = of8.quant_fp8_group_ue8m0_packed(x)
    assert np.array_equal(st.cpu().numpy(), ost)


def test_group_quant_golden_layout():
    d = json.load(open(os.path.join(GOLD, "ue8m0_layout.json")))["layout"]
    T, G, D = d["T"], d["G"], d["D"]
    x = np.zeros((T, G, D), np.float32)
    for g in range(G):
        for j in range(D // 128):
            x[0, g, j * 128 + 5] = 448.0 * 2.0 ** (j - 2 + 3 * g)
    _, st = gpu_group_quant(codecs.f32_to_bf16(x))
    assert st.astype("<i4").tobytes().hex() == d["storage_bytes_hex"]


def test_group_quant_empty_tokens():
    x = torch.empty((0, 3, 128), dtype=torch.bfloat16, device="cuda")
    xq, st = fq.quant_fp8_group_ue8m0_packed(x)
    assert tuple(st.shape) == (3, 1, 0)
    assert tuple(fq.scale_view(st, 0).shape) == (0, 3, 1)


def test_logical_view_shape_and_strides():
    x = synth.group_activations(5, 8, 4096, 9)
    _, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(x))
    v = fq.scale_view(st, 5)
    assert tuple(v.shape) == (5, 8, 8) and v.dtype == torch.int32
    assert tuple(v.stride()) == (1, 8 * 8, 8)


@pytest.mark.parametrize("T,G,D", [(1, 8, 4096), (17, 8, 4096), (6, 3, 384), (3, 2, 640)])
def test_fp32_scale_control_and_repack(T, G, D):
    x = synth.group_activations(T, G, D, 5000 + T)
    xg = bf16_to_dev(x)
    xq32, s32 = fq.quant_fp8_group_fp32(xg)
    xqp, stp = fq.quant_fp8_group_ue8m0_packed(xg)
    rep = fq.pack_scales_ue8m0(s32)
    torch.cuda.synchronize()
    _, os32 = of8.quant_fp8_group_fp32_scales(x)
    assert np.array_equal(s32.cpu().numpy().view(np.uint32), os32.view(np.uint32))
    assert torch.equal(xq32.view(torch.uint8), xqp.view(torch.uint8))
    assert torch.equal(rep, stp)
    assert np.array_equal(rep.cpu().numpy(), of8.repack_fp32_scales_to_ue8m0(os32))


@pytest.mark.parametrize("G,N,D", [(2, 256, 384), (1, 128, 128), (8, 1024, 4096)])
def test_weight_block_quant_bit_exact(G, N, D):
    w = synth.fp8_einsum_weights(G, N, D, 6000 + G + N)
    wq, sw = fq.quantize_weight_fp8_block(np_to_dev(w))
    torch.cuda.synchronize()
    owq, osw = of8.quantize_weight_fp8_block(w)
    assert np.array_equal(sw.cpu().numpy().view(np.uint32), osw.view(np.uint32))
    assert np.array_equal(e4m3_to_np(wq), owq)


_W_CACHE = {}


def einsum_weights(G, N, D, seed):
    key = (G, N, D, seed)
    if key not in _W_CACHE:
        w = synth.fp8_einsum_weights(G, N, D, seed)
        owq, osw = of8.quantize_weight_fp8_block(w)
        wq, sw = fq.quantize_weight_fp8_block(np_to_dev(w))
        _W_CACHE[key] = (owq, osw, wq, sw)
    return _W_CACHE[key]


@pytest.mark.parametrize("T,G,D,N", [(1, 8, 4096, 1024), (4, 8, 4096, 1024), (16, 8, 4096, 1024),
                                     (64, 8, 4096, 1024), (256, 8, 4096, 1024), (3, 2, 384, 256),
                                     (1, 1, 128, 128), (100, 3, 640, 384)])
def test_einsum_within_tolerance_and_scale_formats_identical(T, G, D, N):
    x = synth.group_activations(T, G, D, 7000 + T + G)
    owq, osw, wq, sw = einsum_weights(G, N, D, 7)
    xg = bf16_to_dev(x)
    xq, st = fq.quant_fp8_group_ue8m0_packed(xg)
    _, s32 = fq.quant_fp8_group_fp32(xg)
    y_packed = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw)
    y_f32 = fq.fp8_group_einsum(xq, s32, fq.SCALE_FP32, wq, sw)
    torch.cuda.synchronize()
    assert torch.equal(y_packed.view(torch.int16), y_f32.view(torch.int16))      # bit-identical
    oxq, ost = of8.quant_fp8_group_ue8m0_packed(x)
    want = of8.fp8_group_einsum(oxq, of8.unpack_scales(ost, T, D // 128), owq, osw)
    ok, info = within_tol(bf16_to_np(y_packed), want)
    assert ok, info


@pytest.mark.parametrize("kd", [1, 2, 4])
@pytest.mark.parametrize("bm", [128, 64])
@pytest.mark.parametrize("sched", ["dp", "streamk"])
@pytest.mark.parametrize("T,G,D,N", [(1, 8, 4096, 1024), (5, 8, 4096, 1024), (16, 8, 4096, 1024),
                                     (40, 8, 4096, 1024), (3, 3, 640, 384), (9, 2, 384, 256),
                                     (2, 2, 768, 256), (3, 2, 8192, 256), (1, 1, 5120, 128)])
def test_einsum_both_schedules(kd, bm, sched, T, G, D, N, monkeypatch):
    """Whole tiles, one per CTA (dp), and tiles split over CTAs by chunks of
    K blocks (stream-K); 128 and 64 weight rows per tile (M = 128 and M = 64
    MMAs); 1, 2 or 4 K blocks per pipeline stage (one 3-D copy each; a count
    that does not divide the K blocks or leaves too few stages is not taken);
    D = 8192 and 5120 take the promotion factors in several pieces per tile:
    each within tolerance, packed and fp32 scales identical, repeat calls
    identical."""
    monkeypatch.setenv("FQ_FORCE_SCHEDULE", sched)
    monkeypatch.setenv("FQ_EINSUM_BM", str(bm))
    monkeypatch.setenv("FQ_EINSUM_KD", str(kd))
    x = synth.group_activations(T, G, D, 7300 + T + G)
    owq, osw, wq, sw = einsum_weights(G, N, D, 9)
    xg = bf16_to_dev(x)
    xq, st = fq.quant_fp8_group_ue8m0_packed(xg)
    _, s32 = fq.quant_fp8_group_fp32(xg)
    y1 = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw)
    y2 = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw)
    yf = fq.fp8_group_einsum(xq, s32, fq.SCALE_FP32, wq, sw)
    torch.cuda.synchronize()
    assert torch.equal(y1.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y1.view(torch.int16), yf.view(torch.int16))
    oxq, ost = of8.quant_fp8_group_ue8m0_packed(x)
    assert_within_tol(bf16_to_np(y1), of8.fp8_group_einsum(oxq, of8.unpack_scales(ost, T, D // 128), owq, osw))
    assert fq.device_error() == (0, 0)


def test_einsum_integer_case_exact():
    """Unit scales and small-integer E4M3 operands: every sum is an exact integer."""
    T, G, D, N = 5, 2, 256, 128
    r = np.random.default_rng(3)
    xi = r.integers(-8, 9, (T, G, D))
    wi = r.integers(-8, 9, (G, N, D))
    xq = e4m3_to_dev(codecs.e4m3_encode(xi))
    wq = e4m3_to_dev(codecs.e4m3_encode(wi))
    st = np.zeros((G, 1, 8), np.int32)
    st.view(np.uint8).reshape(G, 1, 8, 4)[:, :, :T, :2] = 127           # 2^0 for both k-blocks
    sw = torch.ones((G, 2, 1), dtype=torch.float32, device="cuda")
    y = fq.fp8_group_einsum(xq, np_to_dev(st), fq.SCALE_UE8M0_PACKED, wq, sw)
    want = codecs.f64_to_bf16(np.einsum("tgd,gnd->tgn", xi, wi).astype(np.float64))
    assert np.array_equal(bf16_to_np(y), want)


@pytest.mark.parametrize("T", [1, 4, 16])
def test_einsum_repeatable(T):
    """Twelve identical calls give identical bits.  Guards the stage hand-back:
    stages read with ld.shared must be fenced against the next TMA write
    (generic -> async proxy) before the producer may refill them."""
    G, D, N = 8, 4096, 1024
    x = synth.group_activations(T, G, D, 99 + T)
    _, _, wq, sw = einsum_weights(G, N, D, 7)
    xq, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(x))
    ys = [fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw).view(torch.int16).clone() for _ in range(12)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_einsum_many_operand_addresses():
    """Hundreds of calls whose weight and activation tensors sit at different
    addresses: the encoded TMA descriptors are cached by address and shape, and
    a weight descriptor must survive the activation lookup even when both keys
    share a cache slot (with 256 slots, 400 calls make that near certain)."""
    T, G, D, N = 4, 1, 256, 128
    _, _, wq, sw = einsum_weights(G, N, D, 21)
    x = synth.group_activations(T, G, D, 22)
    xq, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(x))
    ref = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw).view(torch.int16).clone()
    wbytes, xbytes = wq.view(torch.uint8).reshape(-1), xq.view(torch.uint8).reshape(-1)
    calls = 400
    wbuf = torch.empty(wbytes.numel() + 16 * calls, dtype=torch.uint8, device="cuda")
    xbuf = torch.empty(xbytes.numel() + 16 * calls, dtype=torch.uint8, device="cuda")
    for i in range(calls):
        wo, xo = 16 * i, 16 * ((7 * i) % calls)
        wbuf[wo:wo + wbytes.numel()] = wbytes
        xbuf[xo:xo + xbytes.numel()] = xbytes
        wv = wbuf[wo:wo + wbytes.numel()].view(torch.float8_e4m3fn).view(G, N, D)
        xv = xbuf[xo:xo + xbytes.numel()].view(torch.float8_e4m3fn).view(T, G, D)
        y = fq.fp8_group_einsum(xv, st, fq.SCALE_UE8M0_PACKED, wv, sw)
        assert torch.equal(y.view(torch.int16), ref), "call %d differs" % i
    assert fq.device_error() == (0, 0)


def test_tiny_group_scale_byte_zero():
    """A group whose absmax is tiny but nonzero clamps its exponent to -127
    (byte 0) while its E4M3 codes stay nonzero: the quant must match the
    oracle, and the einsum must decode byte 0 as 2^-127 in both scale formats."""
    T, G, D, N = 2, 2, 256, 128
    x = synth.group_activations(T, G, D, 31)
    xf = codecs.bf16_to_f32(x).astype(np.float64)
    xf[0, 0, :128] *= 2.0 ** -121 / np.abs(xf[0, 0, :128]).max()  # amax 2^-121: exponent clamps to -127
    xf[1, 1, 128:] = 0.0            # and an all-zero group
    xb = codecs.f64_to_bf16(xf)
    xq, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(xb))
    oxq, ost = of8.quant_fp8_group_ue8m0_packed(xb)
    assert np.array_equal(st.cpu().numpy(), ost)
    assert np.array_equal(e4m3_to_np(xq), oxq)
    assert (ost.view(np.uint8).reshape(-1) == 0).any()
    _, s32 = fq.quant_fp8_group_fp32(bf16_to_dev(xb))
    owq, osw, wq, sw = einsum_weights(G, N, D, 32)
    yp = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw)
    yf = fq.fp8_group_einsum(xq, s32, fq.SCALE_FP32, wq, sw)
    assert torch.equal(yp.view(torch.int16), yf.view(torch.int16))
    want = of8.fp8_group_einsum(oxq, of8.unpack_scales(ost, T, D // 128), owq, osw)
    assert_within_tol(bf16_to_np(yp), want)


def test_einsum_rows_independent_of_T():
    """A token's output row does not depend on the other tokens of the call:
    T = 1 and T = 3 give bit-for-bit the first rows of the T = 4 call on the
    same inputs (the schedule depends on the token-tile count, which is the
    same for all three, and each token's sums use only its own column)."""
    G, D, N = 8, 4096, 1024
    x4 = synth.group_activations(4, G, D, 7711)
    _, _, wq, sw = einsum_weights(G, N, D, 7)
    ys = {}
    for T in (1, 3, 4):
        xq, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(np.ascontiguousarray(x4[:T])))
        ys[T] = fq.fp8_group_einsum(xq, st, fq.SCALE_UE8M0_PACKED, wq, sw).view(torch.int16)
    torch.cuda.synchronize()
    assert torch.equal(ys[1], ys[4][:1])
    assert torch.equal(ys[3], ys[4][:3])
