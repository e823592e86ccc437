"""GPU parity of the MoE expert path: sort/gather/grouped GEMM/combine exact,
SwiGLU within one bf16 ulp on rare elements with the re-quant exact given h,
and the whole chain within 1e-2 rel + 1e-3 abs."""
import numpy as np
import pytest
import torch

from oracle import codecs, int8 as oi8, moe as omoe
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import bf16_to_dev, bf16_to_np, np_to_dev, within_tol

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,topk,E", [(256, 8, 256), (64, 4, 16), (1, 8, 256), (37, 3, 5), (300, 2, 1000),
                                      (0, 8, 16)])
def test_sort_exact(T, topk, E):
    ids = synth.zipf_topk(T, topk, E, 10 + T) if T else np.zeros((0, topk), np.int32)
    off, perm, pair_row = fq.moe_sort(np_to_dev(ids), E)
    torch.cuda.synchronize()
    ooff, operm = omoe.moe_sort(ids, E)
    assert np.array_equal(off.cpu().numpy(), ooff)
    assert np.array_equal(perm.cpu().numpy(), operm)
    pr = pair_row.cpu().numpy()
    assert np.array_equal(pr[operm], np.arange(ids.size))


def test_sort_flags_bad_ids_without_writing_out_of_bounds():
    ids = np.array([[0, 1], [5, 2], [-1, 3]], np.int32)      # 5 and -1 are outside E = 4
    off, perm, _ = fq.moe_sort(np_to_dev(ids), 4)
    st, word = fq.device_error()
    assert st == 8 and word == 2
    assert off.cpu().numpy().tolist() == [0, 1, 2, 3, 4]
    st, word = fq.device_error()                                # the word was cleared
    assert st == 0 and word == 0


def test_gather_exact():
    T, topk, K = 33, 4, 512
    x = synth.activations(T, K, 1)
    ids = synth.zipf_topk(T, topk, 16, 2)
    q, s = fq.dynamic_quant_int8(bf16_to_dev(x))
    _, perm, _ = fq.moe_sort(np_to_dev(ids), 16)
    qg, sg = fq.moe_gather_rows_i8(q, s, perm, topk)
    _, operm = omoe.moe_sort(ids, 16)
    oq, os_ = oi8.dynamic_quant_int8(x)
    assert np.array_equal(qg.cpu().numpy(), omoe.gather_rows(oq, operm, topk))
    assert np.array_equal(sg.cpu().numpy(), omoe.gather_rows(os_, operm, topk))


@pytest.mark.parametrize("sched", ["auto", "streamk"])
@pytest.mark.parametrize("R,E,K,N", [(64, 8, 256, 256), (300, 16, 1024, 384), (5, 3, 128, 128), (2048, 64, 512, 256),
                                     (700, 12, 4096, 256), (90, 5, 4224, 128)])
def test_grouped_linear_exact(R, E, K, N, sched, monkeypatch):
    # auto runs the tcgen05 kernel for K <= 4096; streamk forces the mma.sync kernel
    if sched != "auto":
        monkeypatch.setenv("FQ_FORCE_SCHEDULE", sched)
    r = np.random.default_rng(R + E)
    counts = r.multinomial(R, r.dirichlet(np.ones(E) * 0.3))
    counts[0] = 0 if E > 2 else counts[0]                     # an empty expert
    counts[-1] += R - counts.sum()
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    x = synth.activations(R, K, 3)
    q, s = oi8.dynamic_quant_int8(x)
    w = synth.uniform_int8((E, N, K), 4)
    sw = synth.rng(5).uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    y = fq.w8a8_grouped_linear(np_to_dev(q), np_to_dev(s), np_to_dev(off), np_to_dev(w), np_to_dev(sw))
    want = omoe.w8a8_grouped_linear(q, s, off, w, sw)
    assert np.array_equal(bf16_to_np(y), want)


def assert_swiglu_exact(gu):
    """GPU h, hq and sh equal the oracle's bit for bit on the raw inputs."""
    hq, sh, h = fq.swiglu_quant_int8(bf16_to_dev(gu), return_h=True)
    torch.cuda.synchronize()
    ohq, osh, oh = omoe.swiglu_quant_int8(gu)
    hg = bf16_to_np(h)
    bad = np.nonzero(hg != oh)
    assert bad[0].size == 0, ("h differs", bad[0][:4], bad[1][:4], hg[bad][:4], oh[bad][:4])
    assert np.array_equal(hq.cpu().numpy(), ohq)
    assert np.array_equal(sh.cpu().numpy().view(np.uint32), osh.view(np.uint32))


@pytest.mark.parametrize("rows,I", [(2048, 2048), (7, 16), (33, 4096), (1, 128)])
def test_swiglu_quant(rows, I):
    gu = synth.activations(rows, 2 * I, 8 + rows)
    # scale like a gate/up projection output (|v| up to ~100)
    gu = codecs.f32_to_bf16(codecs.bf16_to_f32(gu) * np.float32(8.0))
    assert_swiglu_exact(gu)


def test_swiglu_every_bf16_gate():
    """Every finite bf16 gate value g, each with several up values u (one row per u)."""
    bits = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    g = bits[np.isfinite(bits)]
    g = np.concatenate([g, np.zeros(16 - g.size % 16 if g.size % 16 else 0, np.float32)])
    us = np.array([1.0, -0.75, 0.3671875, -7.5e-3, 2.0 ** -100], np.float32)   # |h| stays finite
    gu = np.concatenate([np.stack([g, np.full_like(g, u)]).reshape(1, -1) for u in us])
    assert_swiglu_exact(codecs.f32_to_bf16(gu))


def test_swiglu_bf16_rounding_boundaries():
    """Pairs (g, u) whose product fp32(silu(g) * u) lies within 24 fp32 ulps of a
    bf16 rounding midpoint - or exactly on one (a tie) - the cases where an fp32
    silu estimate alone could round h either way."""
    r = np.random.default_rng(1234)
    n = 1 << 22
    g = codecs.bf16_to_f32(codecs.f32_to_bf16(r.normal(0, 4, n).astype(np.float32)))
    u = codecs.bf16_to_f32(codecs.f32_to_bf16(r.normal(0, 4, n).astype(np.float32)))
    p = (omoe.silu_f32(g) * u).astype(np.float32).view(np.uint32)
    low = (p & 0xFFFF).astype(np.int64)
    near = np.abs(low - 0x8000) <= 24
    ties = int(np.count_nonzero(low[near] == 0x8000))
    sel = np.nonzero(near)[0]
    assert sel.size > 1000 and ties > 0
    k = sel.size - sel.size % 16
    gu = np.stack([g[sel[:k]], u[sel[:k]]]).reshape(2, -1, 16).transpose(1, 0, 2).reshape(-1, 32)
    assert_swiglu_exact(codecs.f32_to_bf16(gu))


def test_combine_exact():
    T, topk, H = 40, 8, 512
    ids = synth.zipf_topk(T, topk, 64, 6)
    _, operm = omoe.moe_sort(ids, 64)
    y = synth.activations(T * topk, H, 7)
    w = synth.topk_weights(T, topk, 8)
    _, _, pair_row = fq.moe_sort(np_to_dev(ids), 64)
    out = fq.moe_combine(bf16_to_dev(y), pair_row, np_to_dev(w))
    assert np.array_equal(bf16_to_np(out), omoe.moe_combine(y, operm, w, T, topk))


def run_chain_steps(x, ids, w, W):
    """The GPU chain, keeping every intermediate."""
    T, topk = ids.shape
    E = W["w13"].shape[0]
    xq, sx = fq.dynamic_quant_int8(x)
    off, perm, pair_row = fq.moe_sort(ids, E)
    xg, sg = fq.moe_gather_rows_i8(xq, sx, perm, topk)
    y1 = fq.w8a8_grouped_linear(xg, sg, off, W["w13"], W["sw13"])
    hq, sh, h = fq.swiglu_quant_int8(y1, return_h=True)
    y2 = fq.w8a8_grouped_linear(hq, sh, off, W["w2"], W["sw2"])
    out = fq.moe_combine(y2, pair_row, w)
    torch.cuda.synchronize()
    return dict(off=off, perm=perm, xg=xg, sg=sg, y1=y1, hq=hq, sh=sh, h=h, y2=y2, out=out)


def test_moe_chain_small_full_oracle():
    c = synth.moe_case(64, 4, 16, 256, 128, 21)
    W = {k: np_to_dev(c[k]) for k in ("w13", "sw13", "w2", "sw2")}
    g = run_chain_steps(bf16_to_dev(c["x"]), np_to_dev(c["topk_ids"]), np_to_dev(c["topk_w"]), W)
    r = omoe.moe_forward(c["x"], c["topk_ids"], c["topk_w"], c["w13"], c["sw13"], c["w2"], c["sw2"])
    assert np.array_equal(bf16_to_np(g["y1"]), r["y1"])
    assert np.array_equal(bf16_to_np(g["h"]), r["h"])
    assert np.array_equal(g["hq"].cpu().numpy(), r["hq"])
    assert np.array_equal(g["sh"].cpu().numpy().view(np.uint32), r["sh"].view(np.uint32))
    assert np.array_equal(bf16_to_np(g["y2"]), r["y2"])
    assert np.array_equal(bf16_to_np(g["out"]), r["out"])                     # the whole chain is exact


def test_moe_chain_full_size_sampled_tokens():
    """256 tokens, hidden 4096, 256 experts, top-8 Zipf(1.1), W13 [256, 4096, 4096],
    W2 [256, 4096, 2048]: one full-size pass on the GPU; the oracle recomputes a
    sample of tokens through their eight experts."""
    T, topk, E, H, I = 256, 8, 256, 4096, 2048
    c = synth.moe_case(T, topk, E, H, I, 31, with_weights=False)
    W = synth.moe_weights_device(E, H, I, 31, torch.device("cuda"))
    g = run_chain_steps(bf16_to_dev(c["x"]), np_to_dev(c["topk_ids"]), np_to_dev(c["topk_w"]), W)
    q, s = oi8.dynamic_quant_int8(c["x"])
    off, perm = omoe.moe_sort(c["topk_ids"], E)
    assert np.array_equal(g["off"].cpu().numpy(), off) and np.array_equal(g["perm"].cpu().numpy(), perm)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    y1g, hg, y2g, outg = (bf16_to_np(g[k]) for k in ("y1", "h", "y2", "out"))
    hqg, shg = g["hq"].cpu().numpy(), g["sh"].cpu().numpy()
    for t in [0, 1, 77, 128, 200, 255]:
        acc = np.zeros(H, np.float32)
        for j in range(topk):
            e = int(c["topk_ids"][t, j])
            row = int(inv[t * topk + j])
            w13 = W["w13"][e].cpu().numpy()
            y1 = oi8.w8a8_linear(q[t:t + 1], s[t:t + 1], w13, W["sw13"][e].cpu().numpy())
            assert np.array_equal(y1g[row:row + 1], y1)                          # exact
            oq, os_, h = omoe.swiglu_quant_int8(y1)
            assert np.array_equal(hg[row:row + 1], h)                            # exact
            assert np.array_equal(hqg[row:row + 1], oq) and shg[row] == os_[0]
            y2 = oi8.w8a8_linear(oq, os_, W["w2"][e].cpu().numpy(), W["sw2"][e].cpu().numpy())
            assert np.array_equal(y2g[row:row + 1], y2)                          # exact
            acc = (acc + (np.float32(c["topk_w"][t, j]) * codecs.bf16_to_f32(y2[0])).astype(np.float32)).astype(np.float32)
        assert np.array_equal(outg[t], codecs.f32_to_bf16(acc))


@pytest.mark.parametrize("K", [256, 384, 1024])
def test_grouped_linear_few_iterations_many_ctas(K):
    """Fewer (tile, k-block) iterations than CTAs: empty-range CTAs sit between the
    contributors of a split tile and must not be summed."""
    E, N = 8, 256
    counts = np.array([0, 2, 24, 8, 2, 15, 13, 0])
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(counts.sum())
    x = synth.activations(R, K, 13)
    q, s = oi8.dynamic_quant_int8(x)
    w = synth.uniform_int8((E, N, K), 14)
    sw = synth.rng(15).uniform(1e-3, 1e-2, (E, N)).astype(np.float32)
    for _ in range(2):
        y = fq.w8a8_grouped_linear(np_to_dev(q), np_to_dev(s), np_to_dev(off), np_to_dev(w), np_to_dev(sw))
        assert np.array_equal(bf16_to_np(y), omoe.w8a8_grouped_linear(q, s, off, w, sw))
