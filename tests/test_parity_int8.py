"""GPU parity of the INT8 path (dynamic quant, W8A8 linear, fused) against the oracle.

Bar: bit-exact.  The quant is an integer decision taken in fp32 on both sides
and the GEMM accumulates exactly in integers, so the bf16 output has one
correct value.
"""
import numpy as np
import pytest
import torch

from oracle import codecs, int8 as oi8
from fp8_dynamic_quant_gb300 import synth
import fp8_dynamic_quant_gb300 as fq
from _util import bf16_to_dev, bf16_to_np, np_to_dev

pytestmark = pytest.mark.gpu


def gpu_quant(x_bits):
    xq, sx = fq.dynamic_quant_int8(bf16_to_dev(x_bits))
    torch.cuda.synchronize()
    return xq.cpu().numpy(), sx.cpu().numpy()


@pytest.mark.parametrize("M,K", [(1, 4096), (2, 4096), (3, 4096), (4, 4096), (7, 1024), (8, 1024), (9, 4096),
                                 (16, 1024), (32, 4096), (64, 4096), (129, 1024), (5, 16), (3, 4112),
                                 (2, 16400), (300, 64), (1, 2048 * 8 * 4 + 16),
                                 (1216, 4096), (1300, 1024), (2000, 16), (1500, 528),   # warp-per-row path
                                 (1300, 3072), (400, 2064)])  # 128-thread rows, ragged vectors a thread
def test_dynamic_quant_bit_exact(M, K):
    x = synth.activations(M, K, 1000 + M * 7 + K)
    q, s = gpu_quant(x)
    oq, os_ = oi8.dynamic_quant_int8(x)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)


@pytest.mark.parametrize("kernel", ["wide", "row", "ring", "warp", "split"])
@pytest.mark.parametrize("M,K", [(1, 4096), (2, 1024), (3, 4096), (4, 4096), (7, 1024), (8, 4096), (1, 16),
                                 (5, 48), (8, 16384), (6, 2064), (64, 4096), (1300, 1024), (33, 4112),
                                 (2000, 8192), (1217, 16), (999, 2064)])
def test_dynamic_quant_every_kernel(kernel, M, K, monkeypatch):
    """Each quant kernel forced on the same rows (a kernel the shape cannot take
    falls back to the automatic choice): one CTA of up to 1024 threads per row,
    256-thread rows with the next row prefetched, rows staged through a
    shared-memory ring by bulk copies, one warp per row, and the row split along
    K over a cluster (M <= 8)."""
    monkeypatch.setenv("FQ_QUANT_KERNEL", kernel)
    x = synth.activations(M, K, 1500 + M * 5 + K)
    q, s = gpu_quant(x)
    oq, os_ = oi8.dynamic_quant_int8(x)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)
    # the fused op's two-launch path runs the same quant kernel
    if K % 16 == 0 and K <= 4096:
        w = synth.uniform_int8((32, K), 7)
        sw = synth.channel_scales(32, 8)
        y, xq, sx = fq.w8a8_quant_linear(bf16_to_dev(x), np_to_dev(w), np_to_dev(sw), return_quant=True)
        assert np.array_equal(xq.cpu().numpy(), oq) and np.array_equal(sx.cpu().numpy().view(np.uint32),
                                                                       os_.view(np.uint32))
        assert np.array_equal(bf16_to_np(y), oi8.w8a8_linear(oq, os_, w, sw))


def test_dynamic_quant_edge_rows():
    import json, os
    d = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "int8_rows.json")))
    rows = []
    for c in d["cases"]:
        r = np.zeros(16, np.float32)
        r[:len(c["x"])] = c["x"]
        rows.append(r)
    tiny = np.zeros(16, np.float32)
    tiny[:3] = [1e-39, -3e-39, 2e-40]                     # bf16 subnormals
    big = np.zeros(16, np.float32)
    big[:3] = [3.0e38, -1.0e38, 1.0]                       # near the bf16 maximum
    rows += [tiny, big, np.full(16, -7.25, np.float32)]
    x = codecs.f32_to_bf16(np.stack(rows))
    q, s = gpu_quant(x)
    oq, os_ = oi8.dynamic_quant_int8(x)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)
    for i, c in enumerate(d["cases"]):
        assert q[i, :len(c["q"])].tolist() == c["q"] and float(s[i]) == c["s"]


def test_dynamic_quant_near_half_integers():
    """Rows built so that many quotients sit within an ulp of k + 0.5 (the exact-division path)."""
    r = np.random.default_rng(5)
    M, K = 64, 1024
    amax = 127.0 * 1.5
    xs = []
    for m in range(M):
        k = r.integers(-126, 126, K).astype(np.float64) + 0.5
        v = (k * (amax / 127.0)).astype(np.float32)
        v[0] = amax
        xs.append(v)
    x = codecs.f32_to_bf16(np.stack(xs))
    q, s = gpu_quant(x)
    oq, os_ = oi8.dynamic_quant_int8(x)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32)) and np.array_equal(q, oq)


@pytest.mark.parametrize("K", [4096, 2064, 1024])
def test_dynamic_quant_edge_rows_many_rows(K):
    """The many-rows kernels (M above the SM count; 128-thread rows for 2048 < K <= 4096) on zero rows,
    bf16 subnormals, values near the bf16 maximum and quotients at k + 0.5, between ordinary rows."""
    r = np.random.default_rng(17 + K)
    M = 320
    x = r.standard_normal((M, K)).astype(np.float32)
    x[5] = 0.0                                                       # all-zero row: s = 0, q = 0
    x[6] = 0.0
    x[6, :3] = [1e-39, -3e-39, 2e-40]                                # subnormal-only row
    x[7] = r.uniform(-3.0e38, 3.0e38, K).astype(np.float32)         # near the bf16 maximum
    amax = 127.0 * 1.5
    k = r.integers(-126, 126, K).astype(np.float64) + 0.5
    x[8] = (k * (amax / 127.0)).astype(np.float32)                   # quotients at half-integers
    x[8, 0] = amax
    x[M - 1] = -x[M - 1]
    xb = codecs.f32_to_bf16(x)
    q, s = gpu_quant(xb)
    oq, os_ = oi8.dynamic_quant_int8(xb)
    assert np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(q, oq)


def gpu_linear(q, s, w, sw):
    y = fq.w8a8_linear(np_to_dev(q), np_to_dev(s), np_to_dev(w), np_to_dev(sw))
    torch.cuda.synchronize()
    return bf16_to_np(y)


LINEAR_SHAPES = [(4, 4096, 1024)] + [(m, 4096, 1024) for m in (1, 2, 3, 7, 8, 9, 16, 32, 64)] + \
    [(m, 1024, 32768) for m in (1, 2, 3, 4, 7, 8, 9, 16, 32, 64)] + \
    [(65, 1024, 256), (130, 512, 384), (3, 16, 48), (5, 4112, 1040), (1, 4096, 16), (200, 2048, 2048)]


@pytest.mark.parametrize("M,K,N", LINEAR_SHAPES)
def test_w8a8_linear_bit_exact(M, K, N):
    c = synth.int8_linear_case(M, K, N, 2000 + M + K + N)
    q, s = oi8.dynamic_quant_int8(c["x"])
    y = gpu_linear(q, s, c["w_nk"], c["sw"])
    want = oi8.w8a8_linear(q, s, c["w_nk"], c["sw"])
    assert np.array_equal(y, want), np.argwhere(y != want)[:5]


@pytest.mark.parametrize("sched", ["dp", "cluster", "streamk", "umma"])
@pytest.mark.parametrize("M,K,N", [(1, 1024, 4096), (8, 4096, 1024), (9, 2048, 2240), (16, 1024, 32768),
                                   (3, 4112, 1040), (5, 512, 48), (32, 4096, 1024), (64, 1024, 32768),
                                   (50, 3968, 2064), (64, 16, 128), (40, 1024, 128)])
def test_every_schedule_bit_exact(sched, M, K, N, monkeypatch):
    # the host picks one of three schedules by shape; forcing each on the same
    # problems checks that all three give the one correct answer
    monkeypatch.setenv("FQ_FORCE_SCHEDULE", sched)
    c = synth.int8_linear_case(M, K, N, 4000 + M + K + N)
    q, s = oi8.dynamic_quant_int8(c["x"])
    assert np.array_equal(gpu_linear(q, s, c["w_nk"], c["sw"]), oi8.w8a8_linear(q, s, c["w_nk"], c["sw"]))


def test_w8a8_linear_accumulator_extremes():
    """|acc| up to 127*127*K with K = 131072 (the int32 limit) and mixed signs."""
    K, N = 131072, 32
    q = np.full((3, K), 127, np.int8)
    q[1] = -127
    q[2, ::2] = -127
    w = np.full((N, K), 127, np.int8)
    w[1::2] = -127
    s = np.array([1e-3, 2e-3, 3e-3], np.float32)
    sw = np.linspace(1e-4, 1e-3, N).astype(np.float32)
    y = gpu_linear(q, s, w, sw)
    assert np.array_equal(y, oi8.w8a8_linear(q, s, w, sw))


@pytest.mark.parametrize("M,K,N", [(4, 4096, 1024), (1, 1024, 32768), (64, 1024, 32768), (9, 4096, 1024),
                                   (33, 256, 128)])
def test_fused_quant_linear_equals_two_steps(M, K, N):
    c = synth.int8_linear_case(M, K, N, 3000 + M)
    x = bf16_to_dev(c["x"])
    w, sw = np_to_dev(c["w_nk"]), np_to_dev(c["sw"])
    y, xq, sx = fq.w8a8_quant_linear(x, w, sw, return_quant=True)
    y_plain = fq.w8a8_quant_linear(x, w, sw)
    xq2, sx2 = fq.dynamic_quant_int8(x)
    y2 = fq.w8a8_linear(xq2, sx2, w, sw)
    torch.cuda.synchronize()
    assert torch.equal(xq, xq2) and torch.equal(sx, sx2)
    assert torch.equal(y.view(torch.int16), y2.view(torch.int16))
    assert torch.equal(y_plain.view(torch.int16), y2.view(torch.int16))
    want, oq, os_ = oi8.w8a8_quant_linear(c["x"], c["w_nk"], c["sw"])
    assert np.array_equal(bf16_to_np(y), want)


# (M, K, N) where the dense schedule streams one whole 224-row tile per CTA
# (114..148 tiles) with M <= 8 and K <= 1024: the fused op is one launch in
# which every CTA quantizes the activations itself.  Ragged K (1008, 144, 16)
# and N.
FUSED_ONE_LAUNCH = [(1, 1024, 32768), (2, 1024, 32768), (3, 1024, 25600), (7, 1008, 30000), (8, 1024, 33152),
                    (6, 512, 29008), (8, 1024, 32768), (5, 16, 26000), (4, 144, 33008),
                    # 16-token tiles, one row per consumer warp
                    (9, 1024, 32768), (14, 1024, 32768), (12, 1008, 30000), (10, 512, 29008), (13, 16, 26000),
                    (11, 144, 33008)]


def _fused_one_launch(x, w_nk, sw):
    xd, w, s = bf16_to_dev(x), np_to_dev(w_nk), np_to_dev(sw)
    y, xq, sx = fq.w8a8_quant_linear(xd, w, s, return_quant=True)
    y_plain = fq.w8a8_quant_linear(xd, w, s)
    torch.cuda.synchronize()
    return bf16_to_np(y), bf16_to_np(y_plain), xq.cpu().numpy(), sx.cpu().numpy()


@pytest.mark.parametrize("M,K,N", FUSED_ONE_LAUNCH)
def test_fused_one_launch_bit_exact(M, K, N, monkeypatch, capfd):
    """y, xq and sx of the one-launch fused op equal the oracle bit for bit (a zero row included)."""
    monkeypatch.setenv("FQ_DEBUG_SCHEDULE", "1")
    c = synth.int8_linear_case(M, K, N, 5000 + M + K + N)
    x = c["x"].copy()
    if M >= 3:
        x[M - 1, :] = 0  # all-zero row: scale 0, codes 0
    y, y_plain, q, s = _fused_one_launch(x, c["w_nk"], c["sw"])
    assert "schedule=dp224+quant" in capfd.readouterr().err
    want, oq, os_ = oi8.w8a8_quant_linear(x, c["w_nk"], c["sw"])
    assert np.array_equal(q, oq) and np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(y, want), np.argwhere(y != want)[:5]
    assert np.array_equal(y_plain, want)


@pytest.mark.parametrize("M", [1, 3, 8, 14])
def test_fused_one_launch_forced_small_n_and_ties(M, monkeypatch, capfd):
    """Forced data-parallel schedule on a small N, and rows whose quotients sit at k + 0.5."""
    monkeypatch.setenv("FQ_DEBUG_SCHEDULE", "1")
    monkeypatch.setenv("FQ_FORCE_SCHEDULE", "dp")
    r = np.random.default_rng(11 + M)
    K, N = 1024, 2240
    amax = 127.0 * 1.5
    rows = []
    for m in range(M):
        v = ((r.integers(-126, 126, K).astype(np.float64) + 0.5) * (amax / 127.0)).astype(np.float32)
        v[m] = amax
        rows.append(v)
    x = codecs.f32_to_bf16(np.stack(rows))
    w_nk = synth.int8_weights(N, K, 77)
    sw = synth.channel_scales(N, 78)
    y, y_plain, q, s = _fused_one_launch(x, w_nk, sw)
    assert "schedule=dp224+quant" in capfd.readouterr().err
    want, oq, os_ = oi8.w8a8_quant_linear(x, w_nk, sw)
    assert np.array_equal(q, oq) and np.array_equal(s.view(np.uint32), os_.view(np.uint32))
    assert np.array_equal(y, want) and np.array_equal(y_plain, want)


@pytest.mark.parametrize("K,N", [(1024, 8192), (1024, 32768), (4096, 1024)])
def test_linear_right_after_weight_quant(K, N):
    """Per-channel weight quant (dynamic_quant_int8 on W's rows) launched right before the linear with
    nothing else on the stream in between: the linear streams its weights before it waits on the
    previous kernel, so the weight quant must let it start only once it has finished."""
    dev = torch.device("cuda")
    M = 4
    x = synth.activations(M, K, 91)
    q, s = oi8.dynamic_quant_int8(x)
    qd, sd = np_to_dev(q), np_to_dev(s)
    wq = torch.empty(N, K, dtype=torch.int8, device=dev)
    swq = torch.empty(N, dtype=torch.float32, device=dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = fq.new_workspace(fq.workspace_bytes(fq.OP_W8A8_LINEAR, M, K, N), dev)
    for i in range(3):
        wf = synth.activations(N, K, 900 + i + N)
        wd = bf16_to_dev(wf)
        torch.cuda.synchronize()
        fq.dynamic_quant_int8(wd, wq, swq)
        fq.w8a8_linear(qd, sd, wq, swq, y=y, ws=ws)
        torch.cuda.synchronize()
        oq, os_ = oi8.dynamic_quant_int8(wf)
        assert np.array_equal(bf16_to_np(y), oi8.w8a8_linear(q, s, oq, os_))


def test_workspace_counters_return_to_zero():
    c = synth.int8_linear_case(9, 4096, 1024, 11)
    q, s = oi8.dynamic_quant_int8(c["x"])
    gpu_linear(q, s, c["w_nk"], c["sw"])
    dev = torch.device("cuda")
    key = (dev.index if dev.index is not None else torch.cuda.current_device(), torch.cuda.current_stream().cuda_stream)
    ws = fq._WS[key]
    # the fixed counter block at the head of every workspace (256 KiB)
    assert int(ws[: 65536 * 4].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("M,K,N", [(7, 1024, 32768), (4, 4096, 1024), (1, 4096, 1024), (64, 1024, 32768)])
def test_repeated_calls_stay_exact(M, K, N):
    """Twelve back-to-back calls are all bit-exact (stage hand-back race guard)."""
    c = synth.int8_linear_case(M, K, N, 12)
    q, s = oi8.dynamic_quant_int8(c["x"])
    want = oi8.w8a8_linear(q, s, c["w_nk"], c["sw"])
    qd, sd, wd, swd = np_to_dev(q), np_to_dev(s), np_to_dev(c["w_nk"]), np_to_dev(c["sw"])
    ys = [fq.w8a8_linear(qd, sd, wd, swd) for _ in range(12)]
    torch.cuda.synchronize()
    for y in ys:
        assert np.array_equal(bf16_to_np(y), want)


def test_device_error_word_clean_after_valid_calls():
    st, word = fq.device_error()
    assert st == 0 and word == 0


def test_one_workspace_shared_by_different_ops_and_shapes():
    """Split-K scratch of one call must never corrupt the arrival counters of the next:
    an einsum (fp32 partials), a fused linear (quantized activations in the workspace)
    and linears with 8 and 256 tiles run back to back on the same workspace."""
    from oracle import fp8 as of8
    T, G, D, N = 100, 3, 640, 384
    x8 = synth.group_activations(T, G, D, 5)
    w8 = synth.fp8_einsum_weights(G, N, D, 6)
    wq, sw8 = fq.quantize_weight_fp8_block(np_to_dev(w8))
    xq8, st = fq.quant_fp8_group_ue8m0_packed(bf16_to_dev(x8))
    cases = [synth.int8_linear_case(m, k, n, 50 + m) for m, k, n in [(7, 1024, 32768), (4, 4096, 1024), (64, 1024, 32768)]]
    for rep in range(2):
        fq.fp8_group_einsum(xq8, st, fq.SCALE_UE8M0_PACKED, wq, sw8)
        for c in cases:
            fq.w8a8_quant_linear(bf16_to_dev(c["x"]), np_to_dev(c["w_nk"]), np_to_dev(c["sw"]))
            q, s = oi8.dynamic_quant_int8(c["x"])
            y = gpu_linear(q, s, c["w_nk"], c["sw"])
            assert np.array_equal(y, oi8.w8a8_linear(q, s, c["w_nk"], c["sw"]))
