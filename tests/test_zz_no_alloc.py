"""w8a8_linear_noalloc: the W8A8 linear for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (an allocator-free runtime, a plugin that
must not touch its host's memory pool), so they cannot supply the workspace
that w8a8_linear takes.  This entry point keeps its split-K scratch in a fixed
device array inside the library instead.  Its output must be bit-identical to
w8a8_linear and to the oracle - the same tolerance (exact) the other INT8 GEMM
tests use - on two calls in a row, since the shared array keeps the previous
call's contents.  The cases cover every kernel that uses the array (the
mma.sync stream-K kernel with 8-, 16- and 64-token tiles and the tcgen05
stream-K kernel) as well as the schedules that do not (224-row tiles, 4-CTA
clusters); the schedule each call took is read back from FQ_DEBUG_SCHEDULE.
Collected last, so a failure here leaves every other test already run.
"""
import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _noalloc(xq, sx, w, sw, y):
    import fp8_dynamic_quant_gb300 as fq
    M, K = xq.shape
    N = w.shape[0]
    return fq.lib().w8a8_linear_noalloc(ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(sx.data_ptr()), M, K,
                                        ctypes.c_void_p(w.data_ptr()), ctypes.c_void_p(sw.data_ptr()), N,
                                        ctypes.c_void_p(y.data_ptr()), fq._stream())


# (M, K, N, forced schedule or None, schedule the call must report)
CASES = [
    (4, 4096, 1024, None, "cluster4"),
    (9, 4096, 1040, None, "cluster4"),
    (4, 1024, 32768, None, "dp224"),
    (4, 4096, 4096, None, "streamk"),        # mma.sync stream-K, 8-token tiles: uses the array
    (16, 4096, 4096, None, "streamk"),       # mma.sync stream-K, 16-token tiles
    (64, 1024, 32768, None, "umma"),         # tcgen05 stream-K, 64-token tiles
    (64, 4096, 4096, "streamk", "streamk"),  # mma.sync stream-K with the largest slots (64 tokens)
    (8, 2048, 2048, "umma", "umma"),         # tcgen05 stream-K with a short token tile
]


@pytest.mark.parametrize("M,K,N,force,sched", CASES)
def test_noalloc_matches_w8a8_linear_and_oracle_twice(M, K, N, force, sched, monkeypatch, capfd):
    import fp8_dynamic_quant_gb300 as fq
    from fp8_dynamic_quant_gb300 import synth
    from oracle import int8 as oi8
    c = synth.int8_linear_case(M, K, N, 9000 + M + N)
    dev = torch.device("cuda")
    x = torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(c["w_nk"]).to(dev)
    sw = torch.from_numpy(c["sw"]).to(dev)
    if force:
        monkeypatch.setenv("FQ_FORCE_SCHEDULE", force)
    xq, sx = fq.dynamic_quant_int8(x)
    want = fq.w8a8_linear(xq, sx, w, sw)
    q, s = oi8.dynamic_quant_int8(c["x"])
    oracle_y = oi8.w8a8_linear(q, s, c["w_nk"], c["sw"])
    monkeypatch.setenv("FQ_DEBUG_SCHEDULE", "1")
    capfd.readouterr()
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _noalloc(xq, sx, w, sw, y) == 0
        torch.cuda.synchronize()
        got = y.view(torch.int16)
        assert torch.equal(got, want.view(torch.int16))
        assert np.array_equal(got.cpu().numpy().view(np.uint16), oracle_y)
    err = capfd.readouterr().err
    lines = [l for l in err.splitlines() if l.startswith("fq: ")]
    assert len(lines) == 2 and all(("schedule=%s " % sched) in l for l in lines), err


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import fp8_dynamic_quant_gb300 as fq
    dev = torch.device("cuda")
    xq = torch.zeros((65, 128), dtype=torch.int8, device=dev)
    sx = torch.zeros((65,), dtype=torch.float32, device=dev)
    w = torch.zeros((128, 128), dtype=torch.int8, device=dev)
    sw = torch.zeros((128,), dtype=torch.float32, device=dev)
    y = torch.zeros((65, 128), dtype=torch.bfloat16, device=dev)
    assert _noalloc(xq, sx, w, sw, y) == 2                     # M = 65 > 64: FQ_ERR_SHAPE
    # N = 524416: ceil(N / 128) = 4097 tiles > 4096 arrival counters.  The
    # sizes are checked before anything is read, so small buffers suffice.
    L = fq.lib()
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert L.w8a8_linear_noalloc(p(xq), p(sx), 4, 128, p(w), p(sw), 524416, p(y), fq._stream()) == 2
