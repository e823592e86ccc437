"""w8a8_linear_noalloc: the W8A8 linear for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (an allocator-free runtime, a plugin that
must not touch its host's memory pool), so they cannot supply the workspace
that w8a8_linear takes.  This entry point keeps its split-K scratch in a fixed
device array inside the library instead.  Its output must be bit-identical to
w8a8_linear - the same tolerance (exact) the other INT8 GEMM tests use - on
two calls in a row, since the shared array keeps the previous call's contents.
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


@pytest.mark.parametrize("M,K,N", [(4, 4096, 1024), (64, 1024, 32768), (9, 4096, 1040)])
def test_noalloc_matches_w8a8_linear_twice(M, K, N):
    import fp8_dynamic_quant_gb300 as fq
    from fp8_dynamic_quant_gb300 import synth
    c = synth.int8_linear_case(M, K, N, 9000 + M)
    dev = torch.device("cuda")
    x = torch.from_numpy(c["x"].view(np.int16)).view(torch.bfloat16).to(dev)
    w = torch.from_numpy(c["w_nk"]).to(dev)
    sw = torch.from_numpy(c["sw"]).to(dev)
    xq, sx = fq.dynamic_quant_int8(x)
    want = fq.w8a8_linear(xq, sx, w, sw)
    for _ in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _noalloc(xq, sx, w, sw, y) == 0
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), want.view(torch.int16))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import fp8_dynamic_quant_gb300 as fq
    dev = torch.device("cuda")
    xq = torch.zeros((65, 128), dtype=torch.int8, device=dev)
    sx = torch.zeros((65,), dtype=torch.float32, device=dev)
    w = torch.zeros((128, 128), dtype=torch.int8, device=dev)
    sw = torch.zeros((128,), dtype=torch.float32, device=dev)
    y = torch.zeros((65, 128), dtype=torch.bfloat16, device=dev)
    assert _noalloc(xq, sx, w, sw, y) == 2                     # M = 65 > 64: FQ_ERR_SHAPE
