"""GPU parity of the load-time K-major weight repack (through the C ABI)."""
import numpy as np
import pytest
import torch

import fp8_dynamic_quant_gb300 as fq
from fp8_dynamic_quant_gb300 import synth
from oracle import fp8 as of8, int8 as oi8, layout
from _util import bf16_to_np, np_to_dev, e4m3_to_dev, e4m3_to_np

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B,K,N", [(1, 16, 16), (1, 48, 80), (1, 4096, 1024), (3, 208, 144), (2, 1024, 64)])
def test_repack_i8_matches_oracle(B, K, N):
    w = synth.uniform_int8((B, K, N), 40 + K + N)
    got = fq.repack_weight_kmajor_i8(np_to_dev(w))
    assert np.array_equal(got.cpu().numpy(), layout.repack_weight_kmajor(w))


@pytest.mark.parametrize("G,D,N", [(1, 128, 128), (8, 512, 256), (2, 384, 640)])
def test_repack_fp8_matches_oracle(G, D, N):
    codes = synth.rng(50 + D).integers(0, 256, (G, D, N)).astype(np.uint8)
    got = fq.repack_weight_kmajor_fp8(e4m3_to_dev(codes))
    assert np.array_equal(e4m3_to_np(got), layout.repack_weight_kmajor(codes))


def test_repack_then_linear_is_the_logical_linear():
    """Logical W [K, N] -> repack -> w8a8_linear equals the oracle's linear on the logical weight."""
    M, K, N = 4, 4096, 1024
    c = synth.int8_linear_case(M, K, N, 61)
    w_kn = np.ascontiguousarray(c["w_nk"].T)                 # the logical [K, N] weight
    q, s = oi8.dynamic_quant_int8(c["x"])
    w_nk = fq.repack_weight_kmajor_i8(np_to_dev(w_kn))
    y = fq.w8a8_linear(np_to_dev(q), np_to_dev(s), w_nk, np_to_dev(c["sw"]))
    assert np.array_equal(bf16_to_np(y), oi8.w8a8_linear(q, s, c["w_nk"], c["sw"]))


def test_repack_rejects_in_place():
    w = torch.zeros((64, 64), dtype=torch.int8, device="cuda")
    with pytest.raises(fq.FqError) as e:
        fq.repack_weight_kmajor_i8(w, out=w)
    assert e.value.status == 9
