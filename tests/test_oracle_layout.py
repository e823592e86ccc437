"""Pins for the K-major weight repack: hand-placed elements and the linear it feeds."""
import numpy as np

from oracle import int8, layout


def test_repack_places_each_element_by_hand():
    # W[k, n] = 10 * k + n for K = 3, N = 4: stored row n holds (n, 10 + n, 20 + n)
    w = (10 * np.arange(3)[:, None] + np.arange(4)[None, :]).astype(np.int8)
    out = layout.repack_weight_kmajor(w)
    assert out.shape == (4, 3)
    assert out.tolist() == [[0, 10, 20], [1, 11, 21], [2, 12, 22], [3, 13, 23]]
    flat = out.ravel()
    K = 3
    for k in range(3):
        for n in range(4):
            assert flat[n * K + k] == w[k, n]


def test_repack_batched_matrices_are_independent():
    w = np.arange(2 * 2 * 3, dtype=np.int64).reshape(2, 2, 3).astype(np.int8)
    out = layout.repack_weight_kmajor(w)
    assert out.shape == (2, 3, 2)
    assert out[1].tolist() == [[6, 9], [7, 10], [8, 11]]


def test_repacked_weight_gives_the_logical_product():
    """y = x W on the logical weight equals the oracle linear on the repacked one
    (an exact integer case: unit scales, small values)."""
    r = np.random.default_rng(3)
    K, N = 32, 16
    w = r.integers(-3, 4, (K, N)).astype(np.int8)
    q = r.integers(-3, 4, (2, K)).astype(np.int8)
    acc = q.astype(np.int64) @ w.astype(np.int64)
    y = int8.w8a8_linear(q, np.ones(2, np.float32), layout.repack_weight_kmajor(w), np.ones(N, np.float32))
    from oracle.codecs import bf16_to_f32
    assert np.array_equal(bf16_to_f32(y), acc.astype(np.float32))
