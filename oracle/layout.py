"""Load-time weight layout, written from its definition.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[W8A8] section 4: weights are cast once at load time to the layout the
matmul reads best.  The layout here is K-major: a logical weight W[k, n]
(row-major [K, N], or [B, K, N] for B stacked matrices) is stored as
w_nk[n, k], i.e. at flat offset n * K + k of its matrix.
"""
import numpy as np


def repack_weight_kmajor(w_bkn):
    """Logical [K, N] / [B, K, N] -> stored [N, K] / [B, N, K], element by element:
    out[b, n, k] = w[b, k, n]."""
    w = np.asarray(w_bkn)
    squeeze = w.ndim == 2
    w3 = w[None] if squeeze else w
    B, K, N = w3.shape
    out = np.empty((B, N, K), w.dtype)
    for b in range(B):
        for k in range(K):
            out[b, :, k] = w3[b, k, :]           # row k of W becomes column k of the stored matrix
    return out[0] if squeeze else out
