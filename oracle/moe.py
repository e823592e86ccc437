"""MoE expert path on the W8A8 mode, written from definitions.

TEST INFRASTRUCTURE ONLY (see the package docstring).

[DF] section 3.2: sort tokens by expert id before dispatch so that each
expert's rows are contiguous, then gather.  [W8A8] section 5: the grouped
matmul takes group_list = expert_tokens (expert-local row counts M_e).
[DF] section 2.3: SwiGLU fused with quantization.  [W8A8] section 1: the
layer budget includes the combine.

Readings for silent points:
  * sort key (expert, token, slot): a stable sort of the flattened
    [T, topk] ids; offsets are the exclusive scan of per-expert counts;
  * rows are quantized per token before the gather (per-token quant makes
    this identical to quantizing the gathered copies);
  * gate/up layout: the first I columns of the W13 output are the gate g,
    the last I the up projection u;
  * h = bf16_RN(fp32(s * u)) with s = fp32_RN(silu(g)), silu(g) =
    g / (1 + exp(-g)): the exact value rounded once to fp32, evaluated as the
    float64 quotient rounded once to fp32 (for every bf16 g the two agree; a
    test checks all 65536 values against a 200-bit evaluation); then the INT8
    per-token quant of h;
  * combine: out[t] = bf16_RN(sum over slots j = 0..topk-1, in slot order,
    of fp32(w[t, j] * y[row(t, j)])), an fp32 running sum.
"""
import numpy as np

from .codecs import bf16_to_f32, f32_to_bf16
from .int8 import dynamic_quant_int8, w8a8_linear


def moe_sort(topk_ids, E):
    """Stable sort of the flattened (token, slot) pairs by expert id.

    Returns (offsets int32 [E + 1], perm int32 [T * topk]); perm[i] is the
    flat pair index t * topk + j of the i-th pair in expert order.
    """
    ids = np.asarray(topk_ids, np.int64).reshape(-1)
    if ids.size and (ids.min() < 0 or ids.max() >= E):
        raise ValueError("expert id out of range")
    perm = np.argsort(ids, kind="stable")
    counts = np.bincount(ids, minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)])
    return offsets.astype(np.int32), perm.astype(np.int32)


def gather_rows(rows, perm, topk):
    """Rows of the sorted list: row i is source token perm[i] // topk."""
    return np.asarray(rows)[np.asarray(perm, np.int64) // topk]


def w8a8_grouped_linear(q, s, offsets, w_enk, sw_en):
    """Per-expert W8A8 linear over contiguous row ranges; empty experts skipped.

    q int8 [R, K], s fp32 [R], offsets [E + 1], w_enk int8 [E, N, K],
    sw_en fp32 [E, N] -> Y bf16 bits [R, N].
    """
    R = q.shape[0]
    E, N, _ = w_enk.shape
    y = np.zeros((R, N), np.uint16)
    for e in range(E):
        a, b = int(offsets[e]), int(offsets[e + 1])
        if b > a:
            y[a:b] = w8a8_linear(q[a:b], s[a:b], w_enk[e], sw_en[e])
    return y


def silu_f32(g):
    """s = fp32_RN(g / (1 + exp(-g))) for fp32 (bf16-valued) g, via the float64 quotient."""
    g = np.asarray(g, np.float32).astype(np.float64)
    with np.errstate(over="ignore"):                    # exp(-g) = inf for g < -709: silu -> -0
        return (g / (1.0 + np.exp(-g))).astype(np.float32)


def swiglu_bf16(gu_bf16):
    """h = bf16_RN(fp32(silu(g)) * u), g = first half of the columns, u = second."""
    gu = bf16_to_f32(np.asarray(gu_bf16, np.uint16))
    I = gu.shape[1] // 2
    silu = silu_f32(gu[:, :I])
    u = gu[:, I:]
    return f32_to_bf16((silu * u).astype(np.float32))


def swiglu_quant_int8(gu_bf16):
    """SwiGLU then per-token INT8 quant.  Returns (hq, sh, h_bf16)."""
    h = swiglu_bf16(gu_bf16)
    hq, sh = dynamic_quant_int8(h)
    return hq, sh, h


def moe_combine(y_rows_bf16, perm, topk_w, T, topk):
    """out[t] = bf16( fp32 running sum over slots j of fp32(w[t,j] * y[row(t,j)]) )."""
    y = bf16_to_f32(np.asarray(y_rows_bf16, np.uint16))
    perm = np.asarray(perm, np.int64)
    inv = np.empty_like(perm)
    inv[perm] = np.arange(perm.size)
    w = np.asarray(topk_w, np.float32)
    H = y.shape[1]
    acc = np.zeros((T, H), np.float32)
    for j in range(topk):
        rows = inv[np.arange(T) * topk + j]
        acc = (acc + (w[:, j][:, None] * y[rows]).astype(np.float32)).astype(np.float32)
    return f32_to_bf16(acc)


def moe_forward(x_bf16, topk_ids, topk_w, w13, sw13, w2, sw2):
    """Whole expert path: quant -> sort -> gather -> W13 -> SwiGLU+quant -> W2 -> combine.

    Returns a dict with every intermediate so tests can compare each step.
    """
    T, topk = np.asarray(topk_ids).shape
    E = w13.shape[0]
    q, s = dynamic_quant_int8(x_bf16)
    offsets, perm = moe_sort(topk_ids, E)
    qg = gather_rows(q, perm, topk)
    sg = gather_rows(s, perm, topk)
    y1 = w8a8_grouped_linear(qg, sg, offsets, w13, sw13)
    hq, sh, h = swiglu_quant_int8(y1)
    y2 = w8a8_grouped_linear(hq, sh, offsets, w2, sw2)
    out = moe_combine(y2, perm, topk_w, T, topk)
    return dict(q=q, s=s, offsets=offsets, perm=perm, y1=y1, h=h, hq=hq, sh=sh, y2=y2, out=out)
