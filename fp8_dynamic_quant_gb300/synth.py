"""Seeded synthetic inputs for the decode quant + quantized-linear path.

This module only draws random inputs with the shapes and value
distributions of the workloads; it holds none of the path's arithmetic.
Both the CPU oracle (in tests) and the CUDA path (tests, bench) take their
inputs from here.  Every generator is a pure function of its seed.

Workloads (sizes from the pages' DeepSeek-V4 shapes):
  * INT8 linear: X bf16 [M, K] ~ N(0, 1), each entry independently an
    outlier with probability 0.001 and then multiplied by 50; W int8 [N, K]
    uniform on [-127, 127]; per-channel weight scale fp32 U[1e-3, 1e-2].
  * FP8 group quant: x bf16 [T, G, D] ~ N(0, 1) times a per-(t, g) row
    magnitude 10**U[-3, 3].
  * FP8 einsum weights: W fp32 [G, N, D] ~ N(0, 0.02) (logical [G, D, N]).
  * MoE: topk_ids from a Zipf(s=1.1) law over experts (rank r -> expert
    r - 1), duplicates within a token redrawn; topk weights = softmax of
    N(0, 1) logits; W13 int8 [E, 2I, H], W2 int8 [E, H, I], scales as above.
"""
import numpy as np
import torch

SEED_BASE = 0x5EED0000


def rng(seed):
    return np.random.Generator(np.random.PCG64(int(seed)))


def to_bf16_bits(x_f32):
    """float32 array -> bf16 bit patterns via torch's own conversion."""
    t = torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def activations(M, K, seed, outlier_p=0.001, outlier_mul=50.0):
    r = rng(seed)
    x = r.standard_normal((M, K), dtype=np.float32)
    mask = r.random((M, K)) < outlier_p
    x = np.where(mask, x * np.float32(outlier_mul), x).astype(np.float32)
    return to_bf16_bits(x)


def uniform_int8(shape, seed):
    """int8 uniform on [-127, 127] (host)."""
    return rng(seed).integers(-127, 128, size=shape, dtype=np.int8)


def uniform_int8_device(shape, seed, device):
    """int8 uniform on [-127, 127], drawn by torch's seeded generator on `device`.

    Used for multi-GB expert weights; tests hand host copies of the slices
    they check to the oracle.
    """
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.randint(-127, 128, tuple(shape), generator=g, dtype=torch.int8, device=device)


def uniform_f32_device(shape, lo, hi, seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return torch.rand(tuple(shape), generator=g, dtype=torch.float32, device=device) * (hi - lo) + lo


def int8_weights(N, K, seed):
    return uniform_int8((N, K), seed)


def channel_scales(N, seed, lo=1e-3, hi=1e-2):
    return rng(seed).uniform(lo, hi, size=N).astype(np.float32)


def int8_linear_case(M, K, N, seed):
    """Dict(x bf16 [M,K], w_nk int8 [N,K], sw fp32 [N]) for the INT8 linear."""
    return dict(x=activations(M, K, seed), w_nk=int8_weights(N, K, seed + 1),
                sw=channel_scales(N, seed + 2))


def group_activations(T, G, D, seed):
    """x bf16 [T, G, D] ~ N(0,1) * 10**U[-3,3] per (t, g) row."""
    r = rng(seed)
    x = r.standard_normal((T, G, D), dtype=np.float32)
    mag = (10.0 ** r.uniform(-3.0, 3.0, size=(T, G, 1))).astype(np.float32)
    return to_bf16_bits((x * mag).astype(np.float32))


def fp8_einsum_weights(G, N, D, seed, std=0.02):
    """fp32 W stored [G, N, D] (K-major), logical W[g, d, n] = w[g, n, d]."""
    return (rng(seed).standard_normal((G, N, D), dtype=np.float32) * np.float32(std))


def zipf_topk(T, topk, E, seed, s=1.1):
    """topk_ids int32 [T, topk], distinct per token, rank r ~ r**-s over 1..E."""
    r = rng(seed)
    p = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    cdf = np.cumsum(p / p.sum())
    ids = np.empty((T, topk), np.int32)
    for t in range(T):
        chosen = []
        while len(chosen) < topk:
            e = int(np.searchsorted(cdf, r.random(), side="right"))
            e = min(e, E - 1)
            if e not in chosen:
                chosen.append(e)
        ids[t] = chosen
    return ids


def topk_weights(T, topk, seed):
    z = rng(seed).standard_normal((T, topk))
    z = np.exp(z - z.max(axis=1, keepdims=True))
    return (z / z.sum(axis=1, keepdims=True)).astype(np.float32)


def moe_case(T, topk, E, H, I, seed, with_weights=True):
    """Decode MoE batch: tokens, routing, and (host) expert weights."""
    c = dict(x=activations(T, H, seed), topk_ids=zipf_topk(T, topk, E, seed + 1),
             topk_w=topk_weights(T, topk, seed + 2))
    if with_weights:
        c.update(w13=uniform_int8((E, 2 * I, H), seed + 3),
                 sw13=rng(seed + 4).uniform(1e-3, 1e-2, size=(E, 2 * I)).astype(np.float32),
                 w2=uniform_int8((E, H, I), seed + 5),
                 sw2=rng(seed + 6).uniform(1e-3, 1e-2, size=(E, H)).astype(np.float32))
    return c


def moe_weights_device(E, H, I, seed, device):
    """Expert weights on the device: W13 int8 [E, 2I, H], sw13 [E, 2I], W2 int8 [E, H, I], sw2 [E, H]."""
    return dict(w13=uniform_int8_device((E, 2 * I, H), seed + 3, device),
                sw13=uniform_f32_device((E, 2 * I), 1e-3, 1e-2, seed + 4, device),
                w2=uniform_int8_device((E, H, I), seed + 5, device),
                sw2=uniform_f32_device((E, H), 1e-3, 1e-2, seed + 6, device))
