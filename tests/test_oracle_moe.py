"""Pins for the MoE oracle: histogram, reduction to the dense chain, relabelling invariance."""
import json
import os

import numpy as np

from oracle import codecs, int8, moe
from fp8_dynamic_quant_gb300 import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def test_sort_offsets_histogram_and_stability():
    ids = synth.zipf_topk(64, 8, 32, 3)
    off, perm = moe.moe_sort(ids, 32)
    assert np.array_equal(np.diff(off), np.bincount(ids.ravel(), minlength=32))
    assert sorted(perm.tolist()) == list(range(ids.size))
    flat = ids.ravel()
    for e in range(32):
        seg = perm[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e) and np.all(np.diff(seg) > 0)   # stable: ascending pair index


def test_zipf_ids_distinct_per_token():
    ids = synth.zipf_topk(256, 8, 256, 5)
    assert all(len(set(r)) == 8 for r in ids.tolist())


def test_swiglu_golden():
    d = json.load(open(os.path.join(GOLD, "swiglu.json")))
    g = np.array([c["g"] for c in d["cases"]], np.float32)
    u = np.array([c["u"] for c in d["cases"]], np.float32)
    gu = codecs.f32_to_bf16(np.stack([g, u], axis=1))                  # I = 1
    h = codecs.bf16_to_f32(moe.swiglu_bf16(gu))[:, 0]
    assert h.tolist() == [c["h"] for c in d["cases"]]


def small_case(T=16, topk=4, E=8, H=128, I=64, seed=1):
    return synth.moe_case(T, topk, E, H, I, seed)


def test_single_expert_top1_reduces_to_dense_chain():
    c = small_case(T=8, topk=1, E=1)
    ids = np.zeros((8, 1), np.int32)
    w = np.ones((8, 1), np.float32)
    r = moe.moe_forward(c["x"], ids, w, c["w13"], c["sw13"], c["w2"], c["sw2"])
    q, s = int8.dynamic_quant_int8(c["x"])
    y1 = int8.w8a8_linear(q, s, c["w13"][0], c["sw13"][0])
    hq, sh, _ = moe.swiglu_quant_int8(y1)
    y2 = int8.w8a8_linear(hq, sh, c["w2"][0], c["sw2"][0])
    assert np.array_equal(r["out"], y2)                      # 1.0 * y exactly


def test_expert_relabelling_invariance():
    c = small_case()
    base = moe.moe_forward(c["x"], c["topk_ids"], c["topk_w"], c["w13"], c["sw13"], c["w2"], c["sw2"])
    p = np.random.default_rng(0).permutation(8)                 # new label of old expert e is p[e]
    inv = np.argsort(p)
    r = moe.moe_forward(c["x"], p[c["topk_ids"]].astype(np.int32), c["topk_w"],
                        c["w13"][inv], c["sw13"][inv], c["w2"][inv], c["sw2"][inv])
    assert np.array_equal(base["out"], r["out"])


def test_combine_closed_form():
    T, topk, H = 2, 2, 4
    y = codecs.f32_to_bf16(np.array([[1, 2, 3, 4], [10, 20, 30, 40], [-1, -1, -1, -1], [0.5, 0.5, 0.5, 0.5]], np.float32))
    perm = np.array([3, 0, 2, 1], np.int32)     # sorted row i holds pair perm[i]
    w = np.array([[0.5, 0.25], [2.0, 1.0]], np.float32)
    out = codecs.bf16_to_f32(moe.moe_combine(y, perm, w, T, topk))
    # pair 0 -> row 1, pair 1 -> row 3, pair 2 -> row 2, pair 3 -> row 0
    assert out.tolist() == [[0.5 * 10 + 0.25 * 0.5] * 0 + [5.125, 10.125, 15.125, 20.125],
                            [-2 + 1, -2 + 2, -2 + 3, -2 + 4]]


def _correctly_rounded_silu_f32(g_values):
    """fp32 bit patterns of silu(g) = g / (1 + exp(-g)) evaluated with 200-bit
    arithmetic and rounded once to fp32 (subnormals included, ties to even)."""
    mpmath = __import__("pytest").importorskip("mpmath")
    out = np.empty(len(g_values), np.uint32)
    with mpmath.workprec(200):
        for i, g in enumerate(g_values):
            g = float(g)
            sign = 0x80000000 if np.signbit(np.float32(g)) else 0
            if g == 0.0:
                out[i] = sign
                continue
            gm = mpmath.mpf(g)
            s = abs(gm / (1 + mpmath.exp(-gm)))
            e = int(mpmath.floor(mpmath.log(s, 2))) if s > 0 else -200
            ulp = mpmath.mpf(2) ** max(e - 23, -149)
            q = s / ulp
            n = int(mpmath.floor(q))
            frac = q - n
            if frac > 0.5 or (frac == 0.5 and n % 2 == 1):
                n += 1
            mag = np.float32(float(n * ulp))       # n * ulp has <= 25 significant bits: exact
            out[i] = np.uint32(mag.view(np.uint32)) | sign
    return out


def test_silu_f32_is_the_correctly_rounded_silu_for_every_bf16():
    """The oracle's float64 quotient rounded to fp32 equals the exact silu
    rounded once to fp32 for every finite bf16 input (infinities and NaN are
    outside the contract: the gate is a finite GEMM output)."""
    bits = np.arange(65536, dtype=np.uint32) << 16
    g = bits.view(np.float32)
    fin = np.isfinite(g)
    got = moe.silu_f32(g[fin]).view(np.uint32)
    want = _correctly_rounded_silu_f32(g[fin])
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(float(g[fin][i]), hex(got[i]), hex(want[i])) for i in bad[:5]]


def test_silu_near_midpoint_cases_hand_derived():
    """g = -2^-24: silu(g) = -2^-25 (1 - 2^-25 + 2^-72/48 + ...) sits 2^-76.6 above the
    magnitude midpoint 2^-25 - 2^-50, so it rounds to -2^-25; g = 2^-23:
    silu(g) = 2^-24 (1 + 2^-24 - ...) rounds to 2^-24 (the midpoint is 2^-24 (1 + 2^-24))."""
    assert moe.silu_f32(np.float32(-2.0 ** -24)).view(np.uint32) == np.float32(-2.0 ** -25).view(np.uint32)
    assert moe.silu_f32(np.float32(2.0 ** -23)) == np.float32(2.0 ** -24)
