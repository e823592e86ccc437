"""Conversions between the oracle's numpy arrays and CUDA tensors (tests only)."""
import numpy as np
import torch


def bf16_to_dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits, np.uint16).view(np.int16)).view(torch.bfloat16).cuda()


def bf16_to_np(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def e4m3_to_np(t):
    return t.detach().cpu().contiguous().view(torch.uint8).numpy()


def np_to_dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def e4m3_to_dev(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).cuda().view(torch.float8_e4m3fn)


def within_tol(got_bits, want_bits, rtol=1e-2, atol=1e-3):
    """Elementwise |got - want| <= atol + rtol * |want| on bf16 bit arrays; returns (ok, worst index info)."""
    from oracle.codecs import bf16_to_f32
    g = bf16_to_f32(got_bits).astype(np.float64)
    w = bf16_to_f32(want_bits).astype(np.float64)
    err = np.abs(g - w) - (atol + rtol * np.abs(w))
    i = int(np.argmax(err)) if err.size else 0
    return bool(err.size == 0 or err.max() <= 0), (i, g.ravel()[i] if err.size else None, w.ravel()[i] if err.size else None)


def assert_within_tol(got_bits, want_bits, rtol=1e-2, atol=1e-3):
    """Assert within_tol, reporting the worst element (index, got, want) on failure."""
    ok, info = within_tol(got_bits, want_bits, rtol, atol)
    assert ok, info
