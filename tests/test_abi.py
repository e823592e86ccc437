"""The C-ABI library builds, loads and exports every symbol include/fq.h declares.

No compute calls are made here (this runs without a GPU).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fq.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


@pytest.fixture(scope="module")
def libfq():
    from fp8_dynamic_quant_gb300 import build
    path = build.build()
    return ctypes.CDLL(path)


def test_header_declares_the_path():
    names = declared_functions()
    for n in ["dynamic_quant_int8", "quant_fp8_group_ue8m0_packed", "w8a8_linear", "w8a8_quant_linear",
              "fp8_group_einsum", "moe_sort", "w8a8_grouped_linear", "swiglu_quant_int8", "moe_combine",
              "fq_workspace_bytes", "fq_status_string", "fq_device_error", "fq_check_device_error",
              "fq_repack_weight_kmajor_i8", "fq_repack_weight_kmajor_fp8"]:
        assert n in names, n


def test_every_declared_symbol_is_exported(libfq):
    for n in declared_functions():
        assert hasattr(libfq, n), "missing export: " + n


def test_binding_signatures_cover_the_header():
    import fp8_dynamic_quant_gb300 as fq
    assert set(declared_functions()) == set(fq._SIGS.keys())


def test_status_strings(libfq):
    libfq.fq_status_string.restype = ctypes.c_char_p
    libfq.fq_status_string.argtypes = [ctypes.c_int]
    assert libfq.fq_status_string(0) == b"ok"
    for s in range(1, 10):
        assert libfq.fq_status_string(s) not in (b"ok", b"unknown status")
    assert libfq.fq_status_string(1234) == b"unknown status"


def test_host_validation_before_any_device_call(libfq):
    """Shape / null / enum errors are reported on the host, before the device is touched."""
    import fp8_dynamic_quant_gb300 as fq
    L = fq.lib()
    # negative sizes and broken divisibility
    assert L.dynamic_quant_int8(None, -1, 16, None, None, None) == 2
    assert L.dynamic_quant_int8(None, 4, 15, None, None, None) == 2
    assert L.w8a8_linear(None, None, 4, 4096, None, None, 1000, None, None, 0, None) == 2   # N % 16
    assert L.quant_fp8_group_ue8m0_packed(None, 1, 8, 100, None, None, None) == 2         # D % 128
    assert L.fp8_group_einsum(None, None, 7, 1, 8, 4096, None, None, 1024, None, None, 0, None) == 9  # fmt
    # empty problems succeed without launching anything
    assert L.dynamic_quant_int8(None, 0, 4096, None, None, None) == 0
    assert L.w8a8_linear(None, None, 0, 4096, None, None, 1024, None, None, 0, None) == 0
    assert L.quant_fp8_group_ue8m0_packed(None, 0, 3, 128, None, None, None) == 0
    # null pointers on a real problem
    assert L.dynamic_quant_int8(None, 4, 4096, None, None, None) == 1
    assert L.w8a8_linear(None, None, 4, 4096, None, None, 1024, None, None, 0, None) == 1
    # misaligned pointers
    assert L.dynamic_quant_int8(ctypes.c_void_p(0x1008), 4, 4096, ctypes.c_void_p(0x2000),
                                ctypes.c_void_p(0x3000), None) == 3
    # RMSNorm + quant: eps must be finite and >= 0; K % 16 (INT8) / % 128 (FP8); K <= 16384
    assert L.rmsnorm_quant_int8(None, None, -1.0, 4, 4096, None, None, None) == 9
    assert L.rmsnorm_quant_int8(None, None, float("nan"), 4, 4096, None, None, None) == 9
    assert L.rmsnorm_quant_int8(None, None, float("inf"), 4, 4096, None, None, None) == 9
    assert L.rmsnorm_quant_int8(None, None, 1e-6, 4, 4100, None, None, None) == 2
    assert L.rmsnorm_quant_int8(None, None, 1e-6, 4, 16400, None, None, None) == 2
    assert L.rmsnorm_quant_fp8_ue8m0_packed(None, None, 1e-6, 4, 4112, None, None, None) == 2
    assert L.rmsnorm_quant_int8(None, None, 1e-6, 0, 4096, None, None, None) == 0
    assert L.rmsnorm_quant_int8(None, None, 1e-6, 4, 4096, None, None, None) == 1
    # load-time repack: divisibility, empty, null, overlapping buffers
    assert L.fq_repack_weight_kmajor_i8(None, 1, 24, 16, None, None) == 2       # K % 16
    assert L.fq_repack_weight_kmajor_fp8(None, 1, 128, 192, None, None) == 2    # N % 128
    assert L.fq_repack_weight_kmajor_i8(None, 0, 16, 16, None, None) == 0       # empty
    assert L.fq_repack_weight_kmajor_i8(None, 1, 16, 16, None, None) == 1
    assert L.fq_repack_weight_kmajor_i8(ctypes.c_void_p(0x10000), 1, 64, 64, ctypes.c_void_p(0x10800), None) == 9


def test_workspace_sizing_without_device_is_zero():
    import fp8_dynamic_quant_gb300 as fq
    import torch
    if torch.cuda.is_available():
        pytest.skip("device present: sizing is exercised by the GPU tests")
    assert fq.workspace_bytes(fq.OP_W8A8_LINEAR, 4, 4096, 1024) == 0
    assert fq.workspace_bytes(99, 1, 1, 1) == 0
