"""Python binding of the fq C-ABI library (libfq.so, sm_103a).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  torch supplies device memory and the current stream.  The
names match the C entry points in include/fq.h.  There is no CPU fallback:
if the library is missing or the device is not sm_103, calls raise.
"""
import ctypes
import os

import torch

__all__ = [
    "FqError", "lib", "lib_path", "dynamic_quant_int8", "w8a8_linear", "w8a8_quant_linear",
    "quant_fp8_group_ue8m0_packed", "quant_fp8_group_fp32", "pack_scales_ue8m0", "quantize_weight_fp8_block",
    "fp8_group_einsum", "scale_view", "moe_sort", "moe_gather_rows_i8", "w8a8_grouped_linear",
    "swiglu_quant_int8", "moe_combine", "device_error", "selftest_wait_timeout", "rmsnorm_quant_int8",
    "rmsnorm_quant_fp8_ue8m0_packed", "check_device_error", "repack_weight_kmajor_i8",
    "repack_weight_kmajor_fp8", "quant_mxfp8", "mxfp8_linear", "OP_MXFP8_LINEAR", "workspace_bytes", "SCALE_UE8M0_PACKED", "SCALE_FP32",
    "OP_W8A8_LINEAR", "OP_W8A8_QUANT_LINEAR", "OP_FP8_GROUP_EINSUM", "OP_MOE_SORT", "OP_W8A8_GROUPED_LINEAR",
]

SCALE_UE8M0_PACKED = 0
SCALE_FP32 = 1
OP_W8A8_LINEAR, OP_W8A8_QUANT_LINEAR, OP_FP8_GROUP_EINSUM, OP_MOE_SORT, OP_W8A8_GROUPED_LINEAR = 1, 2, 3, 4, 5
OP_MXFP8_LINEAR = 6

_HERE = os.path.dirname(os.path.abspath(__file__))
lib_path = os.path.join(_HERE, "libfq.so")
_LIB = None

_P, _I64, _SZ, _I32, _U32P = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t, ctypes.c_int, ctypes.POINTER(ctypes.c_uint32)
_SIGS = {
    "fq_status_string": ([_I32], ctypes.c_char_p),
    "fq_last_cuda_error": ([], _I32),
    "fq_device_error": ([_P, _U32P], _I32),
    "fq_check_device_error": ([_P], _I32),
    "fq_repack_weight_kmajor_i8": ([_P, _I64, _I64, _I64, _P, _P], _I32),
    "fq_repack_weight_kmajor_fp8": ([_P, _I64, _I64, _I64, _P, _P], _I32),
    "fq_selftest_wait_timeout": ([ctypes.c_uint64, _I32, _P], _I32),
    "rmsnorm_quant_int8": ([_P, _P, ctypes.c_float, _I64, _I64, _P, _P, _P], _I32),
    "rmsnorm_quant_fp8_ue8m0_packed": ([_P, _P, ctypes.c_float, _I64, _I64, _P, _P, _P], _I32),
    "quant_mxfp8": ([_P, _I64, _I64, _P, _P, _P], _I32),
    "mxfp8_linear": ([_P, _P, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P], _I32),
    "fq_workspace_bytes": ([_I32, _I64, _I64, _I64, _I64], _SZ),
    "dynamic_quant_int8": ([_P, _I64, _I64, _P, _P, _P], _I32),
    "w8a8_linear": ([_P, _P, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P], _I32),
    "w8a8_quant_linear": ([_P, _I64, _I64, _P, _P, _I64, _P, _P, _P, _P, _SZ, _P], _I32),
    "w8a8_linear_noalloc": ([_P, _P, _I64, _I64, _P, _P, _I64, _P, _P], _I32),
    "quant_fp8_group_ue8m0_packed": ([_P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "quant_fp8_group_fp32": ([_P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "fq_pack_scales_ue8m0": ([_P, _I64, _I64, _I64, _P, _P], _I32),
    "fq_quantize_weight_fp8_block": ([_P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "fp8_group_einsum": ([_P, _P, _I32, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P], _I32),
    "moe_sort": ([_P, _I64, _I64, _I64, _P, _P, _P, _P, _SZ, _P], _I32),
    "moe_gather_rows_i8": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _P], _I32),
    "w8a8_grouped_linear": ([_P, _P, _P, _I64, _I64, _I64, _P, _P, _I64, _P, _P, _SZ, _P], _I32),
    "swiglu_quant_int8": ([_P, _I64, _I64, _P, _P, _P, _P], _I32),
    "moe_combine": ([_P, _P, _P, _I64, _I64, _I64, _P, _P], _I32),
}


class FqError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = lib().fq_status_string(status).decode()
        if status == 6:
            msg += " (cudaError %d)" % lib().fq_last_cuda_error()
        super().__init__("%s: %s [status %d]" % (fn, msg, status))


def lib():
    """Loads libfq.so (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(lib_path):
            raise RuntimeError("libfq.so is not built; run fp8_dynamic_quant_gb300.build.build()")
        L = ctypes.CDLL(lib_path)
        for name, (args, res) in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = res
        _LIB = L
    return _LIB


def _ptr(t):
    # an int: ctypes converts it for the c_void_p parameters
    return None if t is None else t.data_ptr()


_RAW_STREAM = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream():
    """The current CUDA stream of the current device, as a raw handle."""
    if _RAW_STREAM is not None:
        return ctypes.c_void_p(_RAW_STREAM(torch.cuda.current_device()))
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check(fn, status):
    if status != 0:
        raise FqError(fn, status)


def _cuda(t, dtype, name):
    if isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == dtype and t.is_contiguous():
        return t
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return t


_WS_BYTES = {}


def workspace_bytes(op, a, b=0, c=0, d=0):
    """fq_workspace_bytes for the current device (memoised per device and arguments)."""
    key = (torch.cuda.current_device() if torch.cuda.is_available() else -1, op, a, b, c, d)
    v = _WS_BYTES.get(key)
    if v is None:
        v = int(lib().fq_workspace_bytes(op, a, b, c, d))
        if v:
            _WS_BYTES[key] = v
    return v


# Zero-filled workspaces, one per (device, stream); every call leaves them zero.
_WS = {}


def _workspace(nbytes, device, ws=None):
    """The caller's workspace if given (uint8, zero-filled before first use), else a cached one."""
    if ws is not None:
        _cuda(ws, torch.uint8, "ws")
        if ws.numel() < nbytes:
            raise ValueError("workspace too small: %d < %d bytes" % (ws.numel(), nbytes))
        return ws
    key = (device.index, torch.cuda.current_stream(device).cuda_stream)
    cur = _WS.get(key)
    if cur is None or cur.numel() < nbytes:
        cur = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=device)
        _WS[key] = cur
    return cur


def _workspace_for(op, device, ws, a, b=0, c=0, d=0):
    """The caller's workspace (uint8; the library checks its size and returns
    FQ_ERR_WORKSPACE when it is too small), else a cached zero-filled one."""
    if ws is not None:
        return _cuda(ws, torch.uint8, "ws")
    key = (device.index, op, a, b, c, d)
    nb = _WS_BYTES.get(key)
    if nb is None:
        nb = int(lib().fq_workspace_bytes(op, a, b, c, d))
        if nb:
            _WS_BYTES[key] = nb
    return _workspace(nb, device)


def new_workspace(nbytes, device):
    """A zero-filled workspace tensor for explicit use (e.g. under CUDA graph capture)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def device_error():
    """Synchronises the current stream and returns (status, raw word) of the device error word."""
    w = ctypes.c_uint32(0)
    st = lib().fq_device_error(_stream(), ctypes.byref(w))
    return st, w.value


def check_device_error():
    """Synchronises the current stream; returns the status of the device error word (and clears it)."""
    return int(lib().fq_check_device_error(_stream()))


def repack_weight_kmajor_i8(w_kn, out=None):
    """Logical int8 weights [K, N] or [B, K, N] -> K-major storage [N, K] / [B, N, K] (load time)."""
    _cuda(w_kn, torch.int8, "w_kn")
    squeeze = w_kn.dim() == 2
    w3 = w_kn.unsqueeze(0) if squeeze else w_kn
    B, K, N = w3.shape
    out = torch.empty((B, N, K), dtype=torch.int8, device=w_kn.device) if out is None else out.view(B, N, K)
    _check("fq_repack_weight_kmajor_i8", lib().fq_repack_weight_kmajor_i8(_ptr(w3), B, K, N, _ptr(out), _stream()))
    return out[0] if squeeze else out


def repack_weight_kmajor_fp8(w_gdn, out=None):
    """Logical E4M3 einsum weights [G, D, N] -> K-major storage [G, N, D] (load time)."""
    _cuda(w_gdn, torch.float8_e4m3fn, "w_gdn")
    G, D, N = w_gdn.shape
    out = torch.empty((G, N, D), dtype=torch.float8_e4m3fn, device=w_gdn.device) if out is None else out
    _check("fq_repack_weight_kmajor_fp8",
           lib().fq_repack_weight_kmajor_fp8(_ptr(w_gdn), G, D, N, _ptr(out), _stream()))
    return out


def selftest_wait_timeout(budget_ns=1_000_000, arrive=False):
    """Launch the bounded-wait self-test on the current stream (see fq.h);
    with arrive=False the wait runs out and device_error() then reports
    FQ_ERR_DEVICE_TIMEOUT."""
    _check("fq_selftest_wait_timeout", lib().fq_selftest_wait_timeout(int(budget_ns), 1 if arrive else 0, _stream()))


# ---------------------------------------------------------------- RMSNorm + quant

def rmsnorm_quant_int8(x, gamma, eps=1e-6, xq=None, sx=None):
    """x bf16 [M, K], gamma bf16 [K] -> (xq int8 [M, K], sx fp32 [M]) of RMSNorm(x)."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(gamma, torch.bfloat16, "gamma")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    sx = torch.empty((M,), dtype=torch.float32, device=x.device) if sx is None else sx
    _check("rmsnorm_quant_int8", lib().rmsnorm_quant_int8(_ptr(x), _ptr(gamma), float(eps), M, K, _ptr(xq),
                                                          _ptr(sx), _stream()))
    return xq, sx


def rmsnorm_quant_fp8_ue8m0_packed(x, gamma, eps=1e-6, xq=None, s_packed=None):
    """x bf16 [T, K], gamma bf16 [K] -> (xq float8_e4m3fn [T, K], int32 [1, P, Ta]) of RMSNorm(x)."""
    _cuda(x, torch.bfloat16, "x")
    _cuda(gamma, torch.bfloat16, "gamma")
    T, K = x.shape
    P, Ta = (K // 128 + 3) // 4, (T + 3) // 4 * 4
    xq = torch.empty((T, K), dtype=torch.float8_e4m3fn, device=x.device) if xq is None else xq
    s_packed = torch.empty((1, P, Ta), dtype=torch.int32, device=x.device) if s_packed is None else s_packed
    _check("rmsnorm_quant_fp8_ue8m0_packed",
           lib().rmsnorm_quant_fp8_ue8m0_packed(_ptr(x), _ptr(gamma), float(eps), T, K, _ptr(xq), _ptr(s_packed),
                                                _stream()))
    return xq, s_packed


# ---------------------------------------------------------------- 32-element block-scaled FP8

def quant_mxfp8(x, q=None, sf=None):
    """x bf16 [R, K] -> (q float8_e4m3fn [R, K], blocked scales uint8 [ceil(R/128), K/128, 512])."""
    _cuda(x, torch.bfloat16, "x")
    R, K = x.shape
    q = torch.empty((R, K), dtype=torch.float8_e4m3fn, device=x.device) if q is None else q
    sf = torch.empty(((R + 127) // 128, K // 128, 512), dtype=torch.uint8, device=x.device) if sf is None else sf
    _check("quant_mxfp8", lib().quant_mxfp8(_ptr(x), R, K, _ptr(q), _ptr(sf), _stream()))
    return q, sf


def mxfp8_linear(xq, xsf, wq, wsf, y=None, ws=None):
    """E4M3 xq [M, K] + blocked scales, E4M3 wq [N, K] + blocked scales -> bf16 y [M, N]."""
    _cuda(xq, torch.float8_e4m3fn, "xq"), _cuda(wq, torch.float8_e4m3fn, "wq")
    _cuda(xsf, torch.uint8, "xsf"), _cuda(wsf, torch.uint8, "wsf")
    M, K = xq.shape
    N = wq.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ws = _workspace_for(OP_MXFP8_LINEAR, xq.device, ws, M, K, N)
    _check("mxfp8_linear", lib().mxfp8_linear(_ptr(xq), _ptr(xsf), M, K, _ptr(wq), _ptr(wsf), N, _ptr(y), _ptr(ws),
                                              ws.numel() * ws.element_size(), _stream()))
    return y


# ---------------------------------------------------------------- INT8 path

def dynamic_quant_int8(x, xq=None, sx=None):
    """x bf16 [M, K] -> (xq int8 [M, K], sx fp32 [M])."""
    _cuda(x, torch.bfloat16, "x")
    M, K = x.shape
    xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
    sx = torch.empty((M,), dtype=torch.float32, device=x.device) if sx is None else sx
    _check("dynamic_quant_int8", lib().dynamic_quant_int8(_ptr(x), M, K, _ptr(xq), _ptr(sx), _stream()))
    return xq, sx


def w8a8_linear(xq, sx, w_nk, sw, y=None, ws=None):
    """xq int8 [M, K], sx fp32 [M], w_nk int8 [N, K], sw fp32 [N] -> y bf16 [M, N]."""
    _cuda(xq, torch.int8, "xq"), _cuda(sx, torch.float32, "sx"), _cuda(w_nk, torch.int8, "w_nk")
    _cuda(sw, torch.float32, "sw")
    M, K = xq.shape
    N = w_nk.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ws = _workspace_for(OP_W8A8_LINEAR, xq.device, ws, M, K, N)
    _check("w8a8_linear", lib().w8a8_linear(_ptr(xq), _ptr(sx), M, K, _ptr(w_nk), _ptr(sw), N, _ptr(y),
                                            _ptr(ws), ws.numel(), _stream()))
    return y


def w8a8_quant_linear(x, w_nk, sw, y=None, return_quant=False, ws=None, xq=None, sx=None):
    """x bf16 [M, K] -> y bf16 [M, N] (optionally also (xq, sx))."""
    _cuda(x, torch.bfloat16, "x"), _cuda(w_nk, torch.int8, "w_nk"), _cuda(sw, torch.float32, "sw")
    M, K = x.shape
    N = w_nk.shape[0]
    y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device) if y is None else y
    if return_quant:
        xq = torch.empty((M, K), dtype=torch.int8, device=x.device) if xq is None else xq
        sx = torch.empty((M,), dtype=torch.float32, device=x.device) if sx is None else sx
    ws = _workspace_for(OP_W8A8_QUANT_LINEAR, x.device, ws, M, K, N)
    _check("w8a8_quant_linear", lib().w8a8_quant_linear(_ptr(x), M, K, _ptr(w_nk), _ptr(sw), N, _ptr(y), _ptr(xq),
                                                        _ptr(sx), _ptr(ws), ws.numel(), _stream()))
    return (y, xq, sx) if return_quant else y


# ---------------------------------------------------------------- FP8 path

def packed_dims(T, D):
    NG = D // 128
    return NG, (NG + 3) // 4, (T + 3) // 4 * 4


def quant_fp8_group_ue8m0_packed(x, xq=None, st=None):
    """x bf16 [T, G, D] -> (xq float8_e4m3fn [T, G, D], storage int32 [G, P, Ta])."""
    _cuda(x, torch.bfloat16, "x")
    T, G, D = x.shape
    _, P, Ta = packed_dims(T, D)
    xq = torch.empty((T, G, D), dtype=torch.float8_e4m3fn, device=x.device) if xq is None else xq
    st = torch.empty((G, P, Ta), dtype=torch.int32, device=x.device) if st is None else st
    _check("quant_fp8_group_ue8m0_packed",
           lib().quant_fp8_group_ue8m0_packed(_ptr(x), T, G, D, _ptr(xq), _ptr(st), _stream()))
    return xq, st


def scale_view(storage, T):
    """Logical [T, G, P] view of the [G, P, Ta] storage (strides (1, P*Ta, Ta))."""
    return storage.transpose(-1, -2)[:, :T, :].transpose(0, 1)


def quant_fp8_group_fp32(x, xq=None, s=None):
    """x bf16 [T, G, D] -> (xq float8_e4m3fn, fp32 scales [T, G, D/128])."""
    _cuda(x, torch.bfloat16, "x")
    T, G, D = x.shape
    xq = torch.empty((T, G, D), dtype=torch.float8_e4m3fn, device=x.device) if xq is None else xq
    s = torch.empty((T, G, D // 128), dtype=torch.float32, device=x.device) if s is None else s
    _check("quant_fp8_group_fp32", lib().quant_fp8_group_fp32(_ptr(x), T, G, D, _ptr(xq), _ptr(s), _stream()))
    return xq, s


def pack_scales_ue8m0(s_f32, out=None):
    """fp32 power-of-two scales [T, G, NG] -> packed int32 [G, ceil(NG/4), align4(T)]."""
    _cuda(s_f32, torch.float32, "s_f32")
    T, G, NG = s_f32.shape
    if out is None:
        out = torch.empty((G, (NG + 3) // 4, (T + 3) // 4 * 4), dtype=torch.int32, device=s_f32.device)
    _check("fq_pack_scales_ue8m0", lib().fq_pack_scales_ue8m0(_ptr(s_f32), T, G, NG, _ptr(out), _stream()))
    return out


def quantize_weight_fp8_block(w_gnd):
    """fp32 [G, N, D] -> (wq float8_e4m3fn [G, N, D], sw fp32 [G, D/128, N/128])."""
    _cuda(w_gnd, torch.float32, "w_gnd")
    G, N, D = w_gnd.shape
    wq = torch.empty((G, N, D), dtype=torch.float8_e4m3fn, device=w_gnd.device)
    sw = torch.empty((G, D // 128, N // 128), dtype=torch.float32, device=w_gnd.device)
    _check("fq_quantize_weight_fp8_block",
           lib().fq_quantize_weight_fp8_block(_ptr(w_gnd), G, N, D, _ptr(wq), _ptr(sw), _stream()))
    return wq, sw


def fp8_group_einsum(xq, sx, fmt, wq, sw_blk, y=None, ws=None):
    """xq e4m3 [T, G, D], scales (packed storage or fp32), wq e4m3 [G, N, D], sw [G, D/128, N/128] -> y bf16 [T, G, N]."""
    _cuda(xq, torch.float8_e4m3fn, "xq"), _cuda(wq, torch.float8_e4m3fn, "wq"), _cuda(sw_blk, torch.float32, "sw")
    _cuda(sx, torch.int32 if fmt == SCALE_UE8M0_PACKED else torch.float32, "sx")
    T, G, D = xq.shape
    N = wq.shape[1]
    y = torch.empty((T, G, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ws = _workspace_for(OP_FP8_GROUP_EINSUM, xq.device, ws, T, D, N, G)
    _check("fp8_group_einsum", lib().fp8_group_einsum(_ptr(xq), _ptr(sx), fmt, T, G, D, _ptr(wq), _ptr(sw_blk), N,
                                                      _ptr(y), _ptr(ws), ws.numel(), _stream()))
    return y


# ---------------------------------------------------------------- MoE path

def moe_sort(topk_ids, E, out=None):
    """topk_ids int32 [T, topk] -> (offsets [E+1], perm [T*topk], pair_row [T*topk])."""
    _cuda(topk_ids, torch.int32, "topk_ids")
    T, topk = topk_ids.shape
    dev = topk_ids.device
    if out is not None:
        offsets, perm, pair_row = out
    else:
        offsets = torch.empty((E + 1,), dtype=torch.int32, device=dev)
        perm = torch.empty((T * topk,), dtype=torch.int32, device=dev)
        pair_row = torch.empty((T * topk,), dtype=torch.int32, device=dev)
    _check("moe_sort", lib().moe_sort(_ptr(topk_ids), T, topk, E, _ptr(offsets), _ptr(perm), _ptr(pair_row),
                                      None, 0, _stream()))
    return offsets, perm, pair_row


def moe_gather_rows_i8(xq, sx, perm, topk, out=None):
    _cuda(xq, torch.int8, "xq"), _cuda(sx, torch.float32, "sx"), _cuda(perm, torch.int32, "perm")
    T, K = xq.shape
    R = T * topk
    if out is not None:
        xg, sg = out
    else:
        xg = torch.empty((R, K), dtype=torch.int8, device=xq.device)
        sg = torch.empty((R,), dtype=torch.float32, device=xq.device)
    _check("moe_gather_rows_i8", lib().moe_gather_rows_i8(_ptr(xq), _ptr(sx), _ptr(perm), T, topk, K, _ptr(xg),
                                                          _ptr(sg), _stream()))
    return xg, sg


def w8a8_grouped_linear(xq, sx, offsets, w_enk, sw_en, y=None, ws=None):
    _cuda(xq, torch.int8, "xq"), _cuda(sx, torch.float32, "sx"), _cuda(offsets, torch.int32, "offsets")
    _cuda(w_enk, torch.int8, "w_enk"), _cuda(sw_en, torch.float32, "sw_en")
    R, K = xq.shape
    E, N, _ = w_enk.shape
    y = torch.empty((R, N), dtype=torch.bfloat16, device=xq.device) if y is None else y
    ws = _workspace_for(OP_W8A8_GROUPED_LINEAR, xq.device, ws, R, K, N, E)
    _check("w8a8_grouped_linear", lib().w8a8_grouped_linear(_ptr(xq), _ptr(sx), _ptr(offsets), R, E, K, _ptr(w_enk),
                                                            _ptr(sw_en), N, _ptr(y), _ptr(ws), ws.numel(),
                                                            _stream()))
    return y


def swiglu_quant_int8(gu, return_h=False, out=None):
    """gu bf16 [rows, 2I] -> (hq int8 [rows, I], sh fp32 [rows]) (+ h bf16 [rows, I])."""
    _cuda(gu, torch.bfloat16, "gu")
    rows, I2 = gu.shape
    I = I2 // 2
    if out is not None:
        hq, sh = out
    else:
        hq = torch.empty((rows, I), dtype=torch.int8, device=gu.device)
        sh = torch.empty((rows,), dtype=torch.float32, device=gu.device)
    h = torch.empty((rows, I), dtype=torch.bfloat16, device=gu.device) if return_h else None
    _check("swiglu_quant_int8", lib().swiglu_quant_int8(_ptr(gu), rows, I, _ptr(hq), _ptr(sh), _ptr(h), _stream()))
    return (hq, sh, h) if return_h else (hq, sh)


def moe_combine(y_rows, pair_row, topk_w, out=None):
    _cuda(y_rows, torch.bfloat16, "y_rows"), _cuda(pair_row, torch.int32, "pair_row")
    _cuda(topk_w, torch.float32, "topk_w")
    T, topk = topk_w.shape
    H = y_rows.shape[1]
    out = torch.empty((T, H), dtype=torch.bfloat16, device=y_rows.device) if out is None else out
    _check("moe_combine", lib().moe_combine(_ptr(y_rows), _ptr(pair_row), _ptr(topk_w), T, topk, H, _ptr(out),
                                            _stream()))
    return out


class MoEBuffers:
    """Preallocated intermediates of the expert path (so the chain allocates nothing)."""

    def __init__(self, T, topk, E, H, I, device):
        R = T * topk
        z = dict(device=device)
        self.xq = torch.empty((T, H), dtype=torch.int8, **z)
        self.sx = torch.empty((T,), dtype=torch.float32, **z)
        self.sort = (torch.empty((E + 1,), dtype=torch.int32, **z), torch.empty((R,), dtype=torch.int32, **z),
                     torch.empty((R,), dtype=torch.int32, **z))
        self.gather = (torch.empty((R, H), dtype=torch.int8, **z), torch.empty((R,), dtype=torch.float32, **z))
        self.y1 = torch.empty((R, 2 * I), dtype=torch.bfloat16, **z)
        self.hq = (torch.empty((R, I), dtype=torch.int8, **z), torch.empty((R,), dtype=torch.float32, **z))
        self.y2 = torch.empty((R, H), dtype=torch.bfloat16, **z)
        self.out = torch.empty((T, H), dtype=torch.bfloat16, **z)
        nb = max(workspace_bytes(OP_W8A8_GROUPED_LINEAR, R, H, 2 * I, E),
                 workspace_bytes(OP_W8A8_GROUPED_LINEAR, R, I, H, E))
        self.ws = new_workspace(nb, device)


def moe_forward(x, topk_ids, topk_w, w13, sw13, w2, sw2, bufs=None):
    """The whole expert path: quant -> sort -> gather -> W13 -> SwiGLU+quant -> W2 -> combine."""
    T, topk = topk_ids.shape
    E = w13.shape[0]
    if bufs is None:
        xq, sx = dynamic_quant_int8(x)
        offsets, perm, pair_row = moe_sort(topk_ids, E)
        xg, sg = moe_gather_rows_i8(xq, sx, perm, topk)
        y1 = w8a8_grouped_linear(xg, sg, offsets, w13, sw13)
        hq, sh = swiglu_quant_int8(y1)
        y2 = w8a8_grouped_linear(hq, sh, offsets, w2, sw2)
        return moe_combine(y2, pair_row, topk_w)
    b = bufs
    dynamic_quant_int8(x, b.xq, b.sx)
    offsets, perm, pair_row = moe_sort(topk_ids, E, out=b.sort)
    xg, sg = moe_gather_rows_i8(b.xq, b.sx, perm, topk, out=b.gather)
    w8a8_grouped_linear(xg, sg, offsets, w13, sw13, y=b.y1, ws=b.ws)
    hq, sh = swiglu_quant_int8(b.y1, out=b.hq)
    w8a8_grouped_linear(hq, sh, offsets, w2, sw2, y=b.y2, ws=b.ws)
    return moe_combine(b.y2, pair_row, topk_w, out=b.out)
