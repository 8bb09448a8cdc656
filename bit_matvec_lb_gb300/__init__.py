"""Python binding of the GB300 low-bit product library (liblb.so, C ABI in include/lb.h).

The functions here carry the C names and only marshal arguments: torch tensors (or raw integer
device addresses) become pointers, the stream defaults to torch's current CUDA stream, and a
non-zero status raises :class:`LBError`.  Every step of the computation runs in the library's
CUDA kernels; there is no CPU or PyTorch fallback.  If the library is missing it is built with
nvcc on first use; if that fails, or the device is not sm_103, the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

__all__ = [
    "LBError", "load", "library_path", "status_string", "scale_stride", "lb_device_status",
    "lb_quantize_q8_0", "lb_quantize_i8_absmax", "lb_repack_q1_0", "lb_repack_q2_0_g64",
    "lb_gemv_q1_0", "lb_gemv_q2_0_g64", "lb_gemv_trit_planes", "lb_gemv_bf16",
    "lb_gemv_q1_0_grouped", "lb_gemv_q2_0_g64_grouped", "lb_gemv_trit_planes_grouped",
    "lb_gemm_workspace_bytes", "lb_gemm_q1_0", "lb_gemm_q2_0_g64", "lb_gemm_q1_0_grouped",
    "lb_gemm_q2_0_g64_grouped", "lb_gemm_q2_0_g64_noalloc", "lb_gemm_trit_workspace_bytes",
    "lb_gemm_trit_planes", "lb_gemm_trit_planes_grouped", "lb_quantize_i8_absmax_tiles",
    "lb_gemm_trit_planes_grouped_tiles", "lb_dequantize_q1_0",
    "lb_dequantize_q2_0_g64", "lb_dequantize_trit_planes", "OUT_F32", "OUT_BF16",
    "lb_pack_base3", "lb_gemv_base3", "base3_row_bytes", "lb_test_inject_wait_timeout",
]

LB_STATUS = {0: "LB_OK", -1: "LB_ERR_NULL", -2: "LB_ERR_ALIGN", -3: "LB_ERR_SHAPE",
             -4: "LB_ERR_BATCH", -5: "LB_ERR_ARCH", -6: "LB_ERR_LAUNCH", -7: "LB_ERR_DEVICE"}


class LBError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: str = ""):
        self.status = status
        self.cuda_error = cuda_error
        extra = f", {cuda_error}" if cuda_error else ""
        super().__init__(
            f"{fn} returned {status} ({LB_STATUS.get(status, 'LB_ERR_UNKNOWN')}{extra})")


_lib = None
_lock = threading.Lock()
P = ctypes.c_void_p
I64 = ctypes.c_int64
I32 = ctypes.c_int
F32 = ctypes.c_float

MAX_GROUP = 64


class lb_q_matrix(ctypes.Structure):
    _fields_ = [("bits", P), ("scales", P), ("y", P), ("isum_opt", P), ("N", I64)]


class lb_trit_matrix(ctypes.Structure):
    _fields_ = [("planes", P), ("w_scale", F32), ("y", P), ("acc_opt", P), ("N", I64)]


class lb_gemm_matrix(ctypes.Structure):
    _fields_ = [("bits", P), ("scales", P), ("y", P), ("N", I64)]


GEMM_MAX_GROUP = 8


SIGNATURES = {
    "lb_status_string": (ctypes.c_char_p, [I32]),
    "lb_version": (I32, []),
    "lb_last_cuda_error": (I32, []),
    "lb_cuda_error_name": (ctypes.c_char_p, [I32]),
    "lb_quantize_q8_0": (I32, [P, P, P, I64, I64, P]),
    "lb_quantize_i8_absmax": (I32, [P, P, P, I64, I64, P]),
    "lb_repack_q1_0": (I32, [P, I64, I64, P, P, P]),
    "lb_repack_q2_0_g64": (I32, [P, I64, I64, P, P, P]),
    "lb_gemv_q1_0": (I32, [P, P, P, P, P, P, I64, I64, I32, P]),
    "lb_gemv_q2_0_g64": (I32, [P, P, P, P, P, P, I64, I64, I32, P]),
    "lb_gemv_trit_planes": (I32, [P, F32, P, P, P, P, I64, I64, I32, P]),
    "lb_gemv_bf16": (I32, [P, P, P, I64, I64, I32, P]),
    "lb_device_status": (I32, [P]),
    "lb_test_inject_wait_timeout": (I32, [I32]),
    "lb_gemv_q1_0_grouped": (I32, [ctypes.POINTER(lb_q_matrix), I32, P, P, I64, I32, P]),
    "lb_gemv_q2_0_g64_grouped": (I32, [ctypes.POINTER(lb_q_matrix), I32, P, P, I64, I32, P]),
    "lb_gemv_trit_planes_grouped": (I32, [ctypes.POINTER(lb_trit_matrix), I32, P, P, I64, I32,
                                          P]),
    "lb_gemm_workspace_bytes": (ctypes.c_size_t, [I64, I64]),
    "lb_gemm_q1_0": (I32, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, P]),
    "lb_gemm_q2_0_g64": (I32, [P, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, P]),
    "lb_gemm_q2_0_g64_noalloc": (I32, [P, P, P, P, P, I64, I64, I64, P]),
    "lb_gemm_q1_0_grouped": (I32, [ctypes.POINTER(lb_gemm_matrix), I32, P, P, I64, I64, P,
                                   ctypes.c_size_t, P]),
    "lb_gemm_q2_0_g64_grouped": (I32, [ctypes.POINTER(lb_gemm_matrix), I32, P, P, I64, I64, P,
                                       ctypes.c_size_t, P]),
    "lb_gemm_trit_workspace_bytes": (ctypes.c_size_t, [I64, I64]),
    "lb_gemm_trit_planes": (I32, [P, F32, P, P, P, P, I64, I64, I64, P, ctypes.c_size_t, P]),
    "lb_gemm_trit_planes_grouped": (I32, [ctypes.POINTER(lb_trit_matrix), I32, P, P, I64, I64, P,
                                          ctypes.c_size_t, P]),
    "lb_quantize_i8_absmax_tiles": (I32, [P, P, P, I64, I64, P, ctypes.c_size_t, P]),
    "lb_gemm_trit_planes_grouped_tiles": (I32, [ctypes.POINTER(lb_trit_matrix), I32, P, I64, I64,
                                                P, ctypes.c_size_t, P]),
    "lb_dequantize_q1_0": (I32, [P, P, I64, I64, I32, P, P]),
    "lb_dequantize_q2_0_g64": (I32, [P, P, I64, I64, I32, P, P]),
    "lb_dequantize_trit_planes": (I32, [P, F32, I64, I64, I32, P, P]),
    "lb_pack_base3": (I32, [P, I64, I64, P, P]),
    "lb_gemv_base3": (I32, [P, F32, P, P, P, P, I64, I64, I32, P]),
}

OUT_F32 = 0
OUT_BF16 = 1

NOALLOC_SCRATCH_BYTES = 8 << 20


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True):
    """Load liblb.so (building it with nvcc if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if build_if_missing and not _build.up_to_date():
                path = _build.build()
            if not os.path.exists(path):
                raise RuntimeError(f"GB300 library not built: {path} is missing")
            lib = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def scale_stride(K: int, qk: int) -> int:
    """Row stride (entries) of a repacked scale plane: K/QK rounded up to a multiple of 8."""
    return (K // qk + 7) // 8 * 8


def status_string(status: int) -> str:
    return load().lb_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if hasattr(t, "data_ptr"):
        if not t.is_cuda:
            raise ValueError("lb_* entry points take device tensors")
        if not t.is_contiguous():
            raise ValueError("lb_* entry points take contiguous tensors")
        return t.data_ptr()
    raise TypeError(f"cannot pass {type(t)} as a device pointer")


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, status: int):
    if status != 0:
        cuda = ""
        if status == -6:  # LB_ERR_LAUNCH
            code = load().lb_last_cuda_error()
            if code:
                cuda = load().lb_cuda_error_name(code).decode()
        raise LBError(fn, status, cuda)


def lb_last_cuda_error() -> int:
    """cudaError_t of the library's last failed CUDA call on this thread (then reset), or 0."""
    return int(load().lb_last_cuda_error())


def lb_cuda_error_name(code: int) -> str:
    return load().lb_cuda_error_name(int(code)).decode()


def lb_quantize_q8_0(x, q, d, B: int, K: int, stream=None):
    _check("lb_quantize_q8_0", load().lb_quantize_q8_0(_ptr(x), _ptr(q), _ptr(d), B, K,
                                                       _stream(stream)))


def lb_quantize_i8_absmax(x, q, x_scale, B: int, K: int, stream=None):
    _check("lb_quantize_i8_absmax", load().lb_quantize_i8_absmax(
        _ptr(x), _ptr(q), _ptr(x_scale), B, K, _stream(stream)))


def lb_repack_q1_0(blocks18, N: int, K: int, bits, scales, stream=None):
    _check("lb_repack_q1_0", load().lb_repack_q1_0(_ptr(blocks18), N, K, _ptr(bits),
                                                   _ptr(scales), _stream(stream)))


def lb_repack_q2_0_g64(blocks18, N: int, K: int, codes, scales, stream=None):
    _check("lb_repack_q2_0_g64", load().lb_repack_q2_0_g64(_ptr(blocks18), N, K, _ptr(codes),
                                                           _ptr(scales), _stream(stream)))


def lb_gemv_q1_0(bits, scales, q, d, y, isum, N: int, K: int, B: int, stream=None):
    _check("lb_gemv_q1_0", load().lb_gemv_q1_0(_ptr(bits), _ptr(scales), _ptr(q), _ptr(d),
                                               _ptr(y), _ptr(isum), N, K, B, _stream(stream)))


def lb_gemv_q2_0_g64(codes, scales, q, d, y, isum, N: int, K: int, B: int, stream=None):
    _check("lb_gemv_q2_0_g64", load().lb_gemv_q2_0_g64(
        _ptr(codes), _ptr(scales), _ptr(q), _ptr(d), _ptr(y), _ptr(isum), N, K, B,
        _stream(stream)))


def lb_gemv_trit_planes(planes, w_scale: float, q, x_scale, y, acc, N: int, K: int, B: int,
                        stream=None):
    _check("lb_gemv_trit_planes", load().lb_gemv_trit_planes(
        _ptr(planes), float(w_scale), _ptr(q), _ptr(x_scale), _ptr(y), _ptr(acc), N, K, B,
        _stream(stream)))


def lb_gemv_bf16(w, x, y, N: int, K: int, B: int, stream=None):
    _check("lb_gemv_bf16", load().lb_gemv_bf16(_ptr(w), _ptr(x), _ptr(y), N, K, B,
                                               _stream(stream)))


def lb_device_status(stream=None) -> int:
    """Synchronize the stream and return (and clear) the device error status (0 = OK)."""
    return load().lb_device_status(_stream(stream))


def lb_test_inject_wait_timeout(wait_us: int):
    """Test hook: the next streaming GEMV call starves its first CTA, whose bounded wait then
    gives up after wait_us microseconds (reported by lb_device_status as LB_ERR_DEVICE)."""
    _check("lb_test_inject_wait_timeout", load().lb_test_inject_wait_timeout(int(wait_us)))


def _q_mats(mats):
    if not 1 <= len(mats) <= MAX_GROUP:
        raise ValueError(f"a group holds 1..{MAX_GROUP} matrices")
    arr = (lb_q_matrix * len(mats))()
    for i, (bits, scales, y, isum, N) in enumerate(mats):
        arr[i] = lb_q_matrix(_ptr(bits), _ptr(scales), _ptr(y), _ptr(isum), int(N))
    return arr


def lb_gemv_q1_0_grouped(mats, q, d, K: int, B: int, stream=None):
    """mats: sequence of (bits, scales, y, isum_or_None, N) sharing the activation q, d."""
    arr = _q_mats(mats)
    _check("lb_gemv_q1_0_grouped", load().lb_gemv_q1_0_grouped(
        arr, len(mats), _ptr(q), _ptr(d), K, B, _stream(stream)))


def lb_gemv_q2_0_g64_grouped(mats, q, d, K: int, B: int, stream=None):
    """mats: sequence of (codes, scales, y, isum_or_None, N) sharing the activation q, d."""
    arr = _q_mats(mats)
    _check("lb_gemv_q2_0_g64_grouped", load().lb_gemv_q2_0_g64_grouped(
        arr, len(mats), _ptr(q), _ptr(d), K, B, _stream(stream)))


def lb_gemv_trit_planes_grouped(mats, q, x_scale, K: int, B: int, stream=None):
    """mats: sequence of (planes, w_scale, y, acc_or_None, N) sharing the activation."""
    if not 1 <= len(mats) <= MAX_GROUP:
        raise ValueError(f"a group holds 1..{MAX_GROUP} matrices")
    arr = (lb_trit_matrix * len(mats))()
    for i, (planes, w_scale, y, acc, N) in enumerate(mats):
        arr[i] = lb_trit_matrix(_ptr(planes), float(w_scale), _ptr(y), _ptr(acc), int(N))
    _check("lb_gemv_trit_planes_grouped", load().lb_gemv_trit_planes_grouped(
        arr, len(mats), _ptr(q), _ptr(x_scale), K, B, _stream(stream)))


def lb_gemm_workspace_bytes(M: int, K: int) -> int:
    """Bytes of device scratch lb_gemm_* needs for M tokens of K columns."""
    return int(load().lb_gemm_workspace_bytes(int(M), int(K)))


def _gemm(name, bits, scales, q, d, y, M, N, K, workspace, workspace_bytes, stream):
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    nbytes = int(workspace_bytes)
    _check(name, getattr(load(), name)(_ptr(bits), _ptr(scales), _ptr(q), _ptr(d), _ptr(y),
                                       int(M), int(N), int(K), _ptr(workspace), nbytes,
                                       _stream(stream)))


def lb_gemm_q1_0(bits, scales, q, d, y, M: int, N: int, K: int, workspace,
                 workspace_bytes=None, stream=None):
    """workspace: a device tensor (its size is passed) or a pointer with workspace_bytes."""
    _gemm("lb_gemm_q1_0", bits, scales, q, d, y, M, N, K, workspace, workspace_bytes, stream)


def lb_gemm_q2_0_g64(codes, scales, q, d, y, M: int, N: int, K: int, workspace,
                     workspace_bytes=None, stream=None):
    _gemm("lb_gemm_q2_0_g64", codes, scales, q, d, y, M, N, K, workspace, workspace_bytes,
          stream)


def _gemm_grouped(name, mats, q, d, M, K, workspace, workspace_bytes, stream):
    if not 1 <= len(mats) <= GEMM_MAX_GROUP:
        raise ValueError(f"a GEMM group holds 1..{GEMM_MAX_GROUP} matrices")
    arr = (lb_gemm_matrix * len(mats))()
    for i, (bits, scales, y, N) in enumerate(mats):
        arr[i] = lb_gemm_matrix(_ptr(bits), _ptr(scales), _ptr(y), int(N))
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check(name, getattr(load(), name)(arr, len(mats), _ptr(q), _ptr(d), int(M), int(K),
                                       _ptr(workspace), int(workspace_bytes), _stream(stream)))


def lb_gemm_q1_0_grouped(mats, q, d, M: int, K: int, workspace, workspace_bytes=None,
                         stream=None):
    """mats: sequence of (bits, scales, y, N) sharing the activation q, d (one launch)."""
    _gemm_grouped("lb_gemm_q1_0_grouped", mats, q, d, M, K, workspace, workspace_bytes, stream)


def lb_gemm_q2_0_g64_grouped(mats, q, d, M: int, K: int, workspace, workspace_bytes=None,
                             stream=None):
    """mats: sequence of (codes, scales, y, N) sharing the activation q, d (one launch)."""
    _gemm_grouped("lb_gemm_q2_0_g64_grouped", mats, q, d, M, K, workspace, workspace_bytes,
                  stream)


def lb_gemm_q2_0_g64_noalloc(codes, scales, q, d, y, M: int, N: int, K: int, stream=None):
    """lb_gemm_q2_0_g64 with the library's fixed scratch (no workspace argument)."""
    _check("lb_gemm_q2_0_g64_noalloc", load().lb_gemm_q2_0_g64_noalloc(
        _ptr(codes), _ptr(scales), _ptr(q), _ptr(d), _ptr(y), int(M), int(N), int(K),
        _stream(stream)))


def lb_gemm_trit_workspace_bytes(M: int, K: int) -> int:
    """Bytes of device scratch lb_gemm_trit_planes* needs for M tokens of K columns."""
    return int(load().lb_gemm_trit_workspace_bytes(int(M), int(K)))


def lb_gemm_trit_planes(planes, w_scale: float, q, x_scale, y, acc, M: int, N: int, K: int,
                        workspace, workspace_bytes=None, stream=None):
    """Planar ternary prefill GEMM; workspace: a device tensor (its size is passed) or a
    pointer with workspace_bytes."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("lb_gemm_trit_planes", load().lb_gemm_trit_planes(
        _ptr(planes), float(w_scale), _ptr(q), _ptr(x_scale), _ptr(y), _ptr(acc), int(M),
        int(N), int(K), _ptr(workspace), int(workspace_bytes), _stream(stream)))


def lb_gemm_trit_planes_grouped(mats, q, x_scale, M: int, K: int, workspace,
                                workspace_bytes=None, stream=None):
    """mats: sequence of (planes, w_scale, y, acc_or_None, N) sharing the activation (one
    launch)."""
    if not 1 <= len(mats) <= GEMM_MAX_GROUP:
        raise ValueError(f"a GEMM group holds 1..{GEMM_MAX_GROUP} matrices")
    arr = (lb_trit_matrix * len(mats))()
    for i, (planes, w_scale, y, acc, N) in enumerate(mats):
        arr[i] = lb_trit_matrix(_ptr(planes), float(w_scale), _ptr(y), _ptr(acc), int(N))
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("lb_gemm_trit_planes_grouped", load().lb_gemm_trit_planes_grouped(
        arr, len(mats), _ptr(q), _ptr(x_scale), int(M), int(K), _ptr(workspace),
        int(workspace_bytes), _stream(stream)))


def lb_quantize_i8_absmax_tiles(x, q, x_scale, M: int, K: int, workspace, workspace_bytes=None,
                                stream=None):
    """lb_quantize_i8_absmax that also writes the planar GEMM's activation operand tiles into
    workspace (for lb_gemm_trit_planes_grouped_tiles)."""
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("lb_quantize_i8_absmax_tiles", load().lb_quantize_i8_absmax_tiles(
        _ptr(x), _ptr(q), _ptr(x_scale), int(M), int(K), _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def lb_gemm_trit_planes_grouped_tiles(mats, x_scale, M: int, K: int, workspace,
                                      workspace_bytes=None, stream=None):
    """lb_gemm_trit_planes_grouped from the operand tiles lb_quantize_i8_absmax_tiles wrote."""
    if not 1 <= len(mats) <= GEMM_MAX_GROUP:
        raise ValueError(f"a GEMM group holds 1..{GEMM_MAX_GROUP} matrices")
    arr = (lb_trit_matrix * len(mats))()
    for i, (planes, w_scale, y, acc, N) in enumerate(mats):
        arr[i] = lb_trit_matrix(_ptr(planes), float(w_scale), _ptr(y), _ptr(acc), int(N))
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size()
    _check("lb_gemm_trit_planes_grouped_tiles", load().lb_gemm_trit_planes_grouped_tiles(
        arr, len(mats), _ptr(x_scale), int(M), int(K), _ptr(workspace), int(workspace_bytes),
        _stream(stream)))


def lb_dequantize_q1_0(bits, scales, N: int, K: int, out_format: int, out, stream=None):
    """Every Q1_0 weight as (float)w * d: out [N][K] fp32 (OUT_F32) or bf16 bits (OUT_BF16)."""
    _check("lb_dequantize_q1_0", load().lb_dequantize_q1_0(
        _ptr(bits), _ptr(scales), int(N), int(K), int(out_format), _ptr(out), _stream(stream)))


def lb_dequantize_q2_0_g64(codes, scales, N: int, K: int, out_format: int, out, stream=None):
    _check("lb_dequantize_q2_0_g64", load().lb_dequantize_q2_0_g64(
        _ptr(codes), _ptr(scales), int(N), int(K), int(out_format), _ptr(out), _stream(stream)))


def lb_dequantize_trit_planes(planes, w_scale: float, N: int, K: int, out_format: int, out,
                              stream=None):
    _check("lb_dequantize_trit_planes", load().lb_dequantize_trit_planes(
        _ptr(planes), float(w_scale), int(N), int(K), int(out_format), _ptr(out),
        _stream(stream)))


def base3_row_bytes(K: int) -> int:
    """Bytes per base-3 packed row (LB_BASE3_ROW_BYTES): ceil(K / 80) groups of 16."""
    return (int(K) + 79) // 80 * 16


def lb_pack_base3(planes, N: int, K: int, packed, stream=None):
    _check("lb_pack_base3", load().lb_pack_base3(_ptr(planes), int(N), int(K), _ptr(packed),
                                                 _stream(stream)))


def lb_gemv_base3(packed, w_scale: float, q, x_scale, y, acc, N: int, K: int, B: int,
                  stream=None):
    _check("lb_gemv_base3", load().lb_gemv_base3(
        _ptr(packed), float(w_scale), _ptr(q), _ptr(x_scale), _ptr(y), _ptr(acc), int(N),
        int(K), int(B), _stream(stream)))
