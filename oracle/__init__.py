"""CPU oracle for the packed low-bit products -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its ``cpu_baseline`` leg and
``--impl reference`` arm) may import this package.  The GPU library never imports it, and this
package imports nothing from the GPU library: the two share no code.

The arithmetic lives in ``lb_oracle.c`` (plain scalar C, floating-point contraction off); this
module compiles it with gcc on first use and wraps it for numpy arrays.  Each wrapper names the
page passage its C function follows.

Pages cited:
  [TR] "bankml: verified low-bit inference on commodity CPUs -- a technical report", III.2-III.8
  [BH] bankml BUILD_HISTORY.md, ledger item "P2 -- own the kernels"
  [TA] tritium.technology "Architecture", sections 1-5, 8
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "lb_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
CFLAGS = ["-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
          "-fvisibility=hidden", "-Wall"]

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile lb_oracle.c into oracle/_build/liboracle.so (gcc, contraction off).

    ``LB_ORACLE_SO`` names a prebuilt library instead; the mutation test uses it to load
    deliberately broken copies of the oracle."""
    alt = os.environ.get("LB_ORACLE_SO")
    if alt:
        return alt
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
        os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            I64 = ctypes.c_int64
            sig = {
                "oracle_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_bf16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
                "oracle_quantize_q8_0": (ctypes.c_int, [P, I64, I64, P, P]),
                "oracle_quantize_i8_absmax": (ctypes.c_int, [P, I64, I64, P, P]),
                "oracle_q1_0_product": (None, [P, P, P, I64, I64, I64, P, P, P, P]),
                "oracle_q2_0_g64_product": (None, [P, P, P, I64, I64, I64, P, P, P, P]),
                "oracle_trit_planes_product": (ctypes.c_int, [P, ctypes.c_float, P, P, I64, I64,
                                                              I64, P, P]),
                "oracle_bf16_product": (None, [P, P, I64, I64, I64, P, P]),
                "oracle_repack": (None, [P, I64, I64, P, P]),
                "oracle_dequant": (None, [ctypes.c_int, P, I64, I64, P]),
                "oracle_f32_to_bf16": (ctypes.c_uint16, [ctypes.c_float]),
                "oracle_f32_to_bf16_array": (None, [P, I64, P]),
                "oracle_trit_planes_dequant": (ctypes.c_int, [P, ctypes.c_float, I64, I64, P]),
                "oracle_base3_pack": (ctypes.c_int, [P, I64, I64, P]),
                "oracle_base3_product": (ctypes.c_int, [P, ctypes.c_float, P, P, I64, I64, I64,
                                                        P, P]),
                "oracle_base3_unpack": (None, [P, I64, I64, P]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(lib, name)
                fn.restype = res
                fn.argtypes = args
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


# --------------------------------------------------------------------------------------------
# scalar conversions ([TR] III.2: fp16 scales; [TA] 3: bf16 head)
# --------------------------------------------------------------------------------------------
def f16_to_f32(h: int) -> float:
    return _load().oracle_f16_to_f32(int(h) & 0xFFFF)


def f32_to_f16(f: float) -> int:
    return _load().oracle_f32_to_f16(float(np.float32(f)))


def bf16_to_f32(b: int) -> float:
    return _load().oracle_bf16_to_f32(int(b) & 0xFFFF)


def f16_bits_to_f32_array(h: np.ndarray) -> np.ndarray:
    lib = _load()
    flat = np.ascontiguousarray(h, dtype=np.uint16).ravel()
    return np.array([lib.oracle_f16_to_f32(int(v)) for v in flat], dtype=np.float32).reshape(h.shape)


# --------------------------------------------------------------------------------------------
# activation quantizers
# --------------------------------------------------------------------------------------------
def quantize_q8_0(x: np.ndarray):
    """q8_0 per 32 values ([TR] III.2, [BH]): d = fp16(amax/127), q = rne(x * 127/amax).

    x: float32 [B][K], K % 32 == 0.  Returns (q int8 [B][K], d uint16 fp16-bits [B][K/32]).
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    B, K = x.shape
    assert K % 32 == 0
    q = np.empty((B, K), dtype=np.int8)
    d = np.empty((B, K // 32), dtype=np.uint16)
    rc = _load().oracle_quantize_q8_0(_ptr(x), B, K, _ptr(q), _ptr(d))
    assert rc == 0, "q8_0 code outside [-127, 127]"
    return q, d


def quantize_i8_absmax(x: np.ndarray):
    """Per-token absmax int8 (reading R7): returns (q int8 [B][K], x_scale float32 [B])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    B, K = x.shape
    q = np.empty((B, K), dtype=np.int8)
    s = np.empty((B,), dtype=np.float32)
    _load().oracle_quantize_i8_absmax(_ptr(x), B, K, _ptr(q), _ptr(s))
    return q, s


# --------------------------------------------------------------------------------------------
# products
# --------------------------------------------------------------------------------------------
class QResult:
    """Result of a Q1_0 / Q2_0_g64 product: isum [B][N][K/32] int32, y_exact [B][N] float64,
    y_chain [B][N] float32 (fp32 chain of [TR] III.3) and mag [B][N] = sum |d_w d_x isum|."""

    def __init__(self, isum, y_exact, y_chain, mag):
        self.isum, self.y_exact, self.y_chain, self.mag = isum, y_exact, y_chain, mag

    def tolerance(self, rel: float = 1e-5, abs_: float = 1e-6) -> np.ndarray:
        """|y - y_exact| bound: rel * sum_blocks |d_w d_x isum| + abs_."""
        return rel * self.mag + abs_


def _q_product(fn_name: str, qk: int, blocks: np.ndarray, q: np.ndarray, dx: np.ndarray,
               want_isum: bool = True) -> QResult:
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    dx = np.ascontiguousarray(dx, dtype=np.uint16)
    if q.ndim == 1:
        q = q[None, :]
        dx = dx[None, :]
    B, K = q.shape
    N = blocks.shape[0]
    assert blocks.size == N * (K // qk) * 18, "blocks must be [N][K/QK][18]"
    isum = np.empty((B, N, K // 32), dtype=np.int32) if want_isum else None
    y_exact = np.empty((B, N), dtype=np.float64)
    y_chain = np.empty((B, N), dtype=np.float32)
    mag = np.empty((B, N), dtype=np.float64)
    getattr(_load(), fn_name)(_ptr(blocks), _ptr(q), _ptr(dx), N, K, B, _ptr(isum),
                              _ptr(y_exact), _ptr(y_chain), _ptr(mag))
    return QResult(isum, y_exact, y_chain, mag)


def q1_0_product(blocks, q, dx, want_isum=True) -> QResult:
    """Q1_0 x q8_0 ([TR] III.2-III.3): blocks [N][K/128][18] source bytes."""
    return _q_product("oracle_q1_0_product", 128, blocks, q, dx, want_isum)


def q2_0_g64_product(blocks, q, dx, want_isum=True) -> QResult:
    """Q2_0_g64 x q8_0 ([TR] III.5, III.8): blocks [N][K/64][18] source bytes."""
    return _q_product("oracle_q2_0_g64_product", 64, blocks, q, dx, want_isum)


def trit_planes_product(planes: np.ndarray, w_scale: float, q: np.ndarray, x_scale: np.ndarray):
    """Planar ternary ([TA] 1, 2, 4.1, 5): planes [N][K/64][2] uint64 {pos, neg}.

    Returns (acc int32 [B][N], y float32 [B][N]); raises on an overlapping beat."""
    planes = np.ascontiguousarray(planes, dtype=np.uint64)
    q = np.ascontiguousarray(q, dtype=np.int8)
    if q.ndim == 1:
        q = q[None, :]
    x_scale = np.ascontiguousarray(np.atleast_1d(x_scale), dtype=np.float32)
    B, K = q.shape
    N = planes.shape[0]
    assert planes.size == N * (K // 64) * 2
    acc = np.empty((B, N), dtype=np.int32)
    y = np.empty((B, N), dtype=np.float32)
    rc = _load().oracle_trit_planes_product(_ptr(planes), float(np.float32(w_scale)), _ptr(q),
                                            _ptr(x_scale), N, K, B, _ptr(acc), _ptr(y))
    if rc == -1:
        raise ValueError("planar beat with a column in both the pos and neg planes")
    if rc == -2:
        raise OverflowError("planar accumulator outside int32")
    return acc, y


def bf16_product(w: np.ndarray, x: np.ndarray):
    """Dense bf16 head (reading R8): w uint16 bf16-bits [N][K], x float32 [B][K].

    Returns (y_exact float64 [B][N], mag float64 [B][N] = sum |w x|)."""
    w = np.ascontiguousarray(w, dtype=np.uint16)
    x = np.ascontiguousarray(x, dtype=np.float32)
    if x.ndim == 1:
        x = x[None, :]
    B, K = x.shape
    N = w.shape[0]
    y = np.empty((B, N), dtype=np.float64)
    mag = np.empty((B, N), dtype=np.float64)
    _load().oracle_bf16_product(_ptr(w), _ptr(x), N, K, B, _ptr(y), _ptr(mag))
    return y, mag


def scale_stride(K: int, qk: int) -> int:
    """Row stride (in entries) of the repacked scale plane: K/QK rounded up to a multiple of 8."""
    return (K // qk + 7) // 8 * 8


def repack(blocks: np.ndarray, K: int, qk: int):
    """Split [N][K/QK][18] blocks into (bits uint8 [N][K/QK*16], scales uint16 [N][S]) with
    S = scale_stride(K, qk); scale entries past K/QK are zero padding."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    N = blocks.shape[0]
    nblk = K // qk
    bits = np.empty((N, nblk * 16), dtype=np.uint8)
    scales = np.empty((N, scale_stride(K, qk)), dtype=np.uint16)
    _load().oracle_repack(_ptr(blocks), N, nblk, _ptr(bits), _ptr(scales))
    return bits, scales


def dequant(blocks: np.ndarray, K: int, qk: int) -> np.ndarray:
    """Every weight as float32 w * d, [N][K] ([TR] III.2, III.5)."""
    blocks = np.ascontiguousarray(blocks, dtype=np.uint8)
    N = blocks.shape[0]
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant(qk, _ptr(blocks), N, K, _ptr(out))
    return out


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """binary32 -> bf16 bit patterns, round to nearest, ties to even (reading R10)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().oracle_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


def dequant_bf16(blocks: np.ndarray, K: int, qk: int) -> np.ndarray:
    """Every weight as bf16 bits of the binary32 w * d, [N][K] (reading R10)."""
    return f32_to_bf16(dequant(blocks, K, qk))


def trit_planes_dequant(planes: np.ndarray, w_scale: float, K: int) -> np.ndarray:
    """Planar weights as float32 w * w_scale, [N][K] (readings R5, R10); raises on an
    overlapping beat."""
    planes = np.ascontiguousarray(planes, dtype=np.uint64)
    N = planes.shape[0]
    assert planes.size == N * (K // 64) * 2
    out = np.empty((N, K), dtype=np.float32)
    if _load().oracle_trit_planes_dequant(_ptr(planes), float(np.float32(w_scale)), N, K,
                                          _ptr(out)) == -1:
        raise ValueError("planar beat with a column in both the pos and neg planes")
    return out


def base3_row_bytes(K: int) -> int:
    """Bytes per base-3 packed row: ceil(K / 80) groups of 16 bytes (reading R15)."""
    return (K + 79) // 80 * 16


def base3_pack(planes: np.ndarray, K: int) -> np.ndarray:
    """Planar beats [N][K/64][2] -> base-3 bytes [N][base3_row_bytes(K)] ([TR] III.8, R15)."""
    planes = np.ascontiguousarray(planes, dtype=np.uint64)
    N = planes.shape[0]
    out = np.empty((N, base3_row_bytes(K)), dtype=np.uint8)
    if _load().oracle_base3_pack(_ptr(planes), N, K, _ptr(out)) == -1:
        raise ValueError("planar beat with a column in both the pos and neg planes")
    return out


def base3_unpack(packed: np.ndarray, K: int) -> np.ndarray:
    """Base-3 bytes -> trits int8 [N][K] (R15)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    N = packed.shape[0]
    out = np.empty((N, K), dtype=np.int8)
    _load().oracle_base3_unpack(_ptr(packed), N, K, _ptr(out))
    return out


def base3_product(packed: np.ndarray, w_scale: float, q: np.ndarray, x_scale: np.ndarray):
    """Base-3 packed ternary x int8 (R6, R7, R15). Returns (acc int32 [B][N], y float32)."""
    packed = np.ascontiguousarray(packed, dtype=np.uint8)
    q = np.ascontiguousarray(q, dtype=np.int8)
    if q.ndim == 1:
        q = q[None, :]
    x_scale = np.ascontiguousarray(np.atleast_1d(x_scale), dtype=np.float32)
    B, K = q.shape
    N = packed.shape[0]
    assert packed.shape[1] == base3_row_bytes(K)
    acc = np.empty((B, N), dtype=np.int32)
    y = np.empty((B, N), dtype=np.float32)
    rc = _load().oracle_base3_product(_ptr(packed), float(np.float32(w_scale)), _ptr(q),
                                      _ptr(x_scale), N, K, B, _ptr(acc), _ptr(y))
    if rc == -1:
        raise ValueError("byte above 242 in a base-3 packed matrix")
    if rc == -2:
        raise OverflowError("accumulator outside int32")
    return acc, y
