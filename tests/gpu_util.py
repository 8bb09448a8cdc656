"""Helpers for the GPU parity tests: move numpy arrays to the device and call the C ABI."""
import numpy as np
import torch

import bit_matvec_lb_gb300 as lb

_VIEW = {np.dtype(np.uint16): np.int16, np.dtype(np.uint32): np.int32,
         np.dtype(np.uint64): np.int64}


# Every output buffer a test hands to the library sits between two bands of sentinel bytes;
# check_guards() (run after every test by the conftest fixture) fails if a kernel wrote into one.
GUARD_BYTES = 256
SENTINEL = 0xA5
_LIVE = []


def guarded(shape, dtype, fill=None) -> torch.Tensor:
    """Device tensor of `shape` and `dtype` (filled with `fill`, else a fixed byte pattern) with
    GUARD_BYTES of sentinel on both sides; its address stays 256-byte aligned."""
    if isinstance(shape, int):
        shape = (shape,)
    n = int(np.prod(shape)) if len(shape) else 1
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    raw = torch.full((2 * GUARD_BYTES + (nbytes + 255) // 256 * 256,), SENTINEL,
                     dtype=torch.uint8, device="cuda")
    body = raw[GUARD_BYTES:GUARD_BYTES + nbytes]
    if fill is None:
        body.fill_(0x5C)
    t = body.view(dtype).view(shape)
    if fill is not None:
        t.fill_(fill)
    _LIVE.append((raw, nbytes))
    return t


def check_guards():
    """Assert that no guard band of the buffers made by guarded() since the last call changed."""
    if not _LIVE:
        return
    torch.cuda.synchronize()
    bad = []
    for raw, nbytes in _LIVE:
        head = raw[:GUARD_BYTES]
        tail = raw[GUARD_BYTES + nbytes:]
        if not bool((head == SENTINEL).all()) or not bool((tail == SENTINEL).all()):
            bad.append(nbytes)
    _LIVE.clear()
    assert not bad, f"a kernel wrote outside its output buffer (buffers of {bad} bytes)"


def dev(a: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(a)
    if a.dtype in _VIEW:
        a = a.view(_VIEW[a.dtype])
    return torch.from_numpy(a).cuda()


def host(t: torch.Tensor, dtype=None) -> np.ndarray:
    a = t.detach().cpu().numpy()
    return a.view(dtype) if dtype is not None else a


def scale_stride(K: int, qk: int) -> int:
    return (K // qk + 7) // 8 * 8


def repack_on_gpu(blocks: np.ndarray, K: int, qk: int):
    N = blocks.shape[0]
    src = dev(blocks.reshape(-1))
    bits = guarded(N * (K // qk) * 16, torch.uint8)
    scales = guarded((N * scale_stride(K, qk),), torch.int16, 0x7FFF)
    fn = lb.lb_repack_q1_0 if qk == 128 else lb.lb_repack_q2_0_g64
    fn(src, N, K, bits, scales)
    return bits, scales


def gemv_q(qk: int, blocks: np.ndarray, q: np.ndarray, dx: np.ndarray, want_isum=True):
    """Run lb_gemv_q1_0 (qk=128) or lb_gemv_q2_0_g64 (qk=64); returns (y, isum or None)."""
    N = blocks.shape[0]
    B, K = q.shape
    bits, scales = repack_on_gpu(blocks, K, qk)
    y = guarded((B, N), torch.float32, float("nan"))
    isum = guarded((B, N, K // 32), torch.int32) if want_isum else None
    fn = lb.lb_gemv_q1_0 if qk == 128 else lb.lb_gemv_q2_0_g64
    fn(bits, scales, dev(q), dev(dx), y, isum, N, K, B)
    torch.cuda.synchronize()
    return host(y), (host(isum) if want_isum else None)


def gemv_trit(planes: np.ndarray, w_scale: float, q: np.ndarray, x_scale: np.ndarray):
    N = planes.shape[0]
    B, K = q.shape
    y = guarded((B, N), torch.float32, float("nan"))
    acc = guarded((B, N), torch.int32)
    lb.lb_gemv_trit_planes(dev(planes), w_scale, dev(q), dev(x_scale.astype(np.float32)), y, acc,
                           N, K, B)
    torch.cuda.synchronize()
    return host(acc), host(y)


def gemv_bf16(w: np.ndarray, x: np.ndarray):
    N, K = w.shape
    B = x.shape[0]
    y = guarded((B, N), torch.float32, float("nan"))
    lb.lb_gemv_bf16(dev(w), dev(x), y, N, K, B)
    torch.cuda.synchronize()
    return host(y)


def within(y, y_exact, mag, rel=1e-5, abs_=1e-6):
    err = np.abs(y.astype(np.float64) - y_exact)
    tol = rel * mag + abs_
    ok = err <= tol
    return bool(np.all(ok)), float(np.max(err / tol)) if err.size else 0.0


def gemm_q(qk: int, blocks: np.ndarray, q: np.ndarray, dx: np.ndarray, workspace=None,
           repacked=None):
    """Run lb_gemm_q1_0 (qk=128) or lb_gemm_q2_0_g64 (qk=64) over M = q.shape[0] tokens."""
    N = blocks.shape[0]
    M, K = q.shape
    bits, scales = repacked if repacked is not None else repack_on_gpu(blocks, K, qk)
    if workspace is None:
        workspace = guarded(lb.lb_gemm_workspace_bytes(M, K), torch.uint8)
    y = guarded((M, N), torch.float32, float("nan"))
    fn = lb.lb_gemm_q1_0 if qk == 128 else lb.lb_gemm_q2_0_g64
    fn(bits, scales, dev(q), dev(dx), y, M, N, K, workspace)
    torch.cuda.synchronize()
    return host(y)
