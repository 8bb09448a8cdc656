"""The C-ABI library builds for sm_103a, loads, exports every entry point include/lb.h declares,
and refuses bad arguments on the host before touching the device (no GPU needed)."""
import ctypes
import os
import re

import pytest

import bit_matvec_lb_gb300 as lb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]


def declared_symbols():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names.update(re.findall(r"\b(lb_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    return lb.load()


def test_header_declares_entry_points():
    names = declared_symbols()
    for expected in ("lb_quantize_q8_0", "lb_repack_q1_0", "lb_repack_q2_0_g64",
                     "lb_gemv_q1_0", "lb_gemv_q2_0_g64", "lb_gemv_trit_planes", "lb_gemv_bf16",
                     "lb_status_string"):
        assert expected in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_symbols() if not hasattr(lib, n)]
    assert not missing, f"declared in include/*.h but not exported: {missing}"


def test_binding_names_match_header():
    for n in declared_symbols():
        if n in ("lb_status_string", "lb_version"):
            continue
        assert hasattr(lb, n), f"python binding lacks {n}"
        assert n in lb.SIGNATURES


def test_status_strings(lib):
    for code, name in lb.LB_STATUS.items():
        assert lib.lb_status_string(code).decode() == name
    assert lib.lb_status_string(12345).decode() == "LB_ERR_UNKNOWN"
    assert lib.lb_version() >= 100


def test_cuda_error_query(lib):
    assert lib.lb_last_cuda_error() == 0          # nothing failed on this thread
    assert lib.lb_cuda_error_name(0).decode() == "cudaSuccess"
    assert lb.lb_cuda_error_name(1) == "cudaErrorInvalidValue"


# Host-side refusals: these return before any CUDA call, so they run without a GPU.
A = 0x10000          # 16-byte aligned fake device address (never dereferenced)
MIS = 0x10008        # misaligned


def test_refuse_null(lib):
    assert lib.lb_gemv_q1_0(None, A, A, A, A, None, 4, 128, 1, None) == -1
    assert lib.lb_gemv_q2_0_g64(A, A, A, A, None, None, 4, 64, 1, None) == -1
    assert lib.lb_gemv_trit_planes(A, 1.0, A, None, A, None, 4, 64, 1, None) == -1
    assert lib.lb_gemv_bf16(A, None, A, 4, 8, 1, None) == -1
    assert lib.lb_quantize_q8_0(A, None, A, 1, 32, None) == -1
    assert lib.lb_repack_q1_0(None, 1, 128, A, A, None) == -1


def test_refuse_misaligned(lib):
    assert lib.lb_gemv_q1_0(MIS, A, A, A, A, None, 4, 128, 1, None) == -2
    assert lib.lb_gemv_q2_0_g64(A, A, A, A, A, MIS, 4, 64, 1, None) == -2
    assert lib.lb_gemv_trit_planes(A, 1.0, A, A, MIS, None, 4, 64, 1, None) == -2
    assert lib.lb_gemv_bf16(A, A, MIS, 4, 8, 1, None) == -2
    assert lib.lb_quantize_q8_0(MIS, A, A, 1, 32, None) == -2


@pytest.mark.parametrize("K", [0, 64, 192, 100])
def test_refuse_q1_shape(lib, K):
    assert lib.lb_gemv_q1_0(A, A, A, A, A, None, 4, K, 1, None) == -3


def test_refuse_other_shapes(lib):
    assert lib.lb_gemv_q2_0_g64(A, A, A, A, A, None, 4, 96, 1, None) == -3
    assert lib.lb_gemv_q2_0_g64(A, A, A, A, A, None, 0, 64, 1, None) == -3
    assert lib.lb_gemv_trit_planes(A, 1.0, A, A, A, None, 4, 32, 1, None) == -3
    assert lib.lb_gemv_trit_planes(A, 1.0, A, A, A, None, 4, 262144, 1, None) == -3
    assert lib.lb_gemv_bf16(A, A, A, 4, 12, 1, None) == -3
    assert lib.lb_quantize_q8_0(A, A, A, 1, 48, None) == -3
    assert lib.lb_quantize_q8_0(A, A, A, 0, 32, None) == -3
    assert lib.lb_repack_q2_0_g64(A, 2, 100, A, A, None) == -3


@pytest.mark.parametrize("B", [0, 9, -1])
def test_refuse_batch(lib, B):
    assert lib.lb_gemv_q1_0(A, A, A, A, A, None, 4, 128, B, None) == -4
    assert lib.lb_gemv_q2_0_g64(A, A, A, A, A, None, 4, 64, B, None) == -4
    assert lib.lb_gemv_trit_planes(A, 1.0, A, A, A, None, 4, 64, B, None) == -4
    assert lib.lb_gemv_bf16(A, A, A, 4, 8, B, None) == -4


def test_refuse_without_sm103(lib):
    """Valid arguments on a machine whose current device is not an sm_103 GPU (or that has
    no GPU at all) are refused with LB_ERR_ARCH -- there is no fallback path."""
    import torch
    if torch.cuda.is_available():
        major, minor = torch.cuda.get_device_capability()
        if (major, minor) == (10, 3):
            pytest.skip("an sm_103 device is present")
    assert lib.lb_gemv_q1_0(A, A, A, A, A, None, 4, 128, 1, None) == -5


def test_python_binding_raises_on_error():
    with pytest.raises(lb.LBError) as e:
        lb.lb_gemv_bf16(A, A, A, 4, 12, 1, stream=0)
    assert e.value.status == -3 and "LB_ERR_SHAPE" in str(e.value)


def test_grouped_refusals(lib):
    arr = (lb.lb_q_matrix * 2)()
    arr[0] = lb.lb_q_matrix(A, A, A, None, 4)
    arr[1] = lb.lb_q_matrix(A, A, A, None, 4)
    assert lib.lb_gemv_q2_0_g64_grouped(arr, 0, A, A, 64, 1, None) == -3      # empty group
    assert lib.lb_gemv_q2_0_g64_grouped(arr, 65, A, A, 64, 1, None) == -3     # too many
    arr[1] = lb.lb_q_matrix(A, None, A, None, 4)
    assert lib.lb_gemv_q2_0_g64_grouped(arr, 2, A, A, 64, 1, None) == -1      # NULL scales
    arr[1] = lb.lb_q_matrix(A, A, MIS, None, 4)
    assert lib.lb_gemv_q1_0_grouped(arr, 2, A, A, 128, 1, None) == -2         # misaligned y
    arr[1] = lb.lb_q_matrix(A, A, A, None, 0)
    assert lib.lb_gemv_q1_0_grouped(arr, 2, A, A, 128, 1, None) == -3         # N = 0
    t = (lb.lb_trit_matrix * 1)()
    t[0] = lb.lb_trit_matrix(A, 1.0, A, None, 4)
    assert lib.lb_gemv_trit_planes_grouped(t, 1, A, A, 64, 9, None) == -4


@pytest.mark.parametrize("fn,qk", [("lb_gemm_q1_0_grouped", 128), ("lb_gemm_q2_0_g64_grouped", 64)])
def test_gemm_grouped_refusals(lib, fn, qk):
    f = getattr(lib, fn)
    K = 4 * qk
    ws = lib.lb_gemm_workspace_bytes(16, K)
    arr = (lb.lb_gemm_matrix * 9)()
    for i in range(9):
        arr[i] = lb.lb_gemm_matrix(A, A, A, 8)
    assert f(arr, 0, A, A, 16, K, A, ws, None) == -3      # empty group
    assert f(arr, 9, A, A, 16, K, A, ws, None) == -3      # more than LB_GEMM_MAX_GROUP
    assert f(None, 2, A, A, 16, K, A, ws, None) == -1
    assert f(arr, 2, None, A, 16, K, A, ws, None) == -1
    assert f(arr, 2, A, A, 16, K, None, ws, None) == -1
    assert f(arr, 2, MIS, A, 16, K, A, ws, None) == -2
    assert f(arr, 2, A, A, 16, K + 32, A, ws, None) == -3
    assert f(arr, 2, A, A, 16, K, A, ws - 1, None) == -3  # workspace one byte short
    arr[1] = lb.lb_gemm_matrix(A, None, A, 8)
    assert f(arr, 2, A, A, 16, K, A, ws, None) == -1      # NULL scales of matrix 1
    arr[1] = lb.lb_gemm_matrix(A, A, MIS, 8)
    assert f(arr, 2, A, A, 16, K, A, ws, None) == -2      # misaligned y of matrix 1
    arr[1] = lb.lb_gemm_matrix(A, A, A, 0)
    assert f(arr, 2, A, A, 16, K, A, ws, None) == -3      # N = 0


def test_scale_stride():
    assert lb.scale_stride(512, 128) == 8 and lb.scale_stride(4096, 64) == 64
    assert lb.scale_stride(4224, 128) == 40 and lb.scale_stride(320, 64) == 8


# ---- prefill GEMM: host checks ----
def test_gemm_workspace_bytes(lib):
    assert lib.lb_gemm_workspace_bytes(0, 128) == 0
    assert lib.lb_gemm_workspace_bytes(1, 0) == 0
    # tokens are rounded up to tiles of 128; two bytes per converted code
    assert lib.lb_gemm_workspace_bytes(1, 128) == 128 * 128 * 2
    assert lib.lb_gemm_workspace_bytes(128, 4096) == 128 * 4096 * 2
    assert lib.lb_gemm_workspace_bytes(129, 4096) == 256 * 4096 * 2
    assert lb.lb_gemm_workspace_bytes(512, 12288) == 512 * 12288 * 2


@pytest.mark.parametrize("fn,qk", [("lb_gemm_q1_0", 128), ("lb_gemm_q2_0_g64", 64)])
def test_gemm_refusals(lib, fn, qk):
    f = getattr(lib, fn)
    ws = lib.lb_gemm_workspace_bytes(16, 4 * qk)
    ok = (A, A, A, A, A, 16, 8, 4 * qk, A, ws, None)
    for i in (0, 1, 2, 3, 4, 8):
        args = list(ok)
        args[i] = None
        assert f(*args) == -1
    for i in (0, 1, 2, 3, 4, 8):
        args = list(ok)
        args[i] = MIS
        assert f(*args) == -2
    bad_shapes = [(0, 8, 4 * qk), (16, 0, 4 * qk), (16, 8, qk // 2), (16, 8, 4 * qk + 32),
                  (16, 8, 0), (2**31, 8, 4 * qk)]
    for M, N, K in bad_shapes:
        assert f(A, A, A, A, A, M, N, K, A, 2**40, None) == -3
    # workspace one byte short
    assert f(A, A, A, A, A, 16, 8, 4 * qk, A, ws - 1, None) == -3


# ---- planar prefill GEMM: host checks ----
def test_gemm_trit_workspace_bytes(lib):
    assert lib.lb_gemm_trit_workspace_bytes(0, 64) == 0
    assert lib.lb_gemm_trit_workspace_bytes(1, 0) == 0
    # the activation tiles of the Q GEMMs, nothing else
    for M, K in ((1, 64), (130, 2560), (512, 6912)):
        assert lib.lb_gemm_trit_workspace_bytes(M, K) == lib.lb_gemm_workspace_bytes(M, K)


def test_gemm_trit_refusals(lib):
    f = lib.lb_gemm_trit_planes
    K = 256
    ws = lib.lb_gemm_trit_workspace_bytes(16, K)
    ok = [A, 1.0, A, A, A, None, 16, 8, K, A, ws, None]
    for i in (0, 2, 3, 4, 9):
        args = list(ok)
        args[i] = None
        assert f(*args) == -1
    for i in (0, 2, 3, 4, 5, 9):
        args = list(ok)
        args[i] = MIS
        assert f(*args) == -2
    for M, N, KK in ((0, 8, K), (16, 0, K), (16, 8, 32), (16, 8, K + 32), (16, 8, 0),
                     (2**31, 8, K), (16, 8, (1 << 24) // 128 + 64)):
        assert f(A, 1.0, A, A, A, None, M, N, KK, A, 2**40, None) == -3
    assert f(A, 1.0, A, A, A, None, 16, 8, K, A, ws - 1, None) == -3   # workspace short
    g = lib.lb_gemm_trit_planes_grouped
    arr = (lb.lb_trit_matrix * 9)()
    for i in range(9):
        arr[i] = lb.lb_trit_matrix(A, 1.0, A, None, 8)
    assert g(arr, 0, A, A, 16, K, A, ws, None) == -3      # empty group
    assert g(arr, 9, A, A, 16, K, A, ws, None) == -3      # more than LB_GEMM_MAX_GROUP
    arr[1] = lb.lb_trit_matrix(None, 1.0, A, None, 8)
    assert g(arr, 2, A, A, 16, K, A, ws, None) == -1      # NULL planes of matrix 1
    arr[1] = lb.lb_trit_matrix(A, 1.0, A, MIS, 8)
    assert g(arr, 2, A, A, 16, K, A, ws, None) == -2      # misaligned acc of matrix 1
    arr[1] = lb.lb_trit_matrix(A, 1.0, A, None, 0)
    assert g(arr, 2, A, A, 16, K, A, ws, None) == -3      # N = 0


def test_quantize_tiles_and_pretiled_gemm_refusals(lib):
    """The quantize-then-GEMM pair refuses on the host before anything is enqueued."""
    f = lib.lb_quantize_i8_absmax_tiles
    K = 256
    ws = lib.lb_gemm_trit_workspace_bytes(16, K)
    ok = [A, A, A, 16, K, A, ws, None]
    for i in (0, 1, 2, 5):
        args = list(ok)
        args[i] = None
        assert f(*args) == -1
        args[i] = MIS
        assert f(*args) == -2
    for M, KK in ((0, K), (2**31, K), (16, 32), (16, K + 16), (16, 0),
                  (16, (1 << 24) // 128 + 64)):
        assert f(A, A, A, M, KK, A, 2**40, None) == -3
    assert f(A, A, A, 16, K, A, ws - 1, None) == -3       # workspace short
    g = lib.lb_gemm_trit_planes_grouped_tiles
    arr = (lb.lb_trit_matrix * 9)()
    for i in range(9):
        arr[i] = lb.lb_trit_matrix(A, 1.0, A, None, 8)
    assert g(None, 1, A, 16, K, A, ws, None) == -1        # no matrices
    assert g(arr, 1, None, 16, K, A, ws, None) == -1      # no x_scale
    assert g(arr, 1, A, 16, K, None, ws, None) == -1      # no workspace
    assert g(arr, 1, MIS, 16, K, A, ws, None) == -2
    assert g(arr, 0, A, 16, K, A, ws, None) == -3         # empty group
    assert g(arr, 9, A, 16, K, A, ws, None) == -3         # more than LB_GEMM_MAX_GROUP
    assert g(arr, 1, A, 16, K + 32, A, 2**40, None) == -3  # K % 64
    assert g(arr, 1, A, 16, K, A, ws - 1, None) == -3     # workspace short


# ---- dequantization: host checks ----
@pytest.mark.parametrize("fn,qk", [("lb_dequantize_q1_0", 128), ("lb_dequantize_q2_0_g64", 64)])
def test_dequant_refusals(lib, fn, qk):
    f = getattr(lib, fn)
    assert f(None, A, 4, qk, 0, A, None) == -1
    assert f(A, None, 4, qk, 0, A, None) == -1
    assert f(A, A, 4, qk, 0, None, None) == -1
    assert f(MIS, A, 4, qk, 0, A, None) == -2
    assert f(A, A, 4, qk, 1, MIS, None) == -2
    assert f(A, A, 4, qk // 2, 0, A, None) == -3
    assert f(A, A, 0, qk, 0, A, None) == -3
    assert f(A, A, 4, qk, 2, A, None) == -3      # unknown output format
    assert f(A, A, 4, qk, -1, A, None) == -3


def test_dequant_trit_refusals(lib):
    f = lib.lb_dequantize_trit_planes
    assert f(None, 1.0, 4, 64, 0, A, None) == -1
    assert f(A, 1.0, 4, 64, 0, MIS, None) == -2
    assert f(A, 1.0, 4, 96, 0, A, None) == -3
    assert f(A, 1.0, 4, 64, 3, A, None) == -3


# ---- base-3 packing: host checks ----
def test_base3_refusals(lib):
    assert lib.lb_pack_base3(None, 4, 64, A, None) == -1
    assert lib.lb_pack_base3(A, 4, 64, MIS, None) == -2
    assert lib.lb_pack_base3(A, 4, 96, A, None) == -3
    assert lib.lb_pack_base3(A, 0, 64, A, None) == -3
    g = lib.lb_gemv_base3
    assert g(None, 1.0, A, A, A, None, 4, 64, 1, None) == -1
    assert g(A, 1.0, A, A, MIS, None, 4, 64, 1, None) == -2
    assert g(A, 1.0, A, A, A, MIS, 4, 64, 1, None) == -2
    assert g(A, 1.0, A, A, A, None, 4, 80, 1, None) == -3
    assert g(A, 1.0, A, A, A, None, 4, 64, 0, None) == -4
    assert g(A, 1.0, A, A, A, None, 4, 64, 9, None) == -4
    # 8 tokens of 32768 columns: 8 * 410 * 80 bytes of activation image exceed the limit
    assert g(A, 1.0, A, A, A, None, 4, 32768, 8, None) == -3
    assert lb.base3_row_bytes(2560) == 512 and lb.base3_row_bytes(6912) == 1392


def test_injected_wait_limit_is_range_checked(lib):
    # the failure-detection hook refuses limits outside [1 us, 1 s] on the host
    assert lib.lb_test_inject_wait_timeout(0) == -3
    assert lib.lb_test_inject_wait_timeout(2_000_000) == -3
    assert lib.lb_test_inject_wait_timeout(-5) == -3
