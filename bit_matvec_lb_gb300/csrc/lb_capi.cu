// lb_capi.cu -- status names, version, device status, and the host helpers shared by every
// entry point (device check, error word, cached kernel preparation).
//
// Calls refuse with a reason and never fall back to another path: a device that is not
// compute capability 10.3 gets LB_ERR_ARCH (the pages' rule for kernel selection is the same:
// pin a kernel and error if the machine cannot run it, never fall back silently --
// tritium.technology "Architecture", section 4.2).
#include "lb_common.cuh"

#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <unordered_map>

namespace lb {

static thread_local int g_last_cuda_error = 0;

void record_cuda_error(cudaError_t e) {
    g_last_cuda_error = (int)e;
    cudaGetLastError();
}

static constexpr int kMaxDevices = 64;
static DeviceInfo g_info[kMaxDevices];
static std::mutex g_info_mutex;

int current_device_info(DeviceInfo *out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return LB_ERR_ARCH;
    }
    {
        std::lock_guard<std::mutex> lock(g_info_mutex);
        if (g_info[dev].ok < 0) {
            int major = 0, minor = 0, sms = 0;
            if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) !=
                    cudaSuccess ||
                cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                    cudaSuccess) {
                cudaGetLastError();
                return LB_ERR_ARCH;
            }
            g_info[dev].sms = sms;
            g_info[dev].ok = (major == 10 && minor == 3) ? 1 : 0;
        }
        *out = g_info[dev];
    }
    return out->ok == 1 ? LB_OK : LB_ERR_ARCH;
}

static std::atomic<int> g_injected_wait_us{0};

int take_injected_wait_fault() { return g_injected_wait_us.exchange(0); }

// One error word per device (file-scope device variable; the host passes its address).
__device__ int g_device_error;
static int *g_err_addr[kMaxDevices];

int *device_error_word() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_info_mutex);
    if (!g_err_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        g_err_addr[dev] = static_cast<int *>(p);
    }
    return g_err_addr[dev];
}

struct KernelPrep {
    bool attr_set = false;
    size_t smem = (size_t)-1;
    int threads = 0;
    int blocks_per_sm = 0;
};
static std::unordered_map<const void *, KernelPrep> g_prep;
static std::mutex g_prep_mutex;

int prepare_kernel(const void *kernel, int threads, size_t smem, int *blocks_per_sm) {
    std::lock_guard<std::mutex> lock(g_prep_mutex);
    KernelPrep &p = g_prep[kernel];
    if (!p.attr_set) {
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        // The dynamic limit plus the kernel's static shared memory may not exceed the opt-in
        // maximum.
        cudaFuncAttributes fa{};
        cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - (int)fa.sharedSizeBytes);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return LB_ERR_LAUNCH;
        }
        p.attr_set = true;
    }
    if (p.smem != smem || p.threads != threads) {
        int bps = 0;
        const cudaError_t e =
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bps, kernel, threads, smem);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return LB_ERR_LAUNCH;
        }
        p.smem = smem;
        p.threads = threads;
        p.blocks_per_sm = bps;
    }
    *blocks_per_sm = p.blocks_per_sm;
    return p.blocks_per_sm >= 1 ? LB_OK : LB_ERR_SHAPE;
}

static PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
static std::mutex g_encode_mutex;

int encode_rows_map(CUtensorMap *map, const void *base, uint64_t row_bytes, uint64_t rows,
                    uint32_t box_bytes, uint32_t box_rows, int swizzle_bytes) {
    {
        std::lock_guard<std::mutex> lock(g_encode_mutex);
        if (!g_encode_tiled) {
            void *fn = nullptr;
            cudaDriverEntryPointQueryResult q{};
            const cudaError_t e = cudaGetDriverEntryPointByVersion(
                "cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
            if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) {
                record_cuda_error(e != cudaSuccess ? e : cudaErrorSymbolNotFound);
                return LB_ERR_LAUNCH;
            }
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
    }
    const cuuint64_t dims[2] = {row_bytes, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_bytes, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode_tiled(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base),
                                      dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      swizzle_bytes == 64   ? CU_TENSOR_MAP_SWIZZLE_64B
                                      : swizzle_bytes == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                            : CU_TENSOR_MAP_SWIZZLE_NONE,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? LB_OK : LB_ERR_LAUNCH;
}

}  // namespace lb

LB_EXPORT int lb_last_cuda_error(void) {
    const int e = lb::g_last_cuda_error;
    lb::g_last_cuda_error = 0;
    return e;
}

LB_EXPORT const char *lb_cuda_error_name(int code) {
    return cudaGetErrorName(static_cast<cudaError_t>(code));
}

LB_EXPORT const char *lb_status_string(int status) {
    switch (status) {
        case LB_OK: return "LB_OK";
        case LB_ERR_NULL: return "LB_ERR_NULL";
        case LB_ERR_ALIGN: return "LB_ERR_ALIGN";
        case LB_ERR_SHAPE: return "LB_ERR_SHAPE";
        case LB_ERR_BATCH: return "LB_ERR_BATCH";
        case LB_ERR_ARCH: return "LB_ERR_ARCH";
        case LB_ERR_LAUNCH: return "LB_ERR_LAUNCH";
        case LB_ERR_DEVICE: return "LB_ERR_DEVICE";
    }
    return "LB_ERR_UNKNOWN";
}

LB_EXPORT int lb_version(void) { return 100; }

LB_EXPORT int lb_test_inject_wait_timeout(int wait_us) {
    if (wait_us < 1 || wait_us > 1000000) return LB_ERR_SHAPE;
    lb::g_injected_wait_us.store(wait_us);
    return LB_OK;
}

LB_EXPORT int lb_device_status(void *stream) {
    using namespace lb;
    DeviceInfo di;
    if (int st = current_device_info(&di)) return st;
    int *word = device_error_word();
    if (!word) return LB_ERR_LAUNCH;
    int host = 0;
    cudaStream_t s = as_stream(stream);
    if (cudaMemcpyAsync(&host, word, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(word, 0, sizeof(int), s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return LB_ERR_LAUNCH;
    return host == 0 ? LB_OK : LB_ERR_DEVICE;
}
