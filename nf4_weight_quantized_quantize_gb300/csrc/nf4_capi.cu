// nf4_capi.cu -- the extern "C" front end of libnf4 (declared in include/nf4.h).
//
// Validates arguments on the host, picks the kernel path and enqueues it on
// the caller's stream.  Per device it keeps the device properties and the
// address of a 4-byte error word that kernels set when a bounded wait gives
// up (or, in the checked build, when an index falls outside its buffer).  Nothing here allocates device memory.
#include <atomic>
#include <mutex>

#include "../../include/nf4.h"
#include "nf4_launch.h"

namespace {

constexpr int kMaxDevices = 64;

// One error word per device (a __device__ variable exists once per device
// that loads the module).
__device__ uint32_t g_err_word;

struct State {
    std::mutex mu;
    nf4::DeviceInfo dev[kMaxDevices];
    bool ready[kMaxDevices] = {};
};

State& state() {
    static State s;
    return s;
}

// Current device's info, initialised once: checks for sm_103 and resolves the
// error word's device address with that device current.
nf4_status current_device(const nf4::DeviceInfo** out) {
    int ord = -1;
    if (cudaGetDevice(&ord) != cudaSuccess || ord < 0 || ord >= kMaxDevices) {
        cudaGetLastError();
        return NF4_ERR_DEVICE;
    }
    State& st = state();
    std::lock_guard<std::mutex> lock(st.mu);
    if (!st.ready[ord]) {
        nf4::DeviceInfo d;
        d.ordinal = ord;
        int smem = 0;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, ord) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, ord) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, ord) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, ord) != cudaSuccess) {
            cudaGetLastError();
            return NF4_ERR_DEVICE;
        }
        if (d.cc_major != 10 || d.cc_minor != 3) return NF4_ERR_DEVICE;
        d.smem_optin = static_cast<size_t>(smem);
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) {
            cudaGetLastError();
            return NF4_ERR_CUDA;
        }
        d.err_word = static_cast<uint32_t*>(p);
        st.dev[ord] = d;
        st.ready[ord] = true;
    }
    *out = &st.dev[ord];
    return NF4_OK;
}

inline bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

std::atomic<uint64_t> g_launches{0};

}  // namespace

void nf4::count_launches(int n) { g_launches.fetch_add(static_cast<uint64_t>(n), std::memory_order_relaxed); }

int nf4::current_device_info(const nf4::DeviceInfo** out) { return current_device(out); }

namespace {

bool valid_dtype(int dt) { return dt == NF4_DTYPE_BF16 || dt == NF4_DTYPE_F16 || dt == NF4_DTYPE_F32; }
size_t elem_bytes(int dt) { return dt == NF4_DTYPE_F32 ? 4 : 2; }

// Host-side checks of nf4_linear_ex / nf4_linear_geglu_ex over a weight of
// `rows` rows; NF4_OK with *empty set when there is nothing to do.
nf4_status check_linear(const void* x, int dtype, int64_t M, int64_t K, const uint8_t* packed, const float* absmax,
                        int64_t rows, int32_t block, const void* y, void* workspace, size_t workspace_bytes,
                        bool* empty) {
    *empty = false;
    if (block != NF4_BLOCK) return NF4_ERR_BLOCKSIZE;
    if (!valid_dtype(dtype)) return NF4_ERR_DTYPE;
    if (M < 0 || rows < 0 || K <= 0 || K % NF4_BLOCK != 0) return NF4_ERR_SHAPE;
    // TMA coordinates are 32-bit: keep every extent below 2^31.
    if (M >= (int64_t(1) << 31) || rows >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return NF4_ERR_SHAPE;
    if (M == 0 || rows == 0) {
        *empty = true;
        return NF4_OK;
    }
    if (!x || !packed || !absmax || !y) return NF4_ERR_NULL;
    if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(y, 16) || !aligned(absmax, 4)) return NF4_ERR_ALIGN;
    size_t need = 0;
    nf4_linear_workspace_size(M, rows, K, &need);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return NF4_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return NF4_ERR_ALIGN;
    }
    return NF4_OK;
}

}  // namespace

extern "C" {

nf4_status nf4_quantize_ex(const void* w, nf4_dtype dtype, int64_t numel, int32_t block, uint8_t* packed,
                           float* absmax, void* stream) {
    if (block != NF4_BLOCK) return NF4_ERR_BLOCKSIZE;
    if (!valid_dtype(dtype)) return NF4_ERR_DTYPE;
    if (numel < 0 || numel % 2 != 0) return NF4_ERR_SHAPE;
    if (numel == 0) return NF4_OK;
    if (!w || !packed || !absmax) return NF4_ERR_NULL;
    if (!aligned(w, elem_bytes(dtype)) || !aligned(absmax, 4)) return NF4_ERR_ALIGN;
    const nf4::DeviceInfo* dev = nullptr;
    if (nf4_status st = current_device(&dev); st != NF4_OK) return st;
    cudaError_t e = nf4::launch_quantize(*dev, w, dtype, numel, packed, absmax, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

nf4_status nf4_quantize(const uint16_t* w, int64_t numel, int32_t block, uint8_t* packed,
                        float* absmax, void* stream) {
    return nf4_quantize_ex(w, NF4_DTYPE_BF16, numel, block, packed, absmax, stream);
}

nf4_status nf4_dequantize_ex(const uint8_t* packed, const float* absmax, int64_t numel, int32_t block,
                             nf4_dtype dtype, void* out, void* stream) {
    if (block != NF4_BLOCK) return NF4_ERR_BLOCKSIZE;
    if (!valid_dtype(dtype)) return NF4_ERR_DTYPE;
    if (numel < 0 || numel % 2 != 0) return NF4_ERR_SHAPE;
    if (numel == 0) return NF4_OK;
    if (!packed || !absmax || !out) return NF4_ERR_NULL;
    if (!aligned(out, elem_bytes(dtype)) || !aligned(absmax, 4)) return NF4_ERR_ALIGN;
    const nf4::DeviceInfo* dev = nullptr;
    if (nf4_status st = current_device(&dev); st != NF4_OK) return st;
    cudaError_t e =
        nf4::launch_dequantize(*dev, packed, absmax, numel, dtype, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

nf4_status nf4_dequantize(const uint8_t* packed, const float* absmax, int64_t numel, int32_t block,
                          uint16_t* out, void* stream) {
    return nf4_dequantize_ex(packed, absmax, numel, block, NF4_DTYPE_BF16, out, stream);
}

nf4_status nf4_linear_workspace_size(int64_t M, int64_t N, int64_t K, size_t* bytes) {
    if (!bytes) return NF4_ERR_NULL;
    if (M < 0 || N < 0 || K <= 0 || K % NF4_BLOCK != 0) return NF4_ERR_SHAPE;
    *bytes = (M > 0 && M < 128 && N > 0) ? nf4::skinny_workspace_bytes(nullptr, M, N, K) : 0;
    return NF4_OK;
}

nf4_status nf4_linear_ex(const void* x, nf4_dtype dtype, int64_t M, int64_t K, const uint8_t* packed,
                         const float* absmax, int64_t N, int32_t block, void* y, void* workspace,
                         size_t workspace_bytes, void* stream) {
    bool empty = false;
    if (nf4_status st = check_linear(x, dtype, M, K, packed, absmax, N, block, y, workspace, workspace_bytes, &empty);
        st != NF4_OK || empty)
        return st;
    const nf4::DeviceInfo* dev = nullptr;
    if (nf4_status st = current_device(&dev); st != NF4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = (M >= 128) ? nf4::launch_gemm(*dev, dtype, x, M, K, packed, absmax, N, y, s)
                               : nf4::launch_skinny(*dev, dtype, x, M, K, packed, absmax, N, y, workspace,
                                                    workspace_bytes, s);
    return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

nf4_status nf4_linear(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                      const float* absmax, int64_t N, int32_t block, uint16_t* y, void* workspace,
                      size_t workspace_bytes, void* stream) {
    return nf4_linear_ex(x, NF4_DTYPE_BF16, M, K, packed, absmax, N, block, y, workspace, workspace_bytes, stream);
}

nf4_status nf4_linear_geglu_ex(const void* x, nf4_dtype dtype, int64_t M, int64_t K, const uint8_t* packed,
                               const float* absmax, int64_t F, int32_t block, void* y, void* workspace,
                               size_t workspace_bytes, void* stream) {
    if (F >= (int64_t(1) << 30)) return NF4_ERR_SHAPE;   // 2F weight rows below 2^31
    bool empty = false;
    if (nf4_status st =
            check_linear(x, dtype, M, K, packed, absmax, 2 * F, block, y, workspace, workspace_bytes, &empty);
        st != NF4_OK || empty)
        return st;
    const nf4::DeviceInfo* dev = nullptr;
    if (nf4_status st = current_device(&dev); st != NF4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = (M >= 128) ? nf4::launch_gemm_geglu(*dev, dtype, x, M, K, packed, absmax, F, y, s)
                               : nf4::launch_skinny(*dev, dtype, x, M, K, packed, absmax, 2 * F, y, workspace,
                                                    workspace_bytes, s, true);
    return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

nf4_status nf4_linear_geglu(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                            const float* absmax, int64_t F, int32_t block, uint16_t* y, void* workspace,
                            size_t workspace_bytes, void* stream) {
    return nf4_linear_geglu_ex(x, NF4_DTYPE_BF16, M, K, packed, absmax, F, block, y, workspace, workspace_bytes,
                               stream);
}

nf4_status nf4_last_error(void* stream) {
    const nf4::DeviceInfo* dev = nullptr;
    if (nf4_status st = current_device(&dev); st != NF4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    const uint32_t zero = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess ||
        cudaMemcpyAsync(&word, dev->err_word, sizeof word, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(dev->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return NF4_ERR_CUDA;
    }
    if (word == 0) return NF4_OK;
    return (word >> 8) == (nf4::kErrBounds >> 8) ? NF4_ERR_BOUNDS : NF4_ERR_TIMEOUT;
}

const char* nf4_status_string(nf4_status status) {
    switch (status) {
        case NF4_OK: return "NF4_OK";
        case NF4_ERR_NULL: return "NF4_ERR_NULL";
        case NF4_ERR_SHAPE: return "NF4_ERR_SHAPE";
        case NF4_ERR_ALIGN: return "NF4_ERR_ALIGN";
        case NF4_ERR_BLOCKSIZE: return "NF4_ERR_BLOCKSIZE";
        case NF4_ERR_WORKSPACE: return "NF4_ERR_WORKSPACE";
        case NF4_ERR_DEVICE: return "NF4_ERR_DEVICE";
        case NF4_ERR_CUDA: return "NF4_ERR_CUDA";
        case NF4_ERR_TIMEOUT: return "NF4_ERR_TIMEOUT";
        case NF4_ERR_DTYPE: return "NF4_ERR_DTYPE";
        case NF4_ERR_BOUNDS: return "NF4_ERR_BOUNDS";
    }
    return "NF4_ERR_UNKNOWN";
}

int32_t nf4_version(void) { return 100; }

uint64_t nf4_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

}  // extern "C"
