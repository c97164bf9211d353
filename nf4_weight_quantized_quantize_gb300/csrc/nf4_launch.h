// nf4_launch.h -- internal interface between the C ABI front end
// (nf4_capi.cu) and the kernel launchers.  Not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda_runtime.h>

namespace nf4 {

// Launch `kernel` with programmatic dependent launch allowed: its CTAs may
// start while the previous kernel on the stream is still finishing, run
// their prologue (shared tables, barriers, TMEM allocation), and wait in
// pdl_wait() for that kernel to complete before touching global memory.
// Without a previous kernel the wait returns at once.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct DeviceInfo {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    size_t smem_optin = 0;     // max dynamic shared memory per block (opt-in)
    uint32_t* err_word = nullptr;  // device address of this device's error word
};

// Add n to the process-wide count of enqueued kernels (nf4_launch_count).
void count_launches(int n);

// The current device's cached info (initialised on first use, see
// nf4_capi.cu).  Returns 0 (NF4_OK) or an nf4_status code.
int current_device_info(const DeviceInfo** out);

// dtype: the element type of w / out (0 bf16, 1 fp16, 2 fp32, as nf4_dtype).
cudaError_t launch_quantize(const DeviceInfo& dev, const void* w, int dtype, int64_t numel, uint8_t* packed,
                            float* absmax, cudaStream_t s);

cudaError_t launch_dequantize(const DeviceInfo& dev, const uint8_t* packed, const float* absmax,
                              int64_t numel, int dtype, void* out, cudaStream_t s);

// Fused NF4 GEMM, M >= 128 path (tcgen05 / TMEM).  dtype: the type of x, y
// and the converted weights, bf16 (0), fp16 (1) or fp32 (2, tf32 MMA).
cudaError_t launch_gemm(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t N, void* y,
                        cudaStream_t s);

// Workspace bytes the skinny (M < 128) path needs for this shape.
size_t skinny_workspace_bytes(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K);

// Fused NF4 GEMM of a gate/up pair ([2F, K] weight, gate rows first) with the
// GELU-gated product as epilogue, M >= 128: y [M, F] = gelu(X Wg^T) * (X Wu^T).
cudaError_t launch_gemm_geglu(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                              const uint8_t* packed, const float* absmax, int64_t F, void* y,
                              cudaStream_t s);

// Skinny path: swap-AB tcgen05 GEMM with split-K into an fp32 workspace and an
// ordered reduction.  N is the weight's row count; with geglu the weight is a
// gate/up pair (N = 2F) and the reduction writes gelu(gate) * up, [M, F].
cudaError_t launch_skinny(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                          const uint8_t* packed, const float* absmax, int64_t N, void* y,
                          void* workspace, size_t ws_bytes, cudaStream_t s, bool geglu = false);

}  // namespace nf4
