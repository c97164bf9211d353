// nf4_launch.h -- internal interface between the C ABI front end
// (nf4_capi.cu) and the kernel launchers.  Not installed, not part of the ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>

#include <cuda.h>
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

// Error word codes (the first one recorded wins).  nf4_last_error reports a
// 0x1xx word as a timeout and a 0x2xx word as an index out of bounds.
enum : uint32_t {
    kErrTimeoutFull = 0x101,      // waiting for a loaded stage
    kErrTimeoutEmpty = 0x102,     // waiting for a stage to be released
    kErrTimeoutConverted = 0x103, // waiting for converted weights
    kErrTimeoutAccum = 0x104,     // waiting for the accumulator
    kErrTimeoutDrain = 0x105,     // waiting for copies in flight at exit
    kErrBounds = 0x201,           // checked build: an index outside its buffer
};

struct DeviceInfo {
    int ordinal = -1;
    int sm_count = 0;
    int cc_major = 0;
    int cc_minor = 0;
    size_t smem_optin = 0;     // max dynamic shared memory per block (opt-in)
    uint32_t* err_word = nullptr;  // device address of this device's error word
};

// 2-D row-major tensor map over [rows, cols] elements of `elem` bytes, box
// {box_cols, box_rows}, the given shared-memory swizzle; reads outside the
// tensor fill zeros.  False if the driver entry point is missing or the
// encoding is refused.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t rows,
              uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle);

// Raise a kernel's dynamic shared memory limit, once per (kernel, device).
cudaError_t set_smem(const void* kernel, size_t bytes, int device);

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

// The CTA-pair NF4 GEMM (nf4_gemm_wide.cu): expanded weights in shared
// memory, two TMEM accumulators, pair tiles of 256 weight rows x up to 512
// activation rows (bf16 / fp16 / fp32, M > 256).  wide_applies: whether it beats
// the tile kernel on this shape (a shape-only estimate; N = rows of the
// weight); launch_gemm and launch_gemm_geglu use it then.  N: rows of the
// weight; geglu: the weight is a gate/up pair (N = 2F) and Y is [M, F].
bool wide_applies(int dtype, int64_t M, int64_t N);
cudaError_t launch_gemm_wide(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                             const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s,
                             bool geglu = false);

// Workspace bytes the skinny (M < 128) path needs for this shape.
size_t skinny_workspace_bytes(const DeviceInfo* dev, int64_t M, int64_t N, int64_t K);

// Fused NF4 GEMM of a gate/up pair ([2F, K] weight, gate rows first) with the
// GELU-gated product as epilogue, M >= 128: y [M, F] = gelu(X Wg^T) * (X Wu^T).
cudaError_t launch_gemm_geglu(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                              const uint8_t* packed, const float* absmax, int64_t F, void* y,
                              cudaStream_t s);

// Warp-MMA NF4 linear for M <= 16 at bf16 / fp16 (nf4_gemv.cu): whether it
// takes this shape and dtype, its workspace (a header of arrival counters that
// must be zero before the first call and is zero again after every call,
// followed by split-K partials) and its launcher.  rows: the weight's row
// count (2F for a gate/up pair, whose output is [M, F]).
bool gemv_applies(int dtype, int64_t M, int64_t rows, int64_t K);
size_t gemv_workspace_bytes(int64_t M, int64_t rows, int64_t K);
size_t gemv_header_bytes();
cudaError_t launch_gemv(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t rows, void* y, void* workspace,
                        size_t ws_bytes, cudaStream_t s, bool pair);

// Skinny path (M < 128): the warp-MMA kernel where it applies, else the
// swap-AB tcgen05 GEMM with split-K into an fp32 workspace and an ordered
// reduction.  N is the weight's row count; with geglu the weight is a
// gate/up pair (N = 2F) and the reduction writes gelu(gate) * up, [M, F].
cudaError_t launch_skinny(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                          const uint8_t* packed, const float* absmax, int64_t N, void* y,
                          void* workspace, size_t ws_bytes, cudaStream_t s, bool geglu = false);

}  // namespace nf4
