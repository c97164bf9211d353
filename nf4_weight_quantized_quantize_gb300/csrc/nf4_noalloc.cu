// nf4_noalloc.cu -- nf4_linear_noalloc: the skinny (M < 128) NF4 linear with
// its split-K scratch in a fixed, library-owned device array instead of a
// caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory themselves, e.g. a
// plugin whose host application owns every byte of the device memory pool and
// forbids extensions from allocating, or code on a path where cudaMalloc's
// implicit device-wide synchronization is not acceptable.  They still pass X,
// W and Y; only the scratch moves into this file.
//
// The scratch is a file-scope __device__ array of NF4_NOALLOC_SCRATCH_BYTES
// (16 MiB).  Every GPU that loads the library holds it until the process
// exits.  Host code cannot use the array's name as a device address (on the
// host it names a stand-in object), so the first call on each device, with
// that device current, resolves the real address once with
// cudaGetSymbolAddress and caches it; make that first call before any stream
// capture.  All calls on a device share the one array and it keeps the last
// call's contents.  Its first bytes are the skinny kernel's arrival counters,
// which must start at zero: each call clears them (a cudaMemsetAsync on the
// caller's stream, which allocates nothing) before its kernel, so even a call
// that follows one that timed out starts clean.  Every other element a call
// reads was written earlier in the same call.  Calls that overlap on the GPU
// (concurrent streams, or host threads) race on the array and must be
// serialised by the caller.  No cudaMalloc, cudaFree or allocating library
// routine is called here.
#include <mutex>

#include "../../include/nf4.h"
#include "nf4_launch.h"

namespace {

constexpr size_t kNoallocScratchBytes = NF4_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array, resolved once per device.
nf4_status scratch_address(int ordinal, void** out) {
    if (ordinal < 0 || ordinal >= kMaxDevices) return NF4_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[ordinal] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return NF4_ERR_CUDA;
        }
        g_scratch_ptr[ordinal] = p;
    }
    *out = g_scratch_ptr[ordinal];
    return NF4_OK;
}

inline bool aligned(const void* p, size_t a) { return reinterpret_cast<uintptr_t>(p) % a == 0; }

}  // namespace

extern "C" {

nf4_status nf4_linear_noalloc(const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                              const float* absmax, int64_t N, int32_t block, uint16_t* y, void* stream) {
    if (block != NF4_BLOCK) return NF4_ERR_BLOCKSIZE;
    if (M < 0 || N < 0 || K <= 0 || K % NF4_BLOCK != 0) return NF4_ERR_SHAPE;
    if (M >= 128) return NF4_ERR_SHAPE;   // the tile path needs no scratch: use nf4_linear
    if (N >= (int64_t(1) << 31) || K >= (int64_t(1) << 31)) return NF4_ERR_SHAPE;
    if (M == 0 || N == 0) return NF4_OK;
    if (!x || !packed || !absmax || !y) return NF4_ERR_NULL;
    if (!aligned(x, 16) || !aligned(packed, 16) || !aligned(y, 16) || !aligned(absmax, 4))
        return NF4_ERR_ALIGN;
    const size_t need = nf4::skinny_workspace_bytes(nullptr, M, N, K);
    if (need > kNoallocScratchBytes) return NF4_ERR_WORKSPACE;   // beyond the fixed 16 MiB scratch
    const nf4::DeviceInfo* dev = nullptr;
    if (int st = nf4::current_device_info(&dev); st != NF4_OK) return static_cast<nf4_status>(st);
    void* scratch = nullptr;
    if (nf4_status st = scratch_address(dev->ordinal, &scratch); st != NF4_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(scratch, 0, nf4::gemv_header_bytes(), s) != cudaSuccess) {
        cudaGetLastError();
        return NF4_ERR_CUDA;
    }
    cudaError_t e = nf4::launch_skinny(*dev, NF4_DTYPE_BF16, x, M, K, packed, absmax, N, y, scratch,
                                       kNoallocScratchBytes, s);
    return e == cudaSuccess ? NF4_OK : NF4_ERR_CUDA;
}

}  // extern "C"
