// nf4_quant.cu -- blockwise absmax NF4 quantizer and byte-LUT dequantizer.
//
// Quantizer: diffuseR pull request "Gemma3 NF4 on GPU" (#39), Summary -- the
// projection weights "pack to NF4".  Dequantizer: same paragraph -- the eager
// dequant gathers one lookup-table entry per packed byte straight into the
// output buffer.  Both kernels are HBM-bound streaming kernels.
#include "nf4_device.cuh"
#include "nf4_launch.h"

#include <algorithm>

namespace nf4 {

// ============================================================ quantize

// Code of one normalised value by binary search over the 15 thresholds, held
// in shared memory as a copy of c_thr (s_thr[15] = +inf pads the table).
__device__ __forceinline__ uint32_t code_of(float n, const float* s_thr) {
    uint32_t c = (n > c_thr[7]) ? 8u : 0u;
    c |= (n > s_thr[c + 3]) ? 4u : 0u;
    c |= (n > s_thr[c + 1]) ? 2u : 0u;
    c |= (n > s_thr[c]) ? 1u : 0u;
    return c;
}

// Quantize 8 consecutive bf16 (one 16-byte word) against a block absmax
// `am_bits` (bf16 bit pattern of max |w|) into 4 packed bytes.
__device__ __forceinline__ uint32_t quantize8(uint4 v, uint32_t am_bits, const float* s_thr) {
    const float am = __uint_as_float(am_bits << 16);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // element 2i sits in the low half of word i (lower address)
        float w0 = __uint_as_float(wd[i] << 16);
        float w1 = __uint_as_float(wd[i] & 0xffff0000u);
        uint32_t c0 = 7u, c1 = 7u;
        if (am_bits != 0u) {
            c0 = code_of(__fdiv_rn(w0, am), s_thr);
            c1 = code_of(__fdiv_rn(w1, am), s_thr);
        }
        out |= ((c0 << 4) | c1) << (8 * i);
    }
    return out;
}

// Fast code selection.  n = w / absmax is approximated by q = w * rcp(absmax)
// with a correctly rounded reciprocal: |q - n| <= 3 * 2^-24 * |n|.  A uniform
// grid of 65 cells of width 1/32 over [-1, 1] holds at most one threshold per
// cell, and every threshold sits at least 1e-3 from a cell edge (checked at
// compile time below), so the cell of q and the count of thresholds below it
// are those of n.  Only the cell's own threshold can separate q from n, and
// only when |q - t| <= 2^-20 |t|; such elements (a handful per billion) take
// the exact path: IEEE division and the threshold search.
constexpr int kCells = 65;
constexpr double kCellWidth = 1.0 / 32.0;

constexpr bool grid_is_safe() {
    int prev_cell = -1;
    for (int j = 0; j < 15; ++j) {
        double t = static_cast<double>(threshold(j));
        double x = (t + 1.0) / kCellWidth;
        int cell = static_cast<int>(x);
        double frac = x - cell;
        if (cell <= prev_cell) return false;                      // one threshold per cell
        if (frac * kCellWidth < 1e-3 || (1.0 - frac) * kCellWidth < 1e-3) return false;
        prev_cell = cell;
    }
    return true;
}
static_assert(grid_is_safe(), "quantizer grid: thresholds must be one per cell and away from cell edges");

struct QuantCell {
    float t;          // the threshold inside the cell, or +inf
    float guard;      // |t| * 2^-20: closer than this, decide exactly
    uint32_t base;    // number of thresholds below the cell
    uint32_t pad;
};

__device__ __forceinline__ void build_cells(QuantCell* cells, int tid, int nthreads) {
    for (int i = tid; i < kCells; i += nthreads) {
        const float lo = static_cast<float>(i) * 0.03125f - 1.0f;     // exact
        const float hi = lo + 0.03125f;
        QuantCell c{__int_as_float(0x7f800000), 0.0f, 0u, 0u};
        for (int j = 0; j < 15; ++j) {
            const float t = c_thr[j];
            if (t < lo) ++c.base;
            else if (t < hi) c.t = t, c.guard = fabsf(t) * 0x1p-20f;
        }
        cells[i] = c;
    }
}

__device__ __forceinline__ uint32_t fast_code(float q, const QuantCell* cells, bool& exact_needed) {
    int idx = __float2int_rz(fmaf(q, 32.0f, 32.0f));
    idx = min(max(idx, 0), kCells - 1);
    const QuantCell c = cells[idx];
    exact_needed |= !(fabsf(q - c.t) > c.guard);
    return c.base + (q > c.t ? 1u : 0u);
}

// quantize8 with the fast path: one reciprocal per block, the exact path only
// for elements the grid cannot decide.
__device__ __forceinline__ uint32_t quantize8_fast(uint4 v, uint32_t am_bits, const QuantCell* cells,
                                                   const float* s_thr) {
    if (am_bits == 0u) return 0x77777777u;
    const float am = __uint_as_float(am_bits << 16);
    const float rcp = __frcp_rn(am);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
    bool exact_needed = false;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t c0 = fast_code(__uint_as_float(wd[i] << 16) * rcp, cells, exact_needed);
        const uint32_t c1 = fast_code(__uint_as_float(wd[i] & 0xffff0000u) * rcp, cells, exact_needed);
        out |= ((c0 << 4) | c1) << (8 * i);
    }
    return exact_needed ? quantize8(v, am_bits, s_thr) : out;
}

__device__ __forceinline__ uint32_t absmax_bits8(uint4 v) {
    uint32_t m = max(max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu), max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu));
    m = max(m, max(max(v.z & 0x7fffu, (v.z >> 16) & 0x7fffu), max(v.w & 0x7fffu, (v.w >> 16) & 0x7fffu)));
    return m;
}

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 4;

// Vectorized quantizer for whole blocks.  Thread t of a warp owns the 16-byte
// word t of a 512-byte warp tile (4 blocks); 8 lanes share a block and reduce
// its absmax with shuffles.  Finite bf16 magnitudes order like their 15-bit
// patterns, so the absmax is an integer max over (bits & 0x7fff).
__global__ void __launch_bounds__(kQuantThreads)
quantize_vec_kernel(const uint4* __restrict__ w, int64_t nwords, uint32_t* __restrict__ packed,
                    float* __restrict__ absmax) {
    __shared__ float s_thr[16];
    __shared__ QuantCell s_cells[kCells];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    build_cells(s_cells, threadIdx.x, kQuantThreads);
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kQuantThreads) >> 5;
    const int64_t ntiles = (nwords + 31) >> 5;
    for (int64_t t0 = warp; t0 < ntiles; t0 += nwarps * kQuantUnroll) {
        uint4 v[kQuantUnroll];
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t word = ((t0 + u * nwarps) << 5) + lane;
            v[u] = (t0 + u * nwarps < ntiles && word < nwords) ? ldg_nc_v4(w + word) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t word = ((t0 + u * nwarps) << 5) + lane;
            uint32_t m = absmax_bits8(v[u]);
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
            if (t0 + u * nwarps < ntiles && word < nwords) {
                packed[word] = quantize8_fast(v[u], m, s_cells, s_thr);
                if ((lane & 7) == 0) absmax[word >> 3] = __uint_as_float(m << 16);
            }
        }
    }
}

// Element-wise quantizer: one thread per block, for blocks [b0, b1).  Used for
// a partial last block and for inputs the vectorized kernel cannot take
// (unaligned pointers).
__global__ void quantize_scalar_kernel(const uint16_t* __restrict__ w, int64_t numel, int64_t b0,
                                       int64_t b1, uint8_t* __restrict__ packed,
                                       float* __restrict__ absmax) {
    __shared__ float s_thr[16];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    __syncthreads();
    for (int64_t b = b0 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < b1;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t lo = b * kBlock;
        const int64_t hi = min(lo + kBlock, numel);
        uint32_t m = 0;
        for (int64_t i = lo; i < hi; ++i) m = max(m, static_cast<uint32_t>(w[i]) & 0x7fffu);
        const float am = __uint_as_float(m << 16);
        absmax[b] = am;
        for (int64_t i = lo; i < hi; i += 2) {
            uint32_t c0 = 7u, c1 = 7u;
            if (m != 0u) {
                c0 = code_of(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(w[i]) << 16), am), s_thr);
                c1 = code_of(__fdiv_rn(__uint_as_float(static_cast<uint32_t>(w[i + 1]) << 16), am), s_thr);
            }
            packed[i >> 1] = static_cast<uint8_t>((c0 << 4) | c1);
        }
    }
}

// ============================================================ dequantize

constexpr int kDequantThreads = 256;

// Vectorized byte-LUT dequantizer.  A warp tile is 512 packed bytes (1024
// outputs, 2 KB).  In step i (0..3) lane t reads packed word 32i + t (one
// coalesced 128-byte line per warp), looks its 4 bytes up in the 256-entry
// bf16x2 table, scales by the block absmax and writes one 16-byte word
// (one coalesced 512-byte line per warp).  A warp takes kDequantTiles
// consecutive tiles per iteration, issuing all their loads before the first
// store, so each warp keeps 1 KB of reads in flight.
constexpr int kDequantTiles = 2;

__global__ void __launch_bounds__(kDequantThreads)
dequant_vec_kernel(const uint32_t* __restrict__ packed, const float* __restrict__ absmax,
                   int64_t ntiles, uint4* __restrict__ out) {
    __shared__ uint32_t lut[256];
    for (int e = threadIdx.x; e < 256; e += kDequantThreads) lut[e] = lut_entry(static_cast<uint32_t>(e));
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kDequantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kDequantThreads) >> 5;
    constexpr int U = kDequantTiles;
    for (int64_t t0 = warp * U; t0 < ntiles; t0 += nwarps * U) {
        uint32_t p[4 * U];
        float a[4 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t tile = min(t0 + u, ntiles - 1);   // past the end: reload the last tile, store nothing
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                p[4 * u + i] = ldg_nc_u32(packed + tile * 128 + 32 * i + lane);
                a[4 * u + i] = ldg_nc_f32(absmax + tile * 16 + 4 * i + (lane >> 3));
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t tile = t0 + u;
            if (tile < ntiles) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint32_t q = p[4 * u + i];
                    const float am = a[4 * u + i];
                    uint4 o;
                    o.x = scale_entry(lut[q & 0xffu], am);
                    o.y = scale_entry(lut[(q >> 8) & 0xffu], am);
                    o.z = scale_entry(lut[(q >> 16) & 0xffu], am);
                    o.w = scale_entry(lut[q >> 24], am);
                    stg_v4(out + tile * 128 + 32 * i + lane, o);
                }
            }
        }
    }
}

// Element-pair dequantizer for packed bytes [j0, j1): the tail after the
// last whole tile, or everything when pointers are not aligned for the
// vectorized kernel.
__global__ void dequant_scalar_kernel(const uint8_t* __restrict__ packed,
                                      const float* __restrict__ absmax, int64_t j0, int64_t j1,
                                      uint16_t* __restrict__ out) {
    __shared__ uint32_t lut[256];
    for (int e = threadIdx.x; e < 256; e += blockDim.x) lut[e] = lut_entry(static_cast<uint32_t>(e));
    __syncthreads();
    for (int64_t j = j0 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; j < j1;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const uint32_t v = scale_entry(lut[packed[j]], absmax[(2 * j) / kBlock]);
        out[2 * j] = static_cast<uint16_t>(v & 0xffffu);
        out[2 * j + 1] = static_cast<uint16_t>(v >> 16);
    }
}

// ============================================================ launchers

// rounds x (SMs x resident CTAs per SM), capped at the number of work items
static int grid_for(const DeviceInfo& dev, const void* kernel, int threads, int64_t work_items, int rounds = 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, 0) != cudaSuccess || per_sm < 1)
        per_sm = 1;
    int64_t g = static_cast<int64_t>(dev.sm_count) * per_sm * rounds;
    if (work_items < g) g = work_items;
    return static_cast<int>(g < 1 ? 1 : g);
}

cudaError_t launch_quantize(const DeviceInfo& dev, const uint16_t* w, int64_t numel, uint8_t* packed,
                            float* absmax, cudaStream_t s) {
    const int64_t nblocks = (numel + kBlock - 1) / kBlock;
    const int64_t full = numel / kBlock;
    const bool aligned = (reinterpret_cast<uintptr_t>(w) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(packed) % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(absmax) % 4 == 0);
    int64_t scalar_from = 0;
    if (aligned && full > 0) {
        const int64_t nwords = full * 8;   // 8 bf16 per 16-byte word
        const int64_t ntiles = (nwords + 31) / 32;
        const int grid = grid_for(dev, reinterpret_cast<const void*>(quantize_vec_kernel),
                                  kQuantThreads, (ntiles + kQuantThreads / 32 - 1) / (kQuantThreads / 32));
        quantize_vec_kernel<<<grid, kQuantThreads, 0, s>>>(reinterpret_cast<const uint4*>(w), nwords,
                                                          reinterpret_cast<uint32_t*>(packed), absmax);
        count_launches(1);
        scalar_from = full;
    }
    if (scalar_from < nblocks) {
        const int64_t n = nblocks - scalar_from;
        const int threads = 128;
        const int grid = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 4 * static_cast<int64_t>(dev.sm_count)));
        quantize_scalar_kernel<<<grid, threads, 0, s>>>(w, numel, scalar_from, nblocks, packed, absmax);
        count_launches(1);
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const DeviceInfo& dev, const uint8_t* packed, const float* absmax,
                              int64_t numel, uint16_t* out, cudaStream_t s) {
    const int64_t nbytes = numel / 2;
    const bool aligned = (reinterpret_cast<uintptr_t>(packed) % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(absmax) % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    int64_t scalar_from = 0;
    if (aligned) {
        const int64_t ntiles = nbytes / 512;
        if (ntiles > 0) {
            // twice the resident CTAs: the second round starts on SMs as
            // the first one drains, which evens out the end of the grid
            const int64_t warp_items = (ntiles + kDequantTiles - 1) / kDequantTiles;
            const int grid = grid_for(dev, reinterpret_cast<const void*>(dequant_vec_kernel), kDequantThreads,
                                      (warp_items + kDequantThreads / 32 - 1) / (kDequantThreads / 32), 2);
            dequant_vec_kernel<<<grid, kDequantThreads, 0, s>>>(
                reinterpret_cast<const uint32_t*>(packed), absmax, ntiles, reinterpret_cast<uint4*>(out));
            count_launches(1);
        }
        scalar_from = ntiles * 512;
    }
    if (scalar_from < nbytes) {
        const int64_t n = nbytes - scalar_from;
        const int threads = 256;
        const int grid = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 8 * static_cast<int64_t>(dev.sm_count)));
        dequant_scalar_kernel<<<grid, threads, 0, s>>>(packed, absmax, scalar_from, nbytes, out);
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace nf4
