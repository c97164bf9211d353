// nf4_quant.cu -- blockwise absmax NF4 quantizer and byte-LUT dequantizer.
//
// Quantizer: diffuseR pull request "Gemma3 NF4 on GPU" (#39), Summary -- the
// projection weights are packed to NF4.  Dequantizer: same paragraph -- the
// eager dequant gathers one lookup-table entry per packed byte straight into
// the output buffer.  Both kernels are HBM-bound streaming kernels; each
// takes bf16, fp16 or fp32 weights / outputs.
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

// The fp32 value of a 16-bit magnitude pattern of type DT (the block max).
template <int DT>
__device__ __forceinline__ float am_of(uint32_t m) {
    return unpack2<DT>(m).x;
}

// The packed byte of two values by exact division (the reference path).
__device__ __forceinline__ uint32_t code_byte_exact(float w0, float w1, float am, const float* s_thr) {
    if (am == 0.0f) return 0x77u;
    return (code_of(__fdiv_rn(w0, am), s_thr) << 4) | code_of(__fdiv_rn(w1, am), s_thr);
}

// Quantize 8 consecutive 16-bit values of type DT (one 16-byte word) against
// a block absmax `am_bits` (the 16-bit pattern of max |w|) into 4 packed
// bytes by exact division.
template <int DT>
__device__ __forceinline__ uint32_t quantize8(uint4 v, uint32_t am_bits, const float* s_thr) {
    const float am = am_of<DT>(am_bits);
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    uint32_t out = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 w = unpack2<DT>(wd[i]);   // element 2i in the low half (lower address)
        out |= code_byte_exact(w.x, w.y, am, s_thr) << (8 * i);
    }
    return out;
}

// Fast code selection.  n = w / absmax is approximated by q = w * rcp(absmax)
// with a correctly rounded reciprocal: |q - n| <= 3 * 2^-24 * |n| <= 2^-22.
//
// A degree-5 polynomial h, fitted to h(T_j) ~ j at the 15 thresholds and
// monotone on [-1, 1], gives est = round(h(q)) with est in {code - 1, code}
// for every fp32 q in [-1 - 4 ulp, 1 + 4 ulp] (the true code of q is the
// number of thresholds below q).  That was checked for all 2.1e9 such q; h
// stays at least 0.032 away from the rounding boundaries that would break
// it, far above fp32 evaluation error.  So one comparison with T[est] (T[15]
// = +inf) decides the code of q: code = est + (q > T[est]).  The codes of q
// and n can only differ if a threshold lies between them, and the only
// threshold near q is T[est]; such words (|q - T[est]| <= 2^-21, a few per
// hundred thousand) are redone on the exact path.  The rounding to an
// integer rides on the last FMA: adding 1.5 * 2^23 leaves round(h) in the
// low mantissa bits, so the constant term (7) is kept an integer.
constexpr float kH5 = 1.6238466501235962f;
constexpr float kH4 = 1.0259608030319214f;
constexpr float kH3 = -5.9369730949401855f;
constexpr float kH2 = -0.9115704298019409f;
constexpr float kH1 = 11.66257095336914f;
constexpr float kH0Magic = 12582919.0f;          // 7 + 1.5 * 2^23, exact in fp32
constexpr int kMagicBits = 0x4B400000;           // bits of 1.5 * 2^23
constexpr float kGuard = 0x1p-21f;

// Two fp32 lanes in one 64-bit register pair, for the packed f32x2 ops
// (each lane rounds exactly like the scalar op).
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack_f32x2(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Code of one quotient q given h(q) + 1.5 * 2^23 in `hm`.  For |q| <= 1 + 8
// ulp the estimate round(h(q)) is bits(hm) - bits(1.5 * 2^23), 0 .. 15; the
// magic's low four bits are zero, so that equals bits(hm) & 15 -- which keeps
// the table index in range whatever q is (a non-finite input gives an
// unspecified code, never an out-of-range read).
__device__ __forceinline__ uint32_t code_from_estimate(float q, float hm, const float* s_thr, bool& exact_needed) {
    static_assert((kMagicBits & 15) == 0, "the estimate is the low bits of the rounded sum");
    const uint32_t est = __float_as_uint(hm) & 15u;
    const float t = s_thr[est];
    exact_needed |= !(fabsf(q - t) > kGuard);
    return est + (q > t ? 1u : 0u);
}

// Below the smallest normal fp32 the reciprocal of an absmax can overflow:
// words of such blocks (bf16 or fp32 subnormals only) take the exact path.
constexpr float kMinNormal = 0x1p-126f;

// The packed byte of two values (w0 in the high nibble): the quotients and
// the polynomial run as f32x2 pairs.
__device__ __forceinline__ uint32_t code_pair(float w0, float w1, uint64_t rcp2, const float* s_thr, bool& exact_needed) {
    const uint64_t q2 = mul_f32x2(pack_f32x2(w0, w1), rcp2);
    uint64_t h2 = fma_f32x2(pack_f32x2(kH5, kH5), q2, pack_f32x2(kH4, kH4));
    h2 = fma_f32x2(h2, q2, pack_f32x2(kH3, kH3));
    h2 = fma_f32x2(h2, q2, pack_f32x2(kH2, kH2));
    h2 = fma_f32x2(h2, q2, pack_f32x2(kH1, kH1));
    h2 = fma_f32x2(h2, q2, pack_f32x2(kH0Magic, kH0Magic));
    float q0, q1, h0, h1;
    unpack_f32x2(q2, q0, q1);
    unpack_f32x2(h2, h0, h1);
    const uint32_t c0 = code_from_estimate(q0, h0, s_thr, exact_needed);
    const uint32_t c1 = code_from_estimate(q1, h1, s_thr, exact_needed);
    return (c0 << 4) | c1;   // element 2i in the high nibble
}

// The packed byte of one word of two 16-bit values of type DT.
template <int DT>
__device__ __forceinline__ uint32_t code_pair16(uint32_t word, uint64_t rcp2, const float* s_thr, bool& exact_needed) {
    const float2 w = unpack2<DT>(word);
    return code_pair(w.x, w.y, rcp2, s_thr, exact_needed);
}

// quantize8 with the fast path: one reciprocal per block, the exact path only
// for words the estimate cannot decide.
template <int DT>
__device__ __forceinline__ uint32_t quantize8_fast(uint4 v, uint32_t am_bits, const float* s_thr) {
    if (am_bits == 0u) return 0x77777777u;
    const float am = am_of<DT>(am_bits);
    const float rcp = __frcp_rn(am);
    const uint64_t rcp2 = pack_f32x2(rcp, rcp);
    // a subnormal absmax: the reciprocal may be infinite, the estimates then
    // unspecified (but in range) -- take the exact path for the whole word
    bool exact_needed = am < kMinNormal;
    const uint32_t out = code_pair16<DT>(v.x, rcp2, s_thr, exact_needed) |
                         (code_pair16<DT>(v.y, rcp2, s_thr, exact_needed) << 8) |
                         (code_pair16<DT>(v.z, rcp2, s_thr, exact_needed) << 16) |
                         (code_pair16<DT>(v.w, rcp2, s_thr, exact_needed) << 24);
    return exact_needed ? quantize8<DT>(v, am_bits, s_thr) : out;
}

// Four fp32 values (one 16-byte word) against a block absmax -> 2 packed
// bytes (the first in the low byte), fast path with the exact fallback.
__device__ __forceinline__ uint32_t quantize4_f32_fast(uint4 v, float am, const float* s_thr) {
    if (am == 0.0f) return 0x7777u;
    if (am < kMinNormal)   // as in quantize8_fast; an early exit keeps this kernel within 32 registers
        return code_byte_exact(__uint_as_float(v.x), __uint_as_float(v.y), am, s_thr) |
               (code_byte_exact(__uint_as_float(v.z), __uint_as_float(v.w), am, s_thr) << 8);
    const float rcp = __frcp_rn(am);
    const uint64_t rcp2 = pack_f32x2(rcp, rcp);
    bool exact_needed = false;
    const float w0 = __uint_as_float(v.x), w1 = __uint_as_float(v.y);
    const float w2 = __uint_as_float(v.z), w3 = __uint_as_float(v.w);
    const uint32_t out = code_pair(w0, w1, rcp2, s_thr, exact_needed) | (code_pair(w2, w3, rcp2, s_thr, exact_needed) << 8);
    if (!exact_needed) return out;
    return code_byte_exact(w0, w1, am, s_thr) | (code_byte_exact(w2, w3, am, s_thr) << 8);
}

// Per-halfword unsigned max of two words of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest 15-bit magnitude pattern among the 8 16-bit values of a 16-byte
// word, reduced pairwise on both halves at once.  Finite bf16 and fp16
// magnitudes both order like their 15-bit patterns.
__device__ __forceinline__ uint32_t absmax_bits8(uint4 v) {
    const uint32_t m2 = max_u16x2(max_u16x2(v.x & 0x7fff7fffu, v.y & 0x7fff7fffu),
                                  max_u16x2(v.z & 0x7fff7fffu, v.w & 0x7fff7fffu));
    return max(m2 & 0xffffu, m2 >> 16);
}

constexpr int kQuantThreads = 256;
constexpr int kQuantUnroll = 1;   // 16-byte words in flight per thread

// Vectorized quantizer for whole blocks of a 16-bit type DT.  Thread t of a
// warp owns the 16-byte word t of a 512-byte warp tile (4 blocks); 8 lanes
// share a block and reduce its absmax with shuffles.  Finite bf16 and fp16
// magnitudes order like their 15-bit patterns, so the absmax is an integer
// max over (bits & 0x7fff).  nwords covers whole blocks of the numel values.
template <int DT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_vec_kernel(const uint4* __restrict__ w, int64_t nwords, uint32_t* __restrict__ packed,
                    float* __restrict__ absmax, int64_t numel, uint32_t* err) {
    __shared__ float s_thr[16];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kQuantThreads) >> 5;
    const int64_t ntiles = (nwords + 31) >> 5;
    // kQuantUnroll tiles per warp and iteration; the next iteration's words are
    // loaded before this one's are converted, so each warp keeps a DRAM round
    // trip in flight while it computes
    auto load = [&](int64_t t0, uint4 (&v)[kQuantUnroll]) {
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t word = ((t0 + u * nwarps) << 5) + lane;
            v[u] = (t0 + u * nwarps < ntiles && word < nwords && in_bounds(err, word, numel / 8)) ? ldg_nc_v4(w + word)
                                                                                           : make_uint4(0, 0, 0, 0);
        }
    };
    uint4 v[kQuantUnroll], nv[kQuantUnroll];
    if (warp < ntiles) load(warp, nv);
    for (int64_t t0 = warp; t0 < ntiles; t0 += nwarps * kQuantUnroll) {
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) v[u] = nv[u];
        if (t0 + nwarps * kQuantUnroll < ntiles) load(t0 + nwarps * kQuantUnroll, nv);
#pragma unroll
        for (int u = 0; u < kQuantUnroll; ++u) {
            const int64_t word = ((t0 + u * nwarps) << 5) + lane;
            uint32_t m = absmax_bits8(v[u]);
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
            m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
            if (t0 + u * nwarps < ntiles && word < nwords) {
                if (in_bounds(err, word, numel / 8)) packed[word] = quantize8_fast<DT>(v[u], m, s_thr);
                if ((lane & 7) == 0 && in_bounds(err, word >> 3, (numel + kBlock - 1) / kBlock))
                    absmax[word >> 3] = am_of<DT>(m);
            }
        }
    }
}

// Vectorized quantizer for whole blocks of fp32.  Thread t of a warp owns
// the 16-byte word t (4 values) of a 512-byte warp tile (2 blocks); 16 lanes
// share a block.  Finite fp32 magnitudes order like their 31-bit patterns.
__global__ void __launch_bounds__(kQuantThreads)
quantize_vec_f32_kernel(const uint4* __restrict__ w, int64_t nwords, uint16_t* __restrict__ packed,
                        float* __restrict__ absmax, int64_t numel, uint32_t* err) {
    __shared__ float s_thr[16];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kQuantThreads) >> 5;
    const int64_t ntiles = (nwords + 31) >> 5;
    auto load = [&](int64_t t) {
        const int64_t word = (t << 5) + lane;
        return (t < ntiles && word < nwords && in_bounds(err, word, numel / 4)) ? ldg_nc_v4(w + word)
                                                                                : make_uint4(0, 0, 0, 0);
    };
    uint4 nv = make_uint4(0, 0, 0, 0);
    if (warp < ntiles) nv = load(warp);
    for (int64_t t = warp; t < ntiles; t += nwarps) {
        const uint4 v = nv;
        if (t + nwarps < ntiles) nv = load(t + nwarps);   // next tile's word in flight meanwhile
        const int64_t word = (t << 5) + lane;
        uint32_t m = max(max(v.x & 0x7fffffffu, v.y & 0x7fffffffu), max(v.z & 0x7fffffffu, v.w & 0x7fffffffu));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 4));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 8));
        if (word < nwords) {
            const float am = __uint_as_float(m);
            if (in_bounds(err, word, numel / 4)) packed[word] = static_cast<uint16_t>(quantize4_f32_fast(v, am, s_thr));
            if ((lane & 15) == 0 && in_bounds(err, word >> 4, (numel + kBlock - 1) / kBlock)) absmax[word >> 4] = am;
        }
    }
}

// Element i of a tensor of type DT, widened to fp32 (exact).
template <int DT>
__device__ __forceinline__ float load_elem(const void* w, int64_t i) {
    if constexpr (DT == kF32)
        return static_cast<const float*>(w)[i];
    else
        return unpack2<DT>(static_cast<const uint16_t*>(w)[i]).x;
}

// Element-wise quantizer: one thread per block, for blocks [b0, b1).  Used for
// a partial last block and for inputs the vectorized kernel cannot take
// (unaligned pointers).
template <int DT>
__global__ void quantize_scalar_kernel(const void* __restrict__ w, int64_t numel, int64_t b0,
                                       int64_t b1, uint8_t* __restrict__ packed,
                                       float* __restrict__ absmax, uint32_t* err) {
    __shared__ float s_thr[16];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    for (int64_t b = b0 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; b < b1;
         b += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t lo = b * kBlock;
        const int64_t hi = min(lo + kBlock, numel);
        auto elem = [&](int64_t i) { return in_bounds(err, i, numel) ? load_elem<DT>(w, i) : 0.0f; };
        float am = 0.0f;
        for (int64_t i = lo; i < hi; ++i) am = fmaxf(am, fabsf(elem(i)));
        if (in_bounds(err, b, (numel + kBlock - 1) / kBlock)) absmax[b] = am;
        for (int64_t i = lo; i < hi; i += 2)
            if (in_bounds(err, i >> 1, numel / 2))
                packed[i >> 1] = static_cast<uint8_t>(code_byte_exact(elem(i), elem(i + 1), am, s_thr));
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

template <int DT>
__global__ void __launch_bounds__(kDequantThreads)
dequant_vec_kernel(const uint32_t* __restrict__ packed, const float* __restrict__ absmax,
                   int64_t ntiles, uint4* __restrict__ out, int64_t numel, uint32_t* err) {
    __shared__ uint32_t lut[256];
    for (int e = threadIdx.x; e < 256; e += kDequantThreads) lut[e] = lut_entry<DT>(static_cast<uint32_t>(e));
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
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
                const int64_t pi = tile * 128 + 32 * i + lane, ai = tile * 16 + 4 * i + (lane >> 3);
                p[4 * u + i] = in_bounds(err, pi, numel / 8) ? ldg_nc_u32(packed + pi) : 0u;
                a[4 * u + i] = in_bounds(err, ai, (numel + kBlock - 1) / kBlock) ? ldg_nc_f32(absmax + ai) : 0.0f;
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
                    o.x = scale_entry<DT>(lut[q & 0xffu], am);
                    o.y = scale_entry<DT>(lut[(q >> 8) & 0xffu], am);
                    o.z = scale_entry<DT>(lut[(q >> 16) & 0xffu], am);
                    o.w = scale_entry<DT>(lut[q >> 24], am);
                    if (in_bounds(err, tile * 128 + 32 * i + lane, numel / 8)) stg_v4(out + tile * 128 + 32 * i + lane, o);
                }
            }
        }
    }
}

// fp32 output: a warp tile is 128 packed bytes (256 outputs, 1 KB, 4
// blocks).  In step i (0..1) lane t reads packed halfword 32i + t, looks up
// the fp32 codebook values of its four codes and writes them, scaled by the
// block absmax (one fp32 multiply each), as one 16-byte word: each warp
// store is one coalesced 512-byte line.
constexpr int kDequantTilesF32 = 4;

__global__ void __launch_bounds__(kDequantThreads)
dequant_vec_f32_kernel(const uint16_t* __restrict__ packed, const float* __restrict__ absmax,
                       int64_t ntiles, uint4* __restrict__ out, int64_t numel, uint32_t* err) {
    __shared__ float code[16];
    if (threadIdx.x < 16) code[threadIdx.x] = c_code[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kDequantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kDequantThreads) >> 5;
    constexpr int U = kDequantTilesF32;
    for (int64_t t0 = warp * U; t0 < ntiles; t0 += nwarps * U) {
        uint32_t p[2 * U];
        float a[2 * U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t tile = min(t0 + u, ntiles - 1);   // past the end: reload the last tile, store nothing
#pragma unroll
            for (int i = 0; i < 2; ++i) {
                const int64_t pi = tile * 64 + 32 * i + lane, ai = tile * 4 + 2 * i + (lane >> 4);
                p[2 * u + i] = in_bounds(err, pi, numel / 4) ? packed[pi] : 0u;
                a[2 * u + i] = in_bounds(err, ai, (numel + kBlock - 1) / kBlock) ? ldg_nc_f32(absmax + ai) : 0.0f;
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t tile = t0 + u;
            if (tile < ntiles) {
#pragma unroll
                for (int i = 0; i < 2; ++i) {
                    const uint32_t q = p[2 * u + i];   // byte 0 (lower address) in the low 8 bits
                    const float am = a[2 * u + i];
                    uint4 o;
                    o.x = __float_as_uint(code[(q >> 4) & 15u] * am);
                    o.y = __float_as_uint(code[q & 15u] * am);
                    o.z = __float_as_uint(code[(q >> 12) & 15u] * am);
                    o.w = __float_as_uint(code[(q >> 8) & 15u] * am);
                    if (in_bounds(err, tile * 64 + 32 * i + lane, numel / 4)) stg_v4(out + tile * 64 + 32 * i + lane, o);
                }
            }
        }
    }
}

// Element-pair dequantizer for packed bytes [j0, j1): the tail after the
// last whole tile, or everything when pointers are not aligned for the
// vectorized kernel.
template <int DT>
__global__ void dequant_scalar_kernel(const uint8_t* __restrict__ packed,
                                      const float* __restrict__ absmax, int64_t j0, int64_t j1,
                                      void* __restrict__ out, int64_t numel, uint32_t* err) {
    __shared__ uint32_t lut[256];
    if constexpr (DT != kF32) {
        for (int e = threadIdx.x; e < 256; e += blockDim.x) lut[e] = lut_entry<DT>(static_cast<uint32_t>(e));
    }
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    for (int64_t j = j0 + blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; j < j1;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        if (!in_bounds(err, j, numel / 2) || !in_bounds(err, 2 * j + 1, numel)) continue;
        const uint32_t b = packed[j];
        const float am = in_bounds(err, (2 * j) / kBlock, (numel + kBlock - 1) / kBlock) ? absmax[(2 * j) / kBlock] : 0.0f;
        if constexpr (DT == kF32) {
            float* o = static_cast<float*>(out);
            o[2 * j] = c_code[b >> 4] * am;
            o[2 * j + 1] = c_code[b & 15u] * am;
        } else {
            const uint32_t v = scale_entry<DT>(lut[b], am);
            uint16_t* o = static_cast<uint16_t*>(out);
            o[2 * j] = static_cast<uint16_t>(v & 0xffffu);
            o[2 * j + 1] = static_cast<uint16_t>(v >> 16);
        }
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

namespace {

template <int DT>
cudaError_t launch_quantize_t(const DeviceInfo& dev, const void* w, int64_t numel, uint8_t* packed, float* absmax,
                              cudaStream_t s) {
    constexpr int kElem = DT == kF32 ? 4 : 2;     // bytes per element
    constexpr int kPerWord = 16 / kElem;          // elements per 16-byte word
    cudaError_t e = cudaSuccess;
    const int64_t nblocks = (numel + kBlock - 1) / kBlock;
    const int64_t full = numel / kBlock;
    const bool aligned = (reinterpret_cast<uintptr_t>(w) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(packed) % (kPerWord / 2) == 0) &&
                         (reinterpret_cast<uintptr_t>(absmax) % 4 == 0);
    int64_t scalar_from = 0;
    if (aligned && full > 0) {
        const int64_t nwords = full * (kBlock / kPerWord);
        const int64_t ntiles = (nwords + 31) / 32;
        const int64_t warps_per_cta = kQuantThreads / 32;
        if constexpr (DT == kF32) {
            const int grid = grid_for(dev, reinterpret_cast<const void*>(quantize_vec_f32_kernel), kQuantThreads,
                                      (ntiles + warps_per_cta - 1) / warps_per_cta);
            e = launch_pdl(quantize_vec_f32_kernel, grid, kQuantThreads, 0, s, static_cast<const uint4*>(w), nwords,
                           reinterpret_cast<uint16_t*>(packed), absmax, numel, dev.err_word);
        } else {
            const int grid = grid_for(dev, reinterpret_cast<const void*>(quantize_vec_kernel<DT>), kQuantThreads,
                                      (ntiles + warps_per_cta - 1) / warps_per_cta);
            e = launch_pdl(quantize_vec_kernel<DT>, grid, kQuantThreads, 0, s, static_cast<const uint4*>(w), nwords,
                           reinterpret_cast<uint32_t*>(packed), absmax, numel, dev.err_word);
        }
        if (e != cudaSuccess) return e;
        count_launches(1);
        scalar_from = full;
    }
    if (scalar_from < nblocks) {
        const int64_t n = nblocks - scalar_from;
        const int threads = 128;
        const int grid = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 4 * static_cast<int64_t>(dev.sm_count)));
        e = launch_pdl(quantize_scalar_kernel<DT>, grid, threads, 0, s, w, numel, scalar_from, nblocks, packed, absmax,
                       dev.err_word);
        if (e != cudaSuccess) return e;
        count_launches(1);
    }
    return cudaGetLastError();
}

template <int DT>
cudaError_t launch_dequantize_t(const DeviceInfo& dev, const uint8_t* packed, const float* absmax, int64_t numel,
                                void* out, cudaStream_t s) {
    cudaError_t e = cudaSuccess;
    const int64_t nbytes = numel / 2;
    constexpr int64_t kTileBytes = DT == kF32 ? 128 : 512;   // packed bytes per warp tile
    const bool aligned = (reinterpret_cast<uintptr_t>(packed) % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(absmax) % 4 == 0) &&
                         (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    int64_t scalar_from = 0;
    if (aligned) {
        const int64_t ntiles = nbytes / kTileBytes;
        if (ntiles > 0) {
            // twice the resident CTAs: the second round starts on SMs as
            // the first one drains, which evens out the end of the grid
            constexpr int U = DT == kF32 ? kDequantTilesF32 : kDequantTiles;
            const int64_t warp_items = (ntiles + U - 1) / U;
            const int64_t items = (warp_items + kDequantThreads / 32 - 1) / (kDequantThreads / 32);
            if constexpr (DT == kF32) {
                const int grid = grid_for(dev, reinterpret_cast<const void*>(dequant_vec_f32_kernel), kDequantThreads,
                                          items, 2);
                e = launch_pdl(dequant_vec_f32_kernel, grid, kDequantThreads, 0, s,
                               reinterpret_cast<const uint16_t*>(packed), absmax, ntiles, static_cast<uint4*>(out), numel,
                               dev.err_word);
            } else {
                const int grid = grid_for(dev, reinterpret_cast<const void*>(dequant_vec_kernel<DT>), kDequantThreads,
                                          items, 2);
                e = launch_pdl(dequant_vec_kernel<DT>, grid, kDequantThreads, 0, s,
                               reinterpret_cast<const uint32_t*>(packed), absmax, ntiles, static_cast<uint4*>(out), numel,
                               dev.err_word);
            }
            if (e != cudaSuccess) return e;
            count_launches(1);
        }
        scalar_from = ntiles * kTileBytes;
    }
    if (scalar_from < nbytes) {
        const int64_t n = nbytes - scalar_from;
        const int threads = 256;
        const int grid = static_cast<int>(std::min<int64_t>((n + threads - 1) / threads, 8 * static_cast<int64_t>(dev.sm_count)));
        e = launch_pdl(dequant_scalar_kernel<DT>, grid, threads, 0, s, packed, absmax, scalar_from, nbytes, out, numel,
                       dev.err_word);
        if (e != cudaSuccess) return e;
        count_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quantize(const DeviceInfo& dev, const void* w, int dtype, int64_t numel, uint8_t* packed,
                            float* absmax, cudaStream_t s) {
    switch (dtype) {
        case kBF16: return launch_quantize_t<kBF16>(dev, w, numel, packed, absmax, s);
        case kF16: return launch_quantize_t<kF16>(dev, w, numel, packed, absmax, s);
        case kF32: return launch_quantize_t<kF32>(dev, w, numel, packed, absmax, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_dequantize(const DeviceInfo& dev, const uint8_t* packed, const float* absmax, int64_t numel,
                              int dtype, void* out, cudaStream_t s) {
    switch (dtype) {
        case kBF16: return launch_dequantize_t<kBF16>(dev, packed, absmax, numel, out, s);
        case kF16: return launch_dequantize_t<kF16>(dev, packed, absmax, numel, out, s);
        case kF32: return launch_dequantize_t<kF32>(dev, packed, absmax, numel, out, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace nf4
