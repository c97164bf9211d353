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
// Cell table: q falls in cell c = round(16 q + 16), 0 .. 32 for |q| <= 1 +
// a few ulps -- the fp32 sum 16 q + (16 + 1.5 * 2^23) rounds once, to the
// integer c in the low mantissa bits (16 q is exact).  Cells are 1/16 wide
// and neighbouring thresholds at least 0.08 apart, so the threshold T_k
// nearest a cell's centre is the only one within 0.014 of any q in the cell,
// and T_(k-1) < q < T_(k+1) there: the code of q is k + (q > T_k).  Entry c
// is T_k with its low four fraction bits replaced by k + 1 (T_k moves by less
// than 16 ulp, at most 2^-20).  So code = (bits(e) & 15) - 1 + (q > e), the
// comparison made against the stored value.  It decides the code of q
// correctly, and the code of n too, whenever |q - e| > 2^-19: then q is more
// than 2^-20 from T_k and from every other threshold, farther than n is from
// q.  Words with a quotient within 2^-19 of its entry (about one in 10^4)
// are redone on the exact path.  The index is masked to the 64-entry table,
// so even a non-finite weight (outside the contract) reads inside it.
constexpr float kCellMagic = 12582928.0f;   // 16 + 1.5 * 2^23, exact in fp32
constexpr float kGuard = 0x1p-19f;
static __constant__ uint32_t c_cell[64] = {
    0xbf591cd1u, 0xbf591cd1u, 0xbf591cd1u, 0xbf591cd1u, 0xbf591cd1u, 0xbf1c5272u, 0xbf1c5272u, 0xbf1c5272u,
    0xbeeb8483u, 0xbeeb8483u, 0xbeadea74u, 0xbeadea74u, 0xbe703ce5u, 0xbe703ce5u, 0xbe0d38b6u, 0xbd3a7877u,
    0x3d22faf8u, 0x3d22faf8u, 0x3df64869u, 0x3e5067eau, 0x3e9582dbu, 0x3e9582dbu, 0x3ec753fcu, 0x3ec753fcu,
    0x3f006d0du, 0x3f006d0du, 0x3f248daeu, 0x3f248daeu, 0x3f248daeu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu,
    0x3f5c89dfu,   // cells 33 .. 63 are never hit by a finite quotient; they repeat cell 32
    0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu,
    0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu,
    0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu,
    0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu, 0x3f5c89dfu,
};

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

// Code of one quotient q from its cell value cm = 16 q + 16 + 1.5 * 2^23 (the
// cell index in the low bits); dmin keeps the smallest |q - entry| seen.
__device__ __forceinline__ uint32_t code_from_cell(float q, float cm, const uint32_t* s_cell, float& dmin) {
    const uint32_t e = s_cell[__float_as_uint(cm) & 63u];
    const float d = q - __uint_as_float(e);
    dmin = fminf(dmin, fabsf(d));
    return (e & 15u) - (d > 0.0f ? 0u : 1u);
}

// Below the smallest normal fp32 the reciprocal of an absmax can overflow:
// words of such blocks (bf16 or fp32 subnormals only) take the exact path.
constexpr float kMinNormal = 0x1p-126f;

// The packed byte of two values (w0 in the high nibble): the quotients and
// their cells run as f32x2 pairs.
__device__ __forceinline__ uint32_t code_pair(float w0, float w1, uint64_t rcp2, const uint32_t* s_cell, float& dmin) {
    const uint64_t q2 = mul_f32x2(pack_f32x2(w0, w1), rcp2);
    const uint64_t c2 = fma_f32x2(q2, pack_f32x2(16.0f, 16.0f), pack_f32x2(kCellMagic, kCellMagic));
    float q0, q1, c0, c1;
    unpack_f32x2(q2, q0, q1);
    unpack_f32x2(c2, c0, c1);
    const uint32_t k0 = code_from_cell(q0, c0, s_cell, dmin);
    const uint32_t k1 = code_from_cell(q1, c1, s_cell, dmin);
    return (k0 << 4) | k1;   // element 2i in the high nibble
}

// The packed byte of one word of two 16-bit values of type DT.
template <int DT>
__device__ __forceinline__ uint32_t code_pair16(uint32_t word, uint64_t rcp2, const uint32_t* s_cell, float& dmin) {
    const float2 w = unpack2<DT>(word);
    return code_pair(w.x, w.y, rcp2, s_cell, dmin);
}

// The 4 packed bytes of one word of 8 16-bit values of type DT (the first
// value in the high nibble of the lowest byte), by the cell table.
template <int DT>
__device__ __forceinline__ uint32_t codes8(uint4 v, uint64_t rcp2, const uint32_t* s_cell, float& dmin) {
    return code_pair16<DT>(v.x, rcp2, s_cell, dmin) | (code_pair16<DT>(v.y, rcp2, s_cell, dmin) << 8) |
           (code_pair16<DT>(v.z, rcp2, s_cell, dmin) << 16) | (code_pair16<DT>(v.w, rcp2, s_cell, dmin) << 24);
}

// Two consecutive words of one block (16 values) against its absmax pattern
// `am_bits`: one reciprocal, the cell table, and the exact path for both
// words if any quotient lies within the guard of its entry.
template <int DT>
__device__ __forceinline__ uint2 quantize16_fast(uint4 a, uint4 b, uint32_t am_bits, const float* s_thr,
                                                 const uint32_t* s_cell) {
    if (am_bits == 0u) return make_uint2(0x77777777u, 0x77777777u);
    const float am = am_of<DT>(am_bits);
    const float rcp = __frcp_rn(am);
    const uint64_t rcp2 = pack_f32x2(rcp, rcp);
    // a subnormal absmax: the reciprocal may be infinite, the codes then
    // unspecified (but in range) -- take the exact path
    float dmin = am < kMinNormal ? 0.0f : __int_as_float(0x7f800000);
    const uint2 out = make_uint2(codes8<DT>(a, rcp2, s_cell, dmin), codes8<DT>(b, rcp2, s_cell, dmin));
    if (dmin > kGuard) return out;
    return make_uint2(quantize8<DT>(a, am_bits, s_thr), quantize8<DT>(b, am_bits, s_thr));
}

// The 2 packed bytes of one word of 4 fp32 values (the first in the low
// byte), by the cell table.
__device__ __forceinline__ uint32_t codes4_f32(uint4 v, uint64_t rcp2, const uint32_t* s_cell, float& dmin) {
    return code_pair(__uint_as_float(v.x), __uint_as_float(v.y), rcp2, s_cell, dmin) |
           (code_pair(__uint_as_float(v.z), __uint_as_float(v.w), rcp2, s_cell, dmin) << 8);
}

// The same by exact division.
__device__ __forceinline__ uint32_t codes4_f32_exact(uint4 v, float am, const float* s_thr) {
    return code_byte_exact(__uint_as_float(v.x), __uint_as_float(v.y), am, s_thr) |
           (code_byte_exact(__uint_as_float(v.z), __uint_as_float(v.w), am, s_thr) << 8);
}

// Four consecutive words of one fp32 block (16 values) against its absmax:
// 8 packed bytes, one reciprocal, the cell table, and the exact path for all
// four words if any quotient lies within the guard of its entry (or the
// absmax is subnormal, where the reciprocal may overflow).
__device__ __forceinline__ uint2 quantize16_f32_fast(const uint4 (&v)[4], float am, const float* s_thr,
                                                     const uint32_t* s_cell) {
    if (am == 0.0f) return make_uint2(0x77777777u, 0x77777777u);
    float dmin = 0.0f;
    uint2 out = make_uint2(0u, 0u);
    if (am >= kMinNormal) {
        const float rcp = __frcp_rn(am);
        const uint64_t rcp2 = pack_f32x2(rcp, rcp);
        dmin = __int_as_float(0x7f800000);
        out.x = codes4_f32(v[0], rcp2, s_cell, dmin) | (codes4_f32(v[1], rcp2, s_cell, dmin) << 16);
        out.y = codes4_f32(v[2], rcp2, s_cell, dmin) | (codes4_f32(v[3], rcp2, s_cell, dmin) << 16);
    }
    if (dmin > kGuard) return out;
    return make_uint2(codes4_f32_exact(v[0], am, s_thr) | (codes4_f32_exact(v[1], am, s_thr) << 16),
                      codes4_f32_exact(v[2], am, s_thr) | (codes4_f32_exact(v[3], am, s_thr) << 16));
}

// Per-halfword unsigned max of two words of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Largest 15-bit magnitude pattern among the 16 16-bit values of two 16-byte
// words, reduced pairwise on both halves at once.  Finite bf16 and fp16
// magnitudes both order like their 15-bit patterns.
__device__ __forceinline__ uint32_t absmax_bits16(uint4 a, uint4 b) {
    constexpr uint32_t M = 0x7fff7fffu;
    const uint32_t m2 = max_u16x2(max_u16x2(max_u16x2(a.x & M, a.y & M), max_u16x2(a.z & M, a.w & M)),
                                  max_u16x2(max_u16x2(b.x & M, b.y & M), max_u16x2(b.z & M, b.w & M)));
    return max(m2 & 0xffffu, m2 >> 16);
}

constexpr int kQuantThreads = 256;

// Vectorized quantizer for whole blocks of a 16-bit type DT.  A warp tile is
// 1 KB (8 blocks): lane t owns the 16-byte words 2t and 2t + 1, so 4 lanes
// share a block, reduce its absmax with 2 shuffles and each takes one
// reciprocal for its 16 values.  Finite bf16 and fp16 magnitudes order like
// their 15-bit patterns, so the absmax is an integer max over (bits &
// 0x7fff).  nwords (a multiple of 8) covers whole blocks of the numel values;
// each lane writes its 8 packed bytes at once.
template <int DT>
__global__ void __launch_bounds__(kQuantThreads)
quantize_vec_kernel(const uint4* __restrict__ w, int64_t nwords, uint2* __restrict__ packed,
                    float* __restrict__ absmax, int64_t numel, uint32_t* err) {
    __shared__ float s_thr[16];
    __shared__ uint32_t s_cell[64];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    if (threadIdx.x < 64) s_cell[threadIdx.x] = c_cell[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kQuantThreads) >> 5;
    const int64_t npairs = nwords >> 1;          // word pairs; 4 per block
    const int64_t ntiles = (npairs + 31) >> 5;
    // the next tile's words are loaded before this one's are converted, so
    // each warp keeps a DRAM round trip in flight while it computes
    auto load = [&](int64_t t, uint4& a, uint4& b) {
        const int64_t pr = (t << 5) + lane;
        if (t < ntiles && pr < npairs && in_bounds(err, 2 * pr + 1, numel / 8)) {
            a = ldg_nc_v4(w + 2 * pr);
            b = ldg_nc_v4(w + 2 * pr + 1);
        } else {
            a = b = make_uint4(0, 0, 0, 0);
        }
    };
    uint4 a, b, na, nb;
    if (warp < ntiles) load(warp, na, nb);
    for (int64_t t = warp; t < ntiles; t += nwarps) {
        a = na;
        b = nb;
        if (t + nwarps < ntiles) load(t + nwarps, na, nb);
        const int64_t pr = (t << 5) + lane;
        uint32_t m = absmax_bits16(a, b);
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if (pr < npairs) {
            if (in_bounds(err, pr, numel / 16)) packed[pr] = quantize16_fast<DT>(a, b, m, s_thr, s_cell);
            if ((lane & 3) == 0 && in_bounds(err, pr >> 2, (numel + kBlock - 1) / kBlock))
                absmax[pr >> 2] = am_of<DT>(m);
        }
    }
}

// Vectorized quantizer for whole blocks of fp32.  A warp tile is 2 KB (8
// blocks): lane t owns the 16-byte words 4t .. 4t + 3 (16 values), so 4 lanes
// share a block, reduce its absmax with 2 shuffles and each takes one
// reciprocal for its 16 values.  Finite fp32 magnitudes order like their
// 31-bit patterns.  nwords (a multiple of 16) covers whole blocks of the
// numel values; each lane writes its 8 packed bytes at once.
__global__ void __launch_bounds__(kQuantThreads)
quantize_vec_f32_kernel(const uint4* __restrict__ w, int64_t nwords, uint2* __restrict__ packed,
                        float* __restrict__ absmax, int64_t numel, uint32_t* err) {
    __shared__ float s_thr[16];
    __shared__ uint32_t s_cell[64];
    if (threadIdx.x < 16) s_thr[threadIdx.x] = c_thr[threadIdx.x];
    if (threadIdx.x < 64) s_cell[threadIdx.x] = c_cell[threadIdx.x];
    __syncthreads();
    pdl_wait();                 // the previous kernel on the stream has finished
    pdl_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kQuantThreads + threadIdx.x) >> 5;
    const int64_t nwarps = (static_cast<int64_t>(gridDim.x) * kQuantThreads) >> 5;
    const int64_t nquads = nwords >> 2;          // word quads; 4 per block
    const int64_t ntiles = (nquads + 31) >> 5;
    // the next tile's words are loaded before this one's are converted
    auto load = [&](int64_t t, uint4 (&v)[4]) {
        const int64_t qd = (t << 5) + lane;
        const bool ok = t < ntiles && qd < nquads && in_bounds(err, 4 * qd + 3, numel / 4);
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = ok ? ldg_nc_v4(w + 4 * qd + i) : make_uint4(0, 0, 0, 0);
    };
    uint4 v[4], nv[4];
    if (warp < ntiles) load(warp, nv);
    for (int64_t t = warp; t < ntiles; t += nwarps) {
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = nv[i];
        if (t + nwarps < ntiles) load(t + nwarps, nv);
        const int64_t qd = (t << 5) + lane;
        uint32_t m = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            m = max(m, max(max(v[i].x & 0x7fffffffu, v[i].y & 0x7fffffffu), max(v[i].z & 0x7fffffffu, v[i].w & 0x7fffffffu)));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 1));
        m = max(m, __shfl_xor_sync(0xffffffffu, m, 2));
        if (qd < nquads) {
            const float am = __uint_as_float(m);
            if (in_bounds(err, qd, numel / 16)) packed[qd] = quantize16_f32_fast(v, am, s_thr, s_cell);
            if ((lane & 3) == 0 && in_bounds(err, qd >> 2, (numel + kBlock - 1) / kBlock)) absmax[qd >> 2] = am;
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
    constexpr int kPerWord = DT == kF32 ? 4 : 8;  // elements per 16-byte word
    cudaError_t e = cudaSuccess;
    const int64_t nblocks = (numel + kBlock - 1) / kBlock;
    const int64_t full = numel / kBlock;
    // each lane of the vectorized kernels stores 8 packed bytes at once
    const bool aligned = (reinterpret_cast<uintptr_t>(w) % 16 == 0) &&
                         (reinterpret_cast<uintptr_t>(packed) % 8 == 0) &&
                         (reinterpret_cast<uintptr_t>(absmax) % 4 == 0);
    int64_t scalar_from = 0;
    if (aligned && full > 0) {
        const int64_t nwords = full * (kBlock / kPerWord);
        // warp tiles: 128 words (32 quads) of fp32, 64 words (32 pairs) of a 16-bit type
        const int64_t ntiles = DT == kF32 ? (nwords + 127) / 128 : (nwords + 63) / 64;
        const int64_t warps_per_cta = kQuantThreads / 32;
        if constexpr (DT == kF32) {
            const int grid = grid_for(dev, reinterpret_cast<const void*>(quantize_vec_f32_kernel), kQuantThreads,
                                      (ntiles + warps_per_cta - 1) / warps_per_cta);
            e = launch_pdl(quantize_vec_f32_kernel, grid, kQuantThreads, 0, s, static_cast<const uint4*>(w), nwords,
                           reinterpret_cast<uint2*>(packed), absmax, numel, dev.err_word);
        } else {
            const int grid = grid_for(dev, reinterpret_cast<const void*>(quantize_vec_kernel<DT>), kQuantThreads,
                                      (ntiles + warps_per_cta - 1) / warps_per_cta);
            e = launch_pdl(quantize_vec_kernel<DT>, grid, kQuantThreads, 0, s, static_cast<const uint4*>(w), nwords,
                           reinterpret_cast<uint2*>(packed), absmax, numel, dev.err_word);
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
