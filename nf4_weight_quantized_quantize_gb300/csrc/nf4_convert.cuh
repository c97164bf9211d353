// nf4_convert.cuh -- the pieces the fused NF4 GEMM kernels share: the
// packed-weight producer (TMA box of packed bytes plus the fp32 block scales)
// and the converters' codebook expansion of packed bytes into the compute
// dtype (register byte permutes, or a per-lane byte table in shared memory).
#pragma once

#include "nf4_device.cuh"

namespace nf4 {

constexpr int kBK = 64;                    // K per slice = one NF4 block = one 128-byte activation row
constexpr int kPackedRow = kBK / 2;        // 32 packed bytes per weight row per slice

// fp32 weights: one packed word (bytes in address order, code 2j in the high
// nibble of byte j) to eight values C[code] * absmax in fp32 -- the fp32
// dequantizer's values -- rounded to tf32, the part the MMA reads.  `code`
// is the fp32 codebook in shared memory.
__device__ __forceinline__ void expand8_f32(uint32_t p, const float* code, float am, uint32_t* o) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t b = (p >> (8 * j)) & 0xffu;
        o[2 * j] = to_tf32(code[b >> 4] * am);
        o[2 * j + 1] = to_tf32(code[b & 15u] * am);
    }
}

// pfull[p] completes on the TMA bytes plus kPfullArrivals arrivals: the
// weight producer lane's expect-tx arrive and one cp.async arrive per lane.
constexpr int kPfullArrivals = 1 + 32;

// The 16 codebook values of type DT split into low bytes (l) and high bytes
// (h), four codes per register: byte i of l[q] is the low byte of DT(C[4q + i]).
struct CodebookRegs {
    uint32_t l[4], h[4];
};

template <int DT>
__device__ __forceinline__ CodebookRegs codebook_regs() {
    CodebookRegs cb;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        cb.l[q] = 0;
        cb.h[q] = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t bits = round16<DT>(c_code[4 * q + i]);
            cb.l[q] |= (bits & 0xffu) << (8 * i);
            cb.h[q] |= (bits >> 8) << (8 * i);
        }
    }
    return cb;
}

// Look up the four codes held in the low 16 bits of s (nibble k = code k).
// A byte permute picks byte (code & 7) out of eight table bytes; two of them
// cover codes 0-7 and 8-15, and a third picks per byte by code bit 3.  Byte k
// of `lo` / `hi` is the low / high byte of bf16(C[code k]).
__device__ __forceinline__ void lookup4(uint32_t s, const CodebookRegs& cb, uint32_t& lo, uint32_t& hi) {
    const uint32_t s7 = s & 0x7777u;
    const uint32_t pick = ((s >> 1) & 0x4444u) | 0x3210u;
    lo = prmt(prmt(cb.l[0], cb.l[1], s7), prmt(cb.l[2], cb.l[3], s7), pick);
    hi = prmt(prmt(cb.h[0], cb.h[1], s7), prmt(cb.h[2], cb.h[3], s7), pick);
}

// One packed word (bytes in address order; byte j holds code 2j in its high
// nibble) to four words of two DT values, element 2i in the low half of word
// i, each scaled by `am2`.  A product of two bf16 (or two fp16) values is
// exact in fp32, so each value is DT_rne(float(DT(C)) * absmax) -- the
// dequantizer's value -- whenever absmax is a DT value, which every absmax
// nf4_quantize writes for a DT weight is (the max of DT magnitudes).
template <int DT>
__device__ __forceinline__ void expand8(uint32_t p, const CodebookRegs& cb, uint32_t am2, uint32_t* o) {
    uint32_t lo, hi;
    lookup4(p, cb, lo, hi);              // nibbles: code1, code0, code3, code2
    o[0] = mul2<DT>(prmt(lo, hi, 0x4051u), am2);
    o[1] = mul2<DT>(prmt(lo, hi, 0x6273u), am2);
    lookup4(p >> 16, cb, lo, hi);        // code5, code4, code7, code6
    o[2] = mul2<DT>(prmt(lo, hi, 0x4051u), am2);
    o[3] = mul2<DT>(prmt(lo, hi, 0x6273u), am2);
}

// expand8 through the shared-memory byte table instead of register permutes:
// per packed byte one table load (the DT codebook values of its two codes,
// element 2i in the low half) and one paired multiply.  `lut_lane` points at
// this lane's column of the replicated table (entry b at lut_lane[32 b]).
template <int DT>
__device__ __forceinline__ void expand8_lut(uint32_t p, const uint32_t* lut_lane, uint32_t am2, uint32_t* o) {
    o[0] = mul2<DT>(lut_lane[32u * prmt(p, 0u, 0x4440u)], am2);
    o[1] = mul2<DT>(lut_lane[32u * prmt(p, 0u, 0x4441u)], am2);
    o[2] = mul2<DT>(lut_lane[32u * prmt(p, 0u, 0x4442u)], am2);
    o[3] = mul2<DT>(lut_lane[32u * prmt(p, 0u, 0x4443u)], am2);
}

// Whether a converter warp of a tcgen05 kernel reports stage st as
// converted.  Always true in the library.  A test build (-DNF4_TEST_DROP_CONVERTED_ARRIVE) withholds the
// report for stage 0 -- a flag that nothing sets -- so the MMA issuer's bounded
// wait runs out and the timeout path (error word, drain, TMEM release, early
// exit) can be checked on a GPU without faulting or hanging it.
__device__ __forceinline__ bool report_converted(int st) {
#ifdef NF4_TEST_DROP_CONVERTED_ARRIVE
    return st != 0;
#else
    (void)st;
    return true;
#endif
}

// Named barriers among the converter warps of a tcgen05 kernel (barrier 0 is __syncthreads).
// and_all: every converter thread arrives, each with its predicate; returns
// whether all of them were true.
__device__ __forceinline__ bool converters_and_all(bool pred, int threads) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(pred)), "r"(threads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void converters_sync(int threads) {
    asm volatile("bar.sync 2, %0;" ::"r"(threads) : "memory");
}

// Wait (bounded) for the copies a producer issued into the last `slots`
// stages of its ring to land, so no TMA or cp.async write targets shared
// memory after exit.
__device__ __forceinline__ void drain_ring(uint32_t bar0, int slots, int issued, uint32_t* err) {
    int dummy = 0;   // a fresh flag: the CTA-wide abort is already raised here
    for (int st = max(0, issued - slots); st < issued; ++st)
        if (!mbar_wait(bar0 + 8u * (st % slots), (st / slots) & 1, err, &dummy, kErrTimeoutDrain)) break;
}

// Weight producer warp, one stage: lane 0 arms pfull[p] with the TMA byte
// count and loads the packed tile of the whole stage -- one box of 32 * KS
// bytes x ROWS rows from weight row n0, or, for a gate/up PAIR, two boxes of
// ROWS / 2 rows from rows n0 (gate) and n1 (up) -- and every lane copies
// scales with 4-byte cp.async -- K-slice h, rows lane, lane + 32, ... to
// am_dst[h][row] -- and arrives on pfull[p] when its copies land.  Rows of a
// box at or past n_lim (the rows of one half) and K-slices past the weight's
// last block copy a harmless in-range scale (their products are never stored
// or multiply zeros).  absmax holds am_extent scales.
template <int ROWS, int KS, bool PAIR>
__device__ __forceinline__ void produce_weights(uint32_t full, int lane, uint32_t tx_bytes, const CUtensorMap* tm_w,
                                                uint32_t p_dst, int p_col0, int n0, int n1, int n_lim,
                                                uint32_t am_dst, const float* absmax, int am_pitch, int kb_abs0,
                                                int64_t am_extent, uint32_t* err) {
    constexpr int H = PAIR ? ROWS / 2 : ROWS;   // rows per box
    if (lane == 0) {
        mbar_arrive_expect_tx(full, tx_bytes);
        tma_load_2d(p_dst, tm_w, full, p_col0, n0);
        if constexpr (PAIR) tma_load_2d(p_dst + H * kPackedRow * KS, tm_w, full, p_col0, n1);
    }
#pragma unroll
    for (int h = 0; h < KS; ++h) {
        const bool kb_ok = kb_abs0 + h < am_pitch;
#pragma unroll
        for (int i = lane; i < ROWS; i += 32) {
            const int il = i < H ? i : i - H;          // row within its box
            const int n = (i < H ? n0 : n1) + il;
            const bool ok = n0 + il < n_lim && kb_ok;
            const int64_t src = ok ? static_cast<int64_t>(n) * am_pitch + kb_abs0 + h : 0;
            if (in_bounds(err, src, am_extent)) cp_async_4(am_dst + 4u * (h * ROWS + i), absmax + src);
        }
    }
    cp_async_arrive_noinc(full);
}

}  // namespace nf4
