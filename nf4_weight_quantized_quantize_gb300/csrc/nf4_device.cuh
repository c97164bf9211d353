// nf4_device.cuh -- device-side constants and PTX wrappers shared by the
// libnf4 kernels (sm_103a only).
//
// Format (diffuseR pull request "Gemma3 NF4 on GPU" #39, Summary, with the
// format fixed as documented in include/nf4.h): 16-value NF4 codebook,
// 64-element blocks, fp32 absmax, element 2j in the high nibble of byte j.
#pragma once

#include <bit>
#include <cstdint>
#include <type_traits>

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "nf4_launch.h"

#ifndef NF4_WAIT_LIMIT_NS
// A bounded wait gives up after this long (nanoseconds of %globaltimer).
#define NF4_WAIT_LIMIT_NS 1000000000ull
#endif

namespace nf4 {

constexpr int kBlock = 64;

// NormalFloat-4 codebook of QLoRA (arXiv:2305.14314, appendix), ascending.
constexpr float kCode[16] = {
    -1.0f,
    -0.6961928009986877f,
    -0.5250730514526367f,
    -0.39491748809814453f,
    -0.28444138169288635f,
    -0.18477343022823334f,
    -0.09105003625154495f,
    0.0f,
    0.07958029955625534f,
    0.16093020141124725f,
    0.24611230194568634f,
    0.33791524171829224f,
    0.44070982933044434f,
    0.5626170039176941f,
    0.7229568362236023f,
    1.0f,
};

// Decision threshold between codes j and j+1.  The exact midpoint
// m = (C[j] + C[j+1]) / 2 is computed in fp64 (exact for two fp32 values).
// If m is an fp32 value the threshold is m; otherwise it is the largest fp32
// below m.  For every fp32 n, n > threshold exactly when n > m, so
// code(n) = #{ j : n > thr(j) } is the nearest codebook index with ties going
// to the lower index.
constexpr float threshold(int j) {
    double m = (static_cast<double>(kCode[j]) + static_cast<double>(kCode[j + 1])) * 0.5;
    float f = static_cast<float>(m);
    if (static_cast<double>(f) > m) {
        uint32_t u = std::bit_cast<uint32_t>(f);
        u = (f > 0.0f) ? u - 1u : u + 1u;   // one step toward -inf
        f = std::bit_cast<float>(u);
    }
    return f;
}

// Device copies (constant bank).  c_thr[15] = +inf pads the table to 16 so a
// binary search can index it without a bound check.
static __constant__ float c_code[16] = {
    kCode[0], kCode[1], kCode[2],  kCode[3],  kCode[4],  kCode[5],  kCode[6],  kCode[7],
    kCode[8], kCode[9], kCode[10], kCode[11], kCode[12], kCode[13], kCode[14], kCode[15],
};
static __constant__ float c_thr[16] = {
    threshold(0),  threshold(1),  threshold(2),  threshold(3),  threshold(4),
    threshold(5),  threshold(6),  threshold(7),  threshold(8),  threshold(9),
    threshold(10), threshold(11), threshold(12), threshold(13), threshold(14),
    __builtin_huge_valf(),
};

__device__ __forceinline__ void record_error(uint32_t* err, uint32_t code) {
    if (err) atomicCAS(err, 0u, code);
}

// Checked build.  With -DNF4_CHECKED every global access that is not a TMA
// tensor copy first tests its index against the extent of the buffer it
// addresses, both in units of the access.  An index outside [0, extent)
// records kErrBounds and the access is skipped (a skipped load reads zero),
// so an indexing mistake becomes a status instead of a fault.  TMA tensor
// copies need no test: the hardware clips every box to its tensor map, whose
// extents the host sets from the validated sizes.  In the normal build the
// test is the constant true and compiles away.  The test switch
// NF4_TEST_SHRINK_EXTENT tests against extent - 1 instead, so the last
// element of every checked buffer reports while no access leaves its buffer.
#if defined(NF4_CHECKED)
__device__ __forceinline__ bool in_bounds(uint32_t* err, int64_t i, int64_t extent) {
#if defined(NF4_TEST_SHRINK_EXTENT)
    extent -= 1;
#endif
    if (i >= 0 && i < extent) return true;
    record_error(err, kErrBounds);
    return false;
}
#else
__device__ __forceinline__ constexpr bool in_bounds(uint32_t*, int64_t, int64_t) { return true; }
#endif

__device__ __forceinline__ uint64_t globaltimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- loads

__device__ __forceinline__ uint32_t ldg_nc_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ float ldg_nc_f32(const float* p) {
    float v;
    asm volatile("ld.global.nc.L1::no_allocate.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ void stg_v4(void* p, uint4 v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// ---------------------------------------------------------------- element types

// The compute dtype of weights, activations and outputs.  bf16 and fp16
// travel as 16-bit patterns (two per 32-bit word, the element at the lower
// address in the low half), fp32 as itself.
enum : int { kBF16 = 0, kF16 = 1, kF32 = 2 };

// Two fp32 values -> one word of two 16-bit values of type DT (first in the
// low half), each rounded to nearest even by the hardware conversion.
template <int DT>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
    static_assert(DT == kBF16 || DT == kF16, "16-bit types");
    uint32_t r;
    if constexpr (DT == kBF16) {
        __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
        r = *reinterpret_cast<uint32_t*>(&v);
    } else {
        __half2 v = __floats2half2_rn(lo, hi);
        r = *reinterpret_cast<uint32_t*>(&v);
    }
    return r;
}

// A word of two 16-bit values of type DT -> the two fp32 values (exact).
template <int DT>
__device__ __forceinline__ float2 unpack2(uint32_t w) {
    static_assert(DT == kBF16 || DT == kF16, "16-bit types");
    if constexpr (DT == kBF16) {
        return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
    } else {
        __half2 h = *reinterpret_cast<__half2*>(&w);
        return __half22float2(h);
    }
}

// One fp32 -> the 16-bit pattern of type DT, rounded to nearest even.
template <int DT>
__device__ __forceinline__ uint16_t round16(float v) {
    static_assert(DT == kBF16 || DT == kF16, "16-bit types");
    if constexpr (DT == kBF16)
        return __bfloat16_as_ushort(__float2bfloat16_rn(v));
    else
        return __half_as_ushort(__float2half_rn(v));
}

// A LUT entry for packed byte b: DT(C[b >> 4]) in the low half (the element
// at the lower address) and DT(C[b & 15]) in the high half.
template <int DT = kBF16>
__device__ __forceinline__ uint32_t lut_entry(uint32_t b) {
    return pack2<DT>(c_code[b >> 4], c_code[b & 15]);
}

// Scale one LUT entry by the block absmax: each value widened to fp32, one
// fp32 multiply, one rounding back to DT.
template <int DT = kBF16>
__device__ __forceinline__ uint32_t scale_entry(uint32_t e, float am) {
    const float2 v = unpack2<DT>(e);
    return pack2<DT>(v.x * am, v.y * am);
}

// ---------------------------------------------------------------- shared arithmetic

// Whether an fp32 absmax is exactly a value of type DT (then one paired DT
// multiply gives the correctly rounded product).
template <int DT>
__device__ __forceinline__ bool exact_in(float am) {
    if constexpr (DT == kBF16)
        return (__float_as_uint(am) & 0xffffu) == 0u;
    else
        return __half2float(__float2half_rn(am)) == am;
}


__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Multiply of two words of two 16-bit values of type DT (bf16 or fp16),
// one round-to-nearest-even per half.
template <int DT>
__device__ __forceinline__ uint32_t mul2(uint32_t a, uint32_t b) {
    uint32_t d;
    if constexpr (DT == kBF16)
        asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    else
        asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// GELU, tanh form (Hendrycks and Gimpel, "Gaussian Error Linear Units",
// section 2): x/2 * (1 + tanh(y)), y = sqrt(2/pi) * (x + 0.044715 x^3), in
// fp32 through the identity (1 + tanh(y)) / 2 = 1 / (1 + e^(-2y)):
//   gelu(x) = x / (1 + 2^(x (c0 + c1 x^2))),  c0 = -2 sqrt(2/pi) log2(e),
//   c1 = 0.044715 c0,
// with the hardware base-2 exponential and reciprocal (a few 1e-7 relative
// error; no cancellation, the denominator is at least 1).  For large negative
// x the power overflows to +inf, its reciprocal is 0 and the result -0, the
// limit.
__device__ __forceinline__ float gelu_tanh(float x) {
    const float a = x * fmaf(-0.10294324159622192f, x * x, -2.302208185195923f);
    float t, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(t) : "f"(a));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + t));
    return x * r;
}

// Element bytes of a compute dtype.
template <int DT>
constexpr int elem_bytes() {
    return DT == kF32 ? 4 : 2;
}

// Store one output value in the compute dtype (16-bit types: one rounding
// to nearest even).
template <int DT>
__device__ __forceinline__ void store_out(void* y, int64_t i, float v) {
    if constexpr (DT == kF32)
        static_cast<float*>(y)[i] = v;
    else
        static_cast<uint16_t*>(y)[i] = round16<DT>(v);
}

// Store 16 values of output column n, rows m_first .. m_first + 15 of a
// row-major output [M, ld], rounded to DT (fp32: as they are); rows at or
// past M are not stored (a run may start past M: it stores nothing).  One
// pointer advanced by a row per value; the row bound is checked once for the
// whole run unless it ends past M.  (Indexing every element from (m, n) cost
// the GEMM epilogues about half their time.)
template <int DT>
__device__ __forceinline__ void store_col16(void* y, int64_t ld, int m_first, int M, int n, const float (&v)[16],
                                            uint32_t* err) {
    if (m_first < M && (!in_bounds(err, n, ld) || !in_bounds(err, m_first, M))) return;
    using E = typename std::conditional<DT == kF32, float, uint16_t>::type;
    E* p = static_cast<E*>(y) + static_cast<int64_t>(m_first) * ld + n;
    auto cvt = [](float x) -> E {
        if constexpr (DT == kF32)
            return x;
        else
            return round16<DT>(x);
    };
    if (m_first + 15 < M) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            *p = cvt(v[i]);
            p += ld;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if (m_first + i < M) *p = cvt(v[i]);
            p += ld;
        }
    }
}

// ---------------------------------------------------------------- dependent launch

// Wait until the kernel this one was launched after (programmatic dependent
// launch, see launch_pdl) has completed and its memory is visible; a no-op
// for a normal launch.  Every kernel calls it before its first global access.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Let the next kernel on the stream start its prologue (it still waits for
// this one in pdl_wait before touching global memory).
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// NF4_WAIT_LIMIT_NS.  Gives up early when *abort becomes nonzero (another
// role of this CTA gave up).  On giving up, records `code` in the device
// error word, raises *abort and returns false.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint32_t* err,
                                          volatile int* abort, uint32_t code) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > NF4_WAIT_LIMIT_NS) {
            record_error(err, code);
            *abort = 1;
            return false;
        }
    }
}

// ---------------------------------------------------------------- TMA

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

// 2-D tiled load of box {x, y} into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                            int32_t x, int32_t y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

// 4-byte asynchronous global -> shared copy (cached in L1, so neighbouring
// scales of one row are fetched from L2 once).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Arrive on `bar` once every cp.async this thread issued so far has landed.
// The arrival is not pre-counted (.noinc): the barrier's expected count must
// include it.
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     dst_smem),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// D[tmem] (+)= A[tmem] . B[smem]^T: A (M = 128 rows, one per TMEM lane, K packed
// two bf16 per 32-bit column, lower K in the low half) read from tensor memory.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// mma_bf16_ts with the B descriptor passed as its two 32-bit halves, so a
// caller stepping through a tile adds one 32-bit offset per MMA.
__device__ __forceinline__ void mma_bf16_ts2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 bd, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The same with kind::tf32: A (in TMEM) and B hold fp32 values of which the
// tensor core reads the tf32 part (sign, exponent, 10 fraction bits); one MMA
// covers K = 8 (32 bytes of a row, 8 TMEM columns of A).
__device__ __forceinline__ void mma_tf32_ts2(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t b_hi,
                                             uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b64 bd;\n\t"
        "setp.ne.b32 p, %5, 0;\n\t"
        "mov.b64 bd, {%2, %3};\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], bd, %4, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "r"(b_lo), "r"(b_hi), "r"(idesc), "r"(accumulate)
        : "memory");
}

// fp32 -> tf32, rounded to nearest (ties away from zero), as an fp32 bit
// pattern whose low 13 bits are zero.
__device__ __forceinline__ uint32_t to_tf32(float v) {
    uint32_t r;
    asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(v));
    return r;
}

// Each thread stores 32 consecutive 32-bit columns of its own TMEM lane
// (lane = 32 * (warp % 4) + lane id).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
        "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
        "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
        : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
        "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}

__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor for a K-major operand stored with the
// 128-byte swizzle: rows of 128 bytes (64 bf16), 8-row atoms 1024 bytes apart.
// Fields: start address >> 4 (bits 0-13), leading byte offset >> 4 (16-29,
// unused for swizzled K-major, set to 1), stride byte offset >> 4 (32-45),
// fixed 0b001 (46-48), base offset 0 (49-51), swizzle mode 2 = 128B (61-63).
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(1024u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(2u) << 61;
    return d;
}

// Instruction descriptor for kind::f16: A and B both bf16 (DT = kBF16) or
// both fp16 (DT = kF16) -- the two operands of one MMA always have the same
// type -- fp32 D, both K-major, no negation or sparsity; N >> 3 at bits
// 17-22, M >> 4 at bits 24-28.
template <int DT = kBF16>
__host__ __device__ constexpr uint32_t idesc_f16kind_f32(int M, int N) {
    static_assert(DT == kBF16 || DT == kF16, "kind::f16 operand types");
    constexpr uint32_t ab = DT == kBF16 ? 1u : 0u;   // operand format: 0 fp16, 1 bf16
    return (1u << 4)            // D format: f32
           | (ab << 7)          // A format
           | (ab << 10)         // B format
           | (0u << 15)         // A K-major
           | (0u << 16)         // B K-major
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (static_cast<uint32_t>(M >> 4) << 24);
}

// Instruction descriptor for kind::tf32: A and B tf32 (format 2), fp32 D,
// both K-major; the other fields as for kind::f16.
__host__ __device__ constexpr uint32_t idesc_tf32_f32(int M, int N) {
    return (1u << 4)            // D format: f32
           | (2u << 7)          // A format: tf32
           | (2u << 10)         // B format: tf32
           | (static_cast<uint32_t>(N >> 3) << 17)
           | (static_cast<uint32_t>(M >> 4) << 24);
}

}  // namespace nf4
