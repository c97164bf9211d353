// nf4_gemm.cu -- fused NF4 weight-only GEMM on the 5th-generation tensor
// cores: Y[M, N] = X[M, K] . deq(W)[N, K]^T, bf16 in, fp32 accumulate in TMEM,
// bf16 out.
//
// This is the forward of the NF4 linear module of the diffuseR page "Gemma3
// NF4 on GPU" (#39, Summary: ltx23_nf4_linear, dequantize then a dense matmul
// at the compute dtype).  Instead of dequantizing the whole weight to HBM and
// calling a dense GEMM, each CTA expands its packed weight tile through the
// byte lookup table in shared memory and feeds tcgen05.mma directly, so the
// weight crosses HBM at 0.5625 bytes per element.
//
// Two kernels:
//   gemm_kernel   (M >= 128): CTA tile 256 x 256 x 64, two M=128 MMAs per
//                 K-slice sharing one converted B tile, 512 TMEM columns.
//   skinny_kernel (M < 128): swap-AB -- the weight tile (128 rows of N) is the
//                 MMA A operand and the activations (M padded to a multiple of
//                 16) are B; split-K over CTAs into an fp32 workspace, then an
//                 ordered reduction kernel writes bf16 Y.
//
// Warp roles (both kernels): warp 0 lane 0 issues TMA loads (X and packed W),
// warp 1 allocates TMEM and lane 0 issues the MMAs, the remaining warps
// convert packed bytes to bf16 in the 128-byte-swizzled K-major layout the
// MMA reads, then run the epilogue (tcgen05.ld -> bf16 / fp32 -> global).
// Every wait is bounded (NF4_WAIT_LIMIT_NS); on expiry the CTA records an
// error code, drains what it has in flight and returns.
#include <algorithm>
#include <mutex>

#include <cudaTypedefs.h>

#include "nf4_device.cuh"
#include "nf4_launch.h"

namespace nf4 {

// ============================================================ shared pieces

constexpr int kBK = 64;                    // K per pipeline stage = one NF4 block = one 128-byte row
constexpr int kPackedRow = kBK / 2;        // 32 packed bytes per weight row per stage
constexpr int kLutCopies = 32;             // one copy of the byte LUT per lane
constexpr int kLutBytes = 256 * kLutCopies * 4;   // 32 KB

// Barriers of both kernels, in shared memory:
//   full[s1]  TMA landed (activations + packed weights of a K-slice)
//   empty[s1] the MMA of that K-slice completed: its ring slot may be refilled
//   conv[s2]  converter warps finished a converted-weight buffer
//   cfree[s2] the MMA reading that converted buffer completed
//   accum     the accumulator is final; drain: used only on the error path
struct Barriers {
    uint32_t base;
    int s1, s2;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t empty(int s) const { return base + 8u * (s1 + s); }
    __device__ uint32_t conv(int b) const { return base + 8u * (2 * s1 + b); }
    __device__ uint32_t cfree(int b) const { return base + 8u * (2 * s1 + s2 + b); }
    __device__ uint32_t accum() const { return base + 8u * (2 * s1 + 2 * s2); }
    __device__ uint32_t drain() const { return base + 8u * (2 * s1 + 2 * s2 + 1); }
    __host__ __device__ static constexpr int count(int a, int b) { return 2 * a + 2 * b + 2; }
};

// full[s] completes on the TMA bytes plus kFullArrivals arrivals: the
// producer lane's expect-tx arrive and one cp.async arrive per producer lane.
constexpr int kFullArrivals = 1 + 32;

__device__ __forceinline__ void init_barriers(const Barriers& bar, int conv_arrivals) {
    for (int s = 0; s < bar.s1; ++s) {
        mbar_init(bar.full(s), kFullArrivals);
        mbar_init(bar.empty(s), 1);
    }
    for (int b = 0; b < bar.s2; ++b) {
        mbar_init(bar.conv(b), conv_arrivals);
        mbar_init(bar.cfree(b), 1);
    }
    mbar_init(bar.accum(), 1);
    mbar_init(bar.drain(), 1);
}

// The byte LUT replicated once per lane: word (b * 32 + lane) holds the
// bf16x2 codebook pair of byte b.  Lane l only reads copy l, which lives in
// bank l, so the 32 random lookups of a warp never conflict.
__device__ __forceinline__ void build_lut(uint32_t* lut, int tid, int nthreads) {
    for (int i = tid; i < 256 * kLutCopies; i += nthreads) lut[i] = lut_entry(static_cast<uint32_t>(i) >> 5);
}

// bf16x2 multiply with one round-to-nearest-even per half.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Eight weights (one packed 32-bit word, bytes in address order) to four
// bf16x2 words.  The scale enters as bf16x2 `am2`; a bf16 x bf16 product is
// exact in fp32, so each half equals bf16_rne(float(bf16(C)) * absmax) -- the
// dequantizer's value -- whenever absmax is a bf16 value, which every absmax
// nf4_quantize writes is (the max of bf16 magnitudes).
__device__ __forceinline__ uint4 expand8(uint32_t p, const uint32_t* lut_lane, uint32_t am2) {
    uint4 o;
    o.x = bf16x2_mul(lut_lane[(p & 0xffu) * kLutCopies], am2);
    o.y = bf16x2_mul(lut_lane[((p >> 8) & 0xffu) * kLutCopies], am2);
    o.z = bf16x2_mul(lut_lane[((p >> 16) & 0xffu) * kLutCopies], am2);
    o.w = bf16x2_mul(lut_lane[(p >> 24) * kLutCopies], am2);
    return o;
}

// Store one 16-byte chunk c of row r of a 128-byte-swizzled K-major tile
// (the layout TMA's 128-byte swizzle produces and the MMA descriptor reads).
__device__ __forceinline__ void st_sw128(uint8_t* tile, int r, int c, uint4 v) {
    *reinterpret_cast<uint4*>(tile + r * 128 + ((c ^ (r & 7)) << 4)) = v;
}

// Whether a converter warp reports K-slice kb as converted.  Always true in
// the library.  A test build (-DNF4_TEST_DROP_CONVERTED_ARRIVE) withholds the
// report for slice 0 -- a flag that nothing sets -- so the MMA issuer's bounded
// wait runs out and the timeout path (error word, drain, TMEM release, early
// exit) can be checked on a GPU without faulting or hanging it.
__device__ __forceinline__ bool report_converted(int kb) {
#ifdef NF4_TEST_DROP_CONVERTED_ARRIVE
    return kb != 0;
#else
    (void)kb;
    return true;
#endif
}

// Wait (bounded) for the copies a producer issued into the last `s1`
// K-slices to land, so no TMA write targets shared memory after exit.
__device__ __forceinline__ void drain_tma(const Barriers& bar, int issued, uint32_t* err) {
    int dummy = 0;   // a fresh flag: the CTA-wide abort is already raised here
    for (int kb = max(0, issued - bar.s1); kb < issued; ++kb)
        if (!mbar_wait(bar.full(kb % bar.s1), (kb / bar.s1) & 1, err, &dummy, kErrTimeoutDrain)) break;
}

// Error-path exit of the MMA issuer: wait (bounded) until every MMA it issued
// has completed, so TMEM can be released.
__device__ __forceinline__ void drain_mma(const Barriers& bar, uint32_t* err) {
    int dummy = 0;
    mma_commit(bar.drain());
    mbar_wait(bar.drain(), 0, err, &dummy, kErrTimeoutDrain);
}

// Producer warp, one K-slice: lane 0 arms full[s] with the TMA byte count and
// issues the two tile loads; every lane copies the scales of rows
// lane, lane + 32, ... of the slice into `am_dst` with 4-byte cp.async and
// arrives on full[s] when its copies land.  Rows past N copy a harmless
// in-range scale (their outputs are never stored).
template <int ROWS>
__device__ __forceinline__ void produce_slice(const Barriers& bar, int s, int lane, uint32_t tx_bytes,
                                              const CUtensorMap* tm_x, uint32_t x_dst, int x_col, int x_row,
                                              const CUtensorMap* tm_w, uint32_t p_dst, int p_col, int n0,
                                              uint32_t am_dst, const float* absmax, int N, int64_t am_pitch,
                                              int kb_abs) {
    if (lane == 0) {
        mbar_arrive_expect_tx(bar.full(s), tx_bytes);
        tma_load_2d(x_dst, tm_x, bar.full(s), x_col, x_row);
        tma_load_2d(p_dst, tm_w, bar.full(s), p_col, n0);
    }
#pragma unroll
    for (int i = lane; i < ROWS; i += 32) {
        const int n = n0 + i;
        const float* src = absmax + (n < N ? static_cast<int64_t>(n) * am_pitch + kb_abs : 0);
        cp_async_4(am_dst + 4u * i, src);
    }
    cp_async_arrive_noinc(bar.full(s));
}

// ============================================================ large-M kernel

#ifndef NF4_BIG_S1
#define NF4_BIG_S1 3
#endif
#ifndef NF4_BIG_S2
#define NF4_BIG_S2 2
#endif
#ifndef NF4_BIG_CONV_WARPS
#define NF4_BIG_CONV_WARPS 16
#endif

namespace big {
constexpr int BM = 256;
constexpr int BN = 256;
constexpr int S1 = NF4_BIG_S1;               // activation + packed-weight + scale ring
constexpr int S2 = NF4_BIG_S2;               // converted-weight buffers
constexpr int X_BYTES = BM * kBK * 2;        // 32 KB
constexpr int B_BYTES = BN * kBK * 2;        // 32 KB
constexpr int P_BYTES = BN * kPackedRow;     // 8 KB
constexpr int AM_BYTES = BN * 4;             // 1 KB of fp32 scales
constexpr int CONV_WARPS = NF4_BIG_CONV_WARPS;   // 8: one converter thread per weight row, 16: two
constexpr int ROW_SPLIT = CONV_WARPS / 8;    // converter threads per weight row
constexpr int COL_SPLIT = CONV_WARPS / 8;    // epilogue warps per (accumulator, lane quarter)
constexpr int THREADS = 64 + CONV_WARPS * 32;
constexpr int TMEM_COLS = 512;               // two 128 x 256 fp32 accumulators
constexpr int OFF_X = 0;
constexpr int OFF_B = OFF_X + S1 * X_BYTES;
constexpr int OFF_P = OFF_B + S2 * B_BYTES;
constexpr int OFF_LUT = OFF_P + S1 * P_BYTES;
constexpr int OFF_AM = OFF_LUT + kLutBytes;
constexpr int OFF_BAR = OFF_AM + S1 * AM_BYTES;
constexpr int NUM_BARS = Barriers::count(S1, S2);
constexpr size_t SMEM = 1024 + OFF_BAR + NUM_BARS * 8 + 16;
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(OFF_B % 1024 == 0 && X_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "128B-swizzle tiles need 1 KB alignment");
static_assert(CONV_WARPS == 8 || CONV_WARPS == 16, "converter warps: 8 or 16");
}  // namespace big

struct GemmArgs {
    const float* absmax;  // [N, K/64]
    uint16_t* y;          // [M, N]
    int M, N, K;
    uint32_t* err;
};

__global__ void __launch_bounds__(big::THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
            const GemmArgs args) {
    using namespace big;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + OFF_LUT);
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Barriers bar{smem_u32(bar_mem), S1, S2};

    auto x_tile = [&](int s) { return smem + OFF_X + s * X_BYTES; };
    auto b_tile = [&](int b) { return smem + OFF_B + b * B_BYTES; };
    auto p_tile = [&](int s) { return smem + OFF_P + s * P_BYTES; };
    auto am_tile = [&](int s) { return reinterpret_cast<const float*>(smem + OFF_AM + s * AM_BYTES); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles run m-fastest: CTAs resident together share weight tiles through L2
    const int m_tiles = (args.M + BM - 1) / BM;
    const int m0 = static_cast<int>(blockIdx.x % m_tiles) * BM;
    const int n0 = static_cast<int>(blockIdx.x / m_tiles) * BN;
    const int nk = args.K / kBK;

    if (threadIdx.x == 0) {
        init_barriers(bar, CONV_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
        tmem_relinquish();
    }
    if (warp >= 2) build_lut(lut, threadIdx.x - 64, CONV_WARPS * 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- producer warp
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S1;
            bool ok = true;
            if (kb >= S1)
                ok = mbar_wait(bar.empty(s), ((kb / S1) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            produce_slice<BN>(bar, s, lane, X_BYTES + P_BYTES, &tm_x, smem_u32(x_tile(s)), kb * kBK, m0, &tm_w,
                              smem_u32(p_tile(s)), kb * kPackedRow, n0, smem_u32(am_tile(s)), args.absmax, args.N,
                              nk, kb);
            ++issued;
        }
        if (*abort_flag && lane == 0) drain_tma(bar, issued, args.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
            bool ok = true;
            for (int kb = 0; kb < nk && ok; ++kb) {
                const int s = kb % S1;
                const int b = kb % S2;
                ok = mbar_wait(bar.full(s), (kb / S1) & 1, args.err, abort_flag, kErrTimeoutFull) &&
                     mbar_wait(bar.conv(b), (kb / S2) & 1, args.err, abort_flag, kErrTimeoutConverted);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(x_tile(s));
                const uint32_t b0 = smem_u32(b_tile(b));
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j) {
                    const uint64_t bd = smem_desc_sw128(b0 + 32 * j);
                    const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                    mma_bf16(tmem, smem_desc_sw128(a0 + 32 * j), bd, idesc, acc);
                    mma_bf16(tmem + BN, smem_desc_sw128(a0 + 128 * 128 + 32 * j), bd, idesc, acc);
                }
                mma_commit(bar.empty(s));
                mma_commit(bar.cfree(b));
            }
            if (ok)
                mma_commit(bar.accum());
            else
                drain_mma(bar, args.err);
        }
    } else {
        // ---------------- converters (ROW_SPLIT per weight row), then epilogue
        const int t = threadIdx.x - 64;
        const int r = t & (BN - 1);              // weight row within the tile
        const int h = t >> 8;                    // part of the slice: 32 / ROW_SPLIT packed bytes
        const uint32_t* lut_lane = lut + lane;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S1;
            const int b = kb % S2;
            // every lane polls; the outcome is made warp-uniform before anyone branches
            bool got = mbar_wait(bar.full(s), (kb / S1) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (got && kb >= S2)
                got = mbar_wait(bar.cfree(b), ((kb / S2) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const float am = am_tile(s)[r];
            const uint32_t am2 = pack_bf16x2(am, am);
            uint8_t* bt = b_tile(b);
#pragma unroll
            for (int part = 0; part < 2 / ROW_SPLIT; ++part) {
                const int w16 = 2 / ROW_SPLIT * h + part;    // 16-byte packed word of the row
                const uint4 q = *reinterpret_cast<const uint4*>(p_tile(s) + r * kPackedRow + 16 * w16);
                st_sw128(bt, r, 4 * w16 + 0, expand8(q.x, lut_lane, am2));
                st_sw128(bt, r, 4 * w16 + 1, expand8(q.y, lut_lane, am2));
                st_sw128(bt, r, 4 * w16 + 2, expand8(q.z, lut_lane, am2));
                st_sw128(bt, r, 4 * w16 + 3, expand8(q.w, lut_lane, am2));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && report_converted(kb)) mbar_arrive(bar.conv(b));
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = ok && mbar_wait(bar.accum(), 0, args.err, abort_flag, kErrTimeoutAccum);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const int cw = warp - 2;
            const int q = warp & 3;              // TMEM lane quarter this warp may access
            const int acc = (cw >> 2) & 1;       // accumulator (M half)
            const int ch = cw >> 3;              // column part of the tile (0 with 8 warps)
            constexpr int COLS = BN / COL_SPLIT;
            const int row = m0 + acc * 128 + q * 32 + lane;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN + ch * COLS;
            const bool vec = (args.N % 8) == 0;
            uint16_t* yrow = args.y + static_cast<int64_t>(row) * args.N;
#pragma unroll 1
            for (int c0 = 0; c0 < COLS; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
                uint32_t hv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) hv[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                const int nc = n0 + ch * COLS + c0;
                if (row < args.M && nc < args.N) {
                    if (vec && nc + 16 <= args.N) {
                        stg_v4(yrow + nc, make_uint4(hv[0], hv[1], hv[2], hv[3]));
                        stg_v4(yrow + nc + 8, make_uint4(hv[4], hv[5], hv[6], hv[7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (nc + i < args.N)
                                yrow[nc + i] = static_cast<uint16_t>(i & 1 ? hv[i >> 1] >> 16 : hv[i >> 1] & 0xffffu);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// ============================================================ skinny kernel

#ifndef NF4_SKINNY_SA
#define NF4_SKINNY_SA 3
#endif

namespace skinny {
constexpr int BN = 128;                      // weight rows per CTA (MMA M)
constexpr int SA = NF4_SKINNY_SA;            // converted-weight buffers
constexpr int A_BYTES = BN * kBK * 2;        // 16 KB
constexpr int P_BYTES = BN * kPackedRow;     // 4 KB
constexpr int AM_BYTES = BN * 4;             // 512 B of fp32 scales
constexpr int CONV_WARPS = 8;                // two threads per weight row
constexpr int THREADS = 64 + CONV_WARPS * 32;
constexpr int TARGET_CTAS = 152;             // one wave on a GB300 (152 SMs)
// shared memory left for the activation + packed + scale ring
constexpr int RING_BUDGET = 232448 - 1024 - SA * A_BYTES - kLutBytes - 2048;
__host__ __device__ constexpr int x_bytes(int mpad) { return mpad * kBK * 2; }
__host__ __device__ constexpr int slot_bytes(int mpad) { return P_BYTES + x_bytes(mpad) + AM_BYTES; }
__host__ __device__ constexpr int stages(int mpad) {
    return RING_BUDGET / slot_bytes(mpad) > 16 ? 16 : RING_BUDGET / slot_bytes(mpad);
}
__host__ __device__ constexpr int tmem_cols(int mpad) { return mpad <= 32 ? 32 : mpad <= 64 ? 64 : 128; }
__host__ __device__ constexpr int off_x() { return SA * A_BYTES; }
__host__ __device__ constexpr int off_p(int mpad) { return off_x() + stages(mpad) * x_bytes(mpad); }
__host__ __device__ constexpr int off_am(int mpad) { return off_p(mpad) + stages(mpad) * P_BYTES; }
__host__ __device__ constexpr int off_lut(int mpad) { return off_am(mpad) + stages(mpad) * AM_BYTES; }
__host__ __device__ constexpr int off_bar(int mpad) { return off_lut(mpad) + kLutBytes; }
__host__ __device__ constexpr size_t smem_bytes(int mpad) {
    return 1024 + off_bar(mpad) + Barriers::count(stages(mpad), SA) * 8 + 16;
}
static_assert(smem_bytes(16) <= 232448 && smem_bytes(128) <= 232448, "shared memory budget");
}  // namespace skinny

// Split-K plan of the skinny path: a pure function of the shape, so the
// workspace size needs no device query.
struct SkinnyPlan {
    int mpad, n_tiles, splits, kb_per_split;
};

inline SkinnyPlan skinny_plan(int64_t M, int64_t N, int64_t K) {
    SkinnyPlan p;
    p.mpad = static_cast<int>(((M + 15) / 16) * 16);
    p.n_tiles = static_cast<int>((N + skinny::BN - 1) / skinny::BN);
    const int nk = static_cast<int>(K / kBK);
    int splits = std::max(1, skinny::TARGET_CTAS / std::max(1, p.n_tiles));
    splits = std::min(splits, nk);
    p.kb_per_split = (nk + splits - 1) / splits;
    p.splits = (nk + p.kb_per_split - 1) / p.kb_per_split;   // no empty split
    return p;
}

struct SkinnyArgs {
    const float* absmax;  // [N, K/64]
    float* ws;            // [splits, M, N] fp32 partial sums
    int M, N, K, kb_per_split;
    uint32_t* err;
};

template <int MPAD>
__global__ void __launch_bounds__(skinny::THREADS, 1)
skinny_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
              const SkinnyArgs args) {
    using namespace skinny;
    constexpr int S1 = stages(MPAD);
    constexpr int XB = x_bytes(MPAD);
    constexpr int TCOLS = tmem_cols(MPAD);
    constexpr int NUM_BARS = Barriers::count(S1, SA);
    static_assert(off_x() % 1024 == 0 && XB % 1024 == 0, "128B-swizzle tiles need 1 KB alignment");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + off_lut(MPAD));
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + off_bar(MPAD));
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Barriers bar{smem_u32(bar_mem), S1, SA};

    auto a_tile = [&](int b) { return smem + b * A_BYTES; };
    auto x_tile = [&](int s) { return smem + off_x() + s * XB; };
    auto p_tile = [&](int s) { return smem + off_p(MPAD) + s * P_BYTES; };
    auto am_tile = [&](int s) { return reinterpret_cast<const float*>(smem + off_am(MPAD) + s * AM_BYTES); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int split = blockIdx.y;
    const int nk_total = args.K / kBK;
    const int kb0 = split * args.kb_per_split;
    const int nk = min(args.kb_per_split, nk_total - kb0);

    if (threadIdx.x == 0) {
        init_barriers(bar, CONV_WARPS);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TCOLS);
        tmem_relinquish();
    }
    if (warp >= 2) build_lut(lut, threadIdx.x - 64, CONV_WARPS * 32);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        int issued = 0;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S1;
            bool ok = true;
            if (kb >= S1)
                ok = mbar_wait(bar.empty(s), ((kb / S1) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            produce_slice<BN>(bar, s, lane, XB + P_BYTES, &tm_x, smem_u32(x_tile(s)), (kb0 + kb) * kBK, 0, &tm_w,
                              smem_u32(p_tile(s)), (kb0 + kb) * kPackedRow, n0, smem_u32(am_tile(s)), args.absmax,
                              args.N, nk_total, kb0 + kb);
            ++issued;
        }
        if (*abort_flag && lane == 0) drain_tma(bar, issued, args.err);
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, MPAD);
            bool ok = true;
            for (int kb = 0; kb < nk && ok; ++kb) {
                const int s = kb % S1;
                const int b = kb % SA;
                ok = mbar_wait(bar.full(s), (kb / S1) & 1, args.err, abort_flag, kErrTimeoutFull) &&
                     mbar_wait(bar.conv(b), (kb / SA) & 1, args.err, abort_flag, kErrTimeoutConverted);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(a_tile(b));
                const uint32_t x0 = smem_u32(x_tile(s));
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j)
                    mma_bf16(tmem, smem_desc_sw128(a0 + 32 * j), smem_desc_sw128(x0 + 32 * j), idesc,
                             (kb > 0 || j > 0) ? 1u : 0u);
                mma_commit(bar.empty(s));
                mma_commit(bar.cfree(b));
            }
            if (ok)
                mma_commit(bar.accum());
            else
                drain_mma(bar, args.err);
        }
    } else {
        // two converter threads per weight row: half h holds K elements [32h, 32h + 32)
        const int r = (warp & 3) * 32 + lane;
        const int h = (warp - 2) >> 2;
        const uint32_t* lut_lane = lut + lane;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % S1;
            const int b = kb % SA;
            bool got = mbar_wait(bar.full(s), (kb / S1) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (got && kb >= SA)
                got = mbar_wait(bar.cfree(b), ((kb / SA) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const float am = am_tile(s)[r];
            const uint32_t am2 = pack_bf16x2(am, am);
            const uint4 q = *reinterpret_cast<const uint4*>(p_tile(s) + r * kPackedRow + 16 * h);
            uint8_t* at = a_tile(b);
            st_sw128(at, r, 4 * h + 0, expand8(q.x, lut_lane, am2));
            st_sw128(at, r, 4 * h + 1, expand8(q.y, lut_lane, am2));
            st_sw128(at, r, 4 * h + 2, expand8(q.z, lut_lane, am2));
            st_sw128(at, r, 4 * h + 3, expand8(q.w, lut_lane, am2));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && report_converted(kb)) mbar_arrive(bar.conv(b));
        }
        ok = ok && mbar_wait(bar.accum(), 0, args.err, abort_flag, kErrTimeoutAccum);
        if (warp < 6 && __all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            // TMEM lane = weight row (n), column = activation row (m)
            const int q = warp & 3;
            const int nn = n0 + q * 32 + lane;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16);
            float* ws = args.ws + static_cast<int64_t>(split) * args.M * args.N;
#pragma unroll 1
            for (int c0 = 0; c0 < MPAD; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
                if (nn < args.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = c0 + i;
                        if (m < args.M) ws[static_cast<int64_t>(m) * args.N + nn] = __uint_as_float(v[i]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
    }
}

// Sum the split-K partials in split order and round once to bf16.
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splits, int64_t mn,
                                     uint16_t* __restrict__ y) {
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < mn;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        float acc = ws[i];
        for (int s = 1; s < splits; ++s) acc += ws[static_cast<int64_t>(s) * mn + i];
        y[i] = __bfloat16_as_ushort(__float2bfloat16_rn(acc));
    }
}

// ============================================================ host side

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    });
    return fn;
}

// 2-D row-major tensor [rows, cols] of `elem` bytes per element, box
// {box_cols, box_rows}, optional 128-byte swizzle; out-of-range reads fill 0.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t rows,
              uint64_t cols, uint32_t box_rows, uint32_t box_cols, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<cuuint64_t>(elem)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Raise a kernel's dynamic shared memory limit, once per (kernel, device).
cudaError_t set_smem(const void* kernel, size_t bytes, int device) {
    static std::mutex mu;
    static const void* done_kernel[256] = {};
    static int done_device[256] = {};
    static int n_done = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < n_done; ++i)
        if (done_kernel[i] == kernel && done_device[i] == device) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e == cudaSuccess && n_done < 256) {
        done_kernel[n_done] = kernel;
        done_device[n_done] = device;
        ++n_done;
    }
    return e;
}

}  // namespace

cudaError_t launch_gemm(const DeviceInfo& dev, const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                        const float* absmax, int64_t N, uint16_t* y, cudaStream_t s) {
    using namespace big;
    if (dev.smem_optin < SMEM) return cudaErrorInvalidConfiguration;
    CUtensorMap tm_x, tm_w;
    if (!make_map(&tm_x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, BM, kBK, true) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, BN, kPackedRow, false))
        return cudaErrorInvalidValue;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(gemm_kernel), SMEM, dev.ordinal); e != cudaSuccess) return e;
    GemmArgs a{absmax, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), dev.err_word};
    const int64_t tiles = ((N + BN - 1) / BN) * ((M + BM - 1) / BM);
    if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
    gemm_kernel<<<static_cast<unsigned>(tiles), THREADS, SMEM, s>>>(tm_x, tm_w, a);
    count_launches(1);
    return cudaGetLastError();
}

size_t skinny_workspace_bytes(const DeviceInfo*, int64_t M, int64_t N, int64_t K) {
    const SkinnyPlan p = skinny_plan(M, N, K);
    return p.splits > 1 ? static_cast<size_t>(p.splits) * M * N * sizeof(float) : size_t(M) * N * sizeof(float);
}

template <int MPAD>
static cudaError_t launch_skinny_t(const DeviceInfo& dev, const SkinnyPlan& p, const CUtensorMap& tm_x,
                                   const CUtensorMap& tm_w, const SkinnyArgs& a, cudaStream_t s) {
    const size_t smem = skinny::smem_bytes(MPAD);
    if (dev.smem_optin < smem) return cudaErrorInvalidConfiguration;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(skinny_kernel<MPAD>), smem, dev.ordinal); e != cudaSuccess) return e;
    dim3 grid(static_cast<unsigned>(p.n_tiles), static_cast<unsigned>(p.splits));
    skinny_kernel<MPAD><<<grid, skinny::THREADS, smem, s>>>(tm_x, tm_w, a);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_skinny(const DeviceInfo& dev, const uint16_t* x, int64_t M, int64_t K, const uint8_t* packed,
                          const float* absmax, int64_t N, uint16_t* y, void* workspace, size_t ws_bytes,
                          cudaStream_t s) {
    const SkinnyPlan p = skinny_plan(M, N, K);
    if (ws_bytes < skinny_workspace_bytes(&dev, M, N, K)) return cudaErrorInvalidValue;
    CUtensorMap tm_x, tm_w;
    if (!make_map(&tm_x, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, M, K, p.mpad, kBK, true) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, skinny::BN, kPackedRow, false))
        return cudaErrorInvalidValue;
    SkinnyArgs a{absmax, static_cast<float*>(workspace), static_cast<int>(M), static_cast<int>(N),
                 static_cast<int>(K), p.kb_per_split, dev.err_word};
    cudaError_t e;
    switch (p.mpad) {
        case 16: e = launch_skinny_t<16>(dev, p, tm_x, tm_w, a, s); break;
        case 32: e = launch_skinny_t<32>(dev, p, tm_x, tm_w, a, s); break;
        case 48: e = launch_skinny_t<48>(dev, p, tm_x, tm_w, a, s); break;
        case 64: e = launch_skinny_t<64>(dev, p, tm_x, tm_w, a, s); break;
        case 80: e = launch_skinny_t<80>(dev, p, tm_x, tm_w, a, s); break;
        case 96: e = launch_skinny_t<96>(dev, p, tm_x, tm_w, a, s); break;
        case 112: e = launch_skinny_t<112>(dev, p, tm_x, tm_w, a, s); break;
        case 128: e = launch_skinny_t<128>(dev, p, tm_x, tm_w, a, s); break;
        default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess) return e;
    const int64_t mn = M * N;
    const int threads = 256;
    const int grid = static_cast<int>(std::min<int64_t>((mn + threads - 1) / threads, 4 * static_cast<int64_t>(dev.sm_count)));
    splitk_reduce_kernel<<<grid, threads, 0, s>>>(static_cast<const float*>(workspace), p.splits, mn, y);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace nf4
