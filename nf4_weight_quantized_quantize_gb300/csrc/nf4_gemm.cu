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

struct Barriers {
    // layout in shared memory: full[S], conv[S], empty[S], accum, drain
    uint32_t base;
    int stages;
    __device__ uint32_t full(int s) const { return base + 8u * s; }
    __device__ uint32_t conv(int s) const { return base + 8u * (stages + s); }
    __device__ uint32_t empty(int s) const { return base + 8u * (2 * stages + s); }
    __device__ uint32_t accum() const { return base + 8u * (3 * stages); }
    __device__ uint32_t drain() const { return base + 8u * (3 * stages + 1); }
};

// Convert one weight row of one stage: 32 packed bytes (64 elements) at
// `prow` to 64 bf16 at `brow` in the 128-byte swizzle (16-byte chunk c of row
// r stored at chunk position c ^ (r & 7)).  Chunk c holds packed word c.
__device__ __forceinline__ void convert_row(const uint8_t* prow, uint8_t* brow, int r,
                                            const uint32_t* lut, float am) {
    const uint4 q0 = *reinterpret_cast<const uint4*>(prow);
    const uint4 q1 = *reinterpret_cast<const uint4*>(prow + 16);
    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t p = words[c];
        uint4 o;
        o.x = scale_entry(lut[p & 0xffu], am);
        o.y = scale_entry(lut[(p >> 8) & 0xffu], am);
        o.z = scale_entry(lut[(p >> 16) & 0xffu], am);
        o.w = scale_entry(lut[p >> 24], am);
        *reinterpret_cast<uint4*>(brow + ((c ^ (r & 7)) << 4)) = o;
    }
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

// Wait (bounded) for the copies a producer issued into the last `stages`
// K-slices to land, so no TMA write targets shared memory after exit.
__device__ __forceinline__ void drain_tma(const Barriers& bar, int issued, int stages,
                                          uint32_t* err, volatile int* abort_flag) {
    int dummy = 0;
    for (int kb = max(0, issued - stages); kb < issued; ++kb) {
        const int s = kb % stages;
        // a fresh local flag: the CTA-wide abort is already raised here
        if (!mbar_wait(bar.full(s), (kb / stages) & 1, err, &dummy, kErrTimeoutDrain)) break;
    }
    (void)abort_flag;
}

// ============================================================ large-M kernel

namespace big {
constexpr int BM = 256;
constexpr int BN = 256;
constexpr int STAGES = 3;
constexpr int A_BYTES = BM * kBK * 2;        // 32 KB
constexpr int B_BYTES = BN * kBK * 2;        // 32 KB
constexpr int P_BYTES = BN * kPackedRow;     // 8 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES + P_BYTES;
constexpr int CONV_WARPS = BN / 32;          // one converter thread per weight row
constexpr int THREADS = 64 + CONV_WARPS * 32;
constexpr int TMEM_COLS = 512;               // two 128 x 256 fp32 accumulators
constexpr size_t SMEM = 1024 + size_t(STAGES) * STAGE_BYTES + 1024 + 256;
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(CONV_WARPS == 8, "epilogue maps 8 warps onto 2 accumulators x 4 lane quarters");
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
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + STAGES * STAGE_BYTES);
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(lut + 256);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + 3 * STAGES + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Barriers bar{smem_u32(bar_mem), STAGES};

    auto a_tile = [&](int s) { return smem + s * STAGE_BYTES; };
    auto b_tile = [&](int s) { return smem + s * STAGE_BYTES + A_BYTES; };
    auto p_tile = [&](int s) { return smem + s * STAGE_BYTES + A_BYTES + B_BYTES; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles run m-fastest: CTAs resident together share weight tiles through L2
    const int m_tiles = (args.M + BM - 1) / BM;
    const int m0 = static_cast<int>(blockIdx.x % m_tiles) * BM;
    const int n0 = static_cast<int>(blockIdx.x / m_tiles) * BN;
    const int nk = args.K / kBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar.full(s), 1);
            mbar_init(bar.conv(s), CONV_WARPS);
            mbar_init(bar.empty(s), 1);
        }
        mbar_init(bar.accum(), 1);
        mbar_init(bar.drain(), 1);
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
    if (warp >= 2) {
        for (int e = threadIdx.x - 64; e < 256; e += CONV_WARPS * 32) lut[e] = lut_entry(e);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(bar.empty(s), ((kb / STAGES) - 1) & 1, args.err, abort_flag,
                                               kErrTimeoutEmpty))
                    break;
                if (*abort_flag) break;
                mbar_arrive_expect_tx(bar.full(s), A_BYTES + P_BYTES);
                tma_load_2d(smem_u32(a_tile(s)), &tm_x, bar.full(s), kb * kBK, m0);
                tma_load_2d(smem_u32(p_tile(s)), &tm_w, bar.full(s), kb * kPackedRow, n0);
                ++issued;
            }
            if (*abort_flag) drain_tma(bar, issued, STAGES, args.err, abort_flag);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, BN);
            bool ok = true;
            for (int kb = 0; kb < nk && ok; ++kb) {
                const int s = kb % STAGES;
                const uint32_t par = (kb / STAGES) & 1;
                ok = mbar_wait(bar.full(s), par, args.err, abort_flag, kErrTimeoutFull) &&
                     mbar_wait(bar.conv(s), par, args.err, abort_flag, kErrTimeoutConverted);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(a_tile(s));
                const uint32_t b0 = smem_u32(b_tile(s));
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j) {
                    const uint64_t bd = smem_desc_sw128(b0 + 32 * j);
                    const uint32_t acc = (kb > 0 || j > 0) ? 1u : 0u;
                    mma_bf16(tmem, smem_desc_sw128(a0 + 32 * j), bd, idesc, acc);
                    mma_bf16(tmem + BN, smem_desc_sw128(a0 + 128 * 128 + 32 * j), bd, idesc, acc);
                }
                mma_commit(bar.empty(s));
            }
            if (ok) {
                mma_commit(bar.accum());
            } else {
                int dummy = 0;
                mma_commit(bar.drain());
                mbar_wait(bar.drain(), 0, args.err, &dummy, kErrTimeoutDrain);
            }
        }
    } else {
        // ---------------- converters, then epilogue
        const int r = threadIdx.x - 64;          // weight row within the tile
        const int n = n0 + r;
        const bool valid = n < args.N;
        const float* am_row = args.absmax + static_cast<int64_t>(valid ? n : 0) * nk;
        float am0 = valid ? ldg_nc_f32(am_row) : 0.0f;
        float am1 = (valid && nk > 1) ? ldg_nc_f32(am_row + 1) : 0.0f;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % STAGES;
            const float am = am0;
            am0 = am1;
            am1 = (valid && kb + 2 < nk) ? ldg_nc_f32(am_row + kb + 2) : 0.0f;
            // every lane polls; the outcome is made warp-uniform before anyone branches
            const bool got = mbar_wait(bar.full(s), (kb / STAGES) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            convert_row(p_tile(s) + r * kPackedRow, b_tile(s) + r * 128, r, lut, am);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && report_converted(kb)) mbar_arrive(bar.conv(s));
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = ok && mbar_wait(bar.accum(), 0, args.err, abort_flag, kErrTimeoutAccum);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const int q = warp & 3;              // TMEM lane quarter this warp may access
            const int acc = (warp - 2) >> 2;     // accumulator (M half)
            const int row = m0 + acc * 128 + q * 32 + lane;
            const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
            const bool vec = (args.N % 8) == 0;
            uint16_t* yrow = args.y + static_cast<int64_t>(row) * args.N;
#pragma unroll 1
            for (int c0 = 0; c0 < BN; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(taddr + c0, v);
                tmem_ld_wait();
                uint32_t h[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) h[i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                const int nc = n0 + c0;
                if (row < args.M && nc < args.N) {
                    if (vec && nc + 16 <= args.N) {
                        stg_v4(yrow + nc, make_uint4(h[0], h[1], h[2], h[3]));
                        stg_v4(yrow + nc + 8, make_uint4(h[4], h[5], h[6], h[7]));
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if (nc + i < args.N)
                                yrow[nc + i] = static_cast<uint16_t>(i & 1 ? h[i >> 1] >> 16 : h[i >> 1] & 0xffffu);
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

namespace skinny {
constexpr int BN = 128;                      // weight rows per CTA (MMA M)
constexpr int STAGES = 6;
constexpr int A_BYTES = BN * kBK * 2;        // converted weight, 16 KB
constexpr int P_BYTES = BN * kPackedRow;     // 4 KB
constexpr int CONV_WARPS = BN / 32;          // 4
constexpr int THREADS = 64 + CONV_WARPS * 32;
constexpr int TARGET_CTAS = 152;             // one wave on a GB300 (152 SMs)
__host__ __device__ constexpr int x_bytes(int mpad) { return mpad * kBK * 2; }
__host__ __device__ constexpr int stage_bytes(int mpad) { return A_BYTES + P_BYTES + x_bytes(mpad); }
__host__ __device__ constexpr int tmem_cols(int mpad) { return mpad <= 32 ? 32 : mpad <= 64 ? 64 : 128; }
inline size_t smem_bytes(int mpad) { return 1024 + size_t(STAGES) * stage_bytes(mpad) + 1024 + 256; }
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
    constexpr int XB = x_bytes(MPAD);
    constexpr int SB = stage_bytes(MPAD);
    constexpr int TCOLS = tmem_cols(MPAD);
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + STAGES * SB);
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(lut + 256);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + 3 * STAGES + 2);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Barriers bar{smem_u32(bar_mem), STAGES};

    // stage layout: converted weight (1024-aligned), activations (1024-aligned), packed
    auto a_tile = [&](int s) { return smem + s * SB; };
    auto x_tile = [&](int s) { return smem + s * SB + A_BYTES; };
    auto p_tile = [&](int s) { return smem + s * SB + A_BYTES + XB; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int n0 = blockIdx.x * BN;
    const int split = blockIdx.y;
    const int nk_total = args.K / kBK;
    const int kb0 = split * args.kb_per_split;
    const int nk = min(args.kb_per_split, nk_total - kb0);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar.full(s), 1);
            mbar_init(bar.conv(s), CONV_WARPS);
            mbar_init(bar.empty(s), 1);
        }
        mbar_init(bar.accum(), 1);
        mbar_init(bar.drain(), 1);
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
    if (warp >= 2) {
        for (int e = threadIdx.x - 64; e < 256; e += CONV_WARPS * 32) lut[e] = lut_entry(e);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int issued = 0;
            for (int kb = 0; kb < nk; ++kb) {
                const int s = kb % STAGES;
                if (kb >= STAGES && !mbar_wait(bar.empty(s), ((kb / STAGES) - 1) & 1, args.err, abort_flag,
                                               kErrTimeoutEmpty))
                    break;
                if (*abort_flag) break;
                mbar_arrive_expect_tx(bar.full(s), XB + P_BYTES);
                tma_load_2d(smem_u32(x_tile(s)), &tm_x, bar.full(s), (kb0 + kb) * kBK, 0);
                tma_load_2d(smem_u32(p_tile(s)), &tm_w, bar.full(s), (kb0 + kb) * kPackedRow, n0);
                ++issued;
            }
            if (*abort_flag) drain_tma(bar, issued, STAGES, args.err, abort_flag);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(128, MPAD);
            bool ok = true;
            for (int kb = 0; kb < nk && ok; ++kb) {
                const int s = kb % STAGES;
                const uint32_t par = (kb / STAGES) & 1;
                ok = mbar_wait(bar.full(s), par, args.err, abort_flag, kErrTimeoutFull) &&
                     mbar_wait(bar.conv(s), par, args.err, abort_flag, kErrTimeoutConverted);
                if (!ok) break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(a_tile(s));
                const uint32_t x0 = smem_u32(x_tile(s));
#pragma unroll
                for (int j = 0; j < kBK / 16; ++j)
                    mma_bf16(tmem, smem_desc_sw128(a0 + 32 * j), smem_desc_sw128(x0 + 32 * j), idesc,
                             (kb > 0 || j > 0) ? 1u : 0u);
                mma_commit(bar.empty(s));
            }
            if (ok) {
                mma_commit(bar.accum());
            } else {
                int dummy = 0;
                mma_commit(bar.drain());
                mbar_wait(bar.drain(), 0, args.err, &dummy, kErrTimeoutDrain);
            }
        }
    } else {
        const int r = threadIdx.x - 64;
        const int n = n0 + r;
        const bool valid = n < args.N;
        const float* am_row = args.absmax + static_cast<int64_t>(valid ? n : 0) * nk_total + kb0;
        float am0 = valid ? ldg_nc_f32(am_row) : 0.0f;
        float am1 = (valid && nk > 1) ? ldg_nc_f32(am_row + 1) : 0.0f;
        bool ok = true;
        for (int kb = 0; kb < nk; ++kb) {
            const int s = kb % STAGES;
            const float am = am0;
            am0 = am1;
            am1 = (valid && kb + 2 < nk) ? ldg_nc_f32(am_row + kb + 2) : 0.0f;
            // every lane polls; the outcome is made warp-uniform before anyone branches
            const bool got = mbar_wait(bar.full(s), (kb / STAGES) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            convert_row(p_tile(s) + r * kPackedRow, a_tile(s) + r * 128, r, lut, am);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && report_converted(kb)) mbar_arrive(bar.conv(s));
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = ok && mbar_wait(bar.accum(), 0, args.err, abort_flag, kErrTimeoutAccum);
        if (__all_sync(0xffffffffu, ok)) {
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
