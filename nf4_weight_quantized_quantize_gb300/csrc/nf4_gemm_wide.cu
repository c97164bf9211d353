// nf4_gemm_wide.cu -- the fused NF4 GEMM for larger batches (M > 256):
// Y[M, N] = X[M, K] . deq(W)[N, K]^T at bf16 or fp16, fp32 accumulation in
// TMEM, tcgen05 kind::f16.
//
// This is the forward of the NF4 linear module of the diffuseR page "Gemma3
// NF4 on GPU" (#39, Summary: ltx23_nf4_linear) for the prompt batches of the
// text encoder.  Like the tile kernel (nf4_gemm.cu) it runs swap-AB -- the
// expanded weight tile is operand A (128 weight rows), the activations are
// operand B, the accumulator holds Y^T -- but the expanded weights go to
// shared memory instead of tensor memory.  That frees all 512 TMEM columns
// for two accumulators of up to 256 activation rows each, so every expanded
// 128 x 64 weight slab feeds up to 512 activation rows: half the expansion
// work per FLOP of the tile kernel, whose converter warps, not the tensor
// pipe, set its pace.
//
// Per CTA: a tile of 128 weight rows x 2 NX activation rows over the whole K.
// Three rings:
//   activations: SX slots of one half K-slice (32 values = 64 bytes of each
//     of the 2 NX rows; two TMA boxes of NX rows, 64-byte swizzle), each
//     released by its own MMA commit, so loads run up to SX - 1 half-slices
//     ahead of the tensor core;
//   expanded weights: SA slots of two K-slices, 128 rows x 128 bytes each in
//     the K-major 128-byte-swizzle layout the MMA descriptor reads (16-byte
//     chunk c of row r at chunk c ^ (r % 8)), written by the converter warps
//     with st.shared and released by a commit after the stage's MMAs;
//   packed weights: SP slots of two K-slices of packed bytes and fp32 scales
//     (the tile kernel's weight producer).
// Warps: 0 loads activations (TMA, lane 0); 1 allocates TMEM and its lane 0
// issues the MMAs; 2-17 are converters (one thread per weight row and half
// K-slice: 16 packed bytes expanded through register byte permutes, scaled
// by the block absmax exactly as the dequantizer does), then the epilogue;
// 18 loads the packed weights.  Every wait is bounded (NF4_WAIT_LIMIT_NS);
// on expiry the CTA records an error code, drains what it has in flight,
// frees TMEM and returns.
#include <algorithm>
#include <cmath>

#include <cudaTypedefs.h>

#include "nf4_convert.cuh"
#include "nf4_device.cuh"
#include "nf4_launch.h"

namespace nf4 {

namespace {

constexpr int kWdKs = 2;                               // K-slices per stage
constexpr int kWdRs = 2;                               // converter threads per weight row and K-slice
constexpr int kWdConvWarps = 4 * kWdKs * kWdRs;        // 16
constexpr int kWdWprodWarp = 2 + kWdConvWarps;         // 18
constexpr int kWdThreads = 32 * (kWdWprodWarp + 1);    // 608
constexpr int kWdSmemLimit = 232448;
constexpr int kWdAccStride = 256;                      // TMEM columns between the two accumulators

template <int NX>
struct WdCfg {
    static constexpr int BW = 128;                             // weight rows per tile
    static constexpr int XH = 2 * NX * 64;                     // activation half-slice slot
    static constexpr int A_KS = BW * 128;                      // one expanded K-slice (16 KB)
    static constexpr int A_SLOT = kWdKs * A_KS;
    static constexpr int P_BYTES = BW * kPackedRow * kWdKs;    // packed bytes of a stage
    static constexpr int AM_BYTES = BW * 4 * kWdKs;            // scales of a stage
    static constexpr int P_SLOT = (P_BYTES + AM_BYTES + 1023) / 1024 * 1024;
    static constexpr int SA = 2;
    static constexpr int SP = 3;
    static constexpr int BUDGET = kWdSmemLimit - 1024 - 512;   // alignment slack; barriers and flags
    static constexpr int SX_FIT = (BUDGET - SA * A_SLOT - SP * P_SLOT) / XH;
    static constexpr int SX = SX_FIT > 8 ? 8 : SX_FIT;
    static constexpr int OFF_A = SX * XH;
    static constexpr int OFF_P = OFF_A + SA * A_SLOT;
    static constexpr int OFF_BAR = OFF_P + SP * P_SLOT;
    static constexpr int NBAR = 2 * SX + 2 * SA + 2 * SP + 2;   // + accum, drain
    static constexpr size_t SMEM = 1024 + OFF_BAR + 8 * NBAR + 16;
    static_assert(NX % 16 == 0 && NX >= 16 && NX <= 256, "MMA N");
    static_assert(XH % 1024 == 0, "slot alignment");
    static_assert(SX >= 3, "activation ring depth");
    static_assert(SMEM <= kWdSmemLimit, "shared memory budget");
    // packed tile: rows of 64 bytes loaded with the 64-byte swizzle (16-byte
    // chunk c of row r at c ^ ((r / 2) % 4)), so a warp's reads of one chunk
    // from 32 rows spread over all banks
    __device__ static uint32_t packed_offset(int row, int chunk) {
        const uint32_t o = static_cast<uint32_t>(row * kPackedRow * kWdKs + 16 * chunk);
        return o ^ (((o >> 7) & 3u) << 4);
    }
};

struct WdArgs {
    const float* absmax;   // [N, K / 64]
    void* y;               // [M, N]
    int M, N, K;
    int m_tiles;
    uint32_t* err;
};

// Shared-memory descriptor of a K-major operand in the 64-byte swizzle: rows
// of 64 bytes, 8-row groups 512 bytes apart (fields as for the 128-byte
// form: start >> 4, leading offset 1 (unused), stride 512 >> 4, the fixed
// 0b001 at bits 46-48, swizzle mode 4 = 64 bytes at bits 61-63).
__device__ __forceinline__ uint64_t smem_desc_sw64(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
    d |= static_cast<uint64_t>(1u) << 16;
    d |= static_cast<uint64_t>(512u >> 4) << 32;
    d |= static_cast<uint64_t>(1u) << 46;
    d |= static_cast<uint64_t>(4u) << 61;
    return d;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

template <int NX, int DT>
__global__ void __launch_bounds__(kWdThreads, 1)
wide_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, const WdArgs args) {
    using C = WdCfg<NX>;
    static_assert(DT == kBF16 || DT == kF16, "kind::f16 operand types");
    constexpr int SX = C::SX, SA = C::SA, SP = C::SP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1 KB aligned
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + C::NBAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const uint32_t b0 = smem_u32(bar_mem);
    auto xfull = [&](int i) { return b0 + 8u * i; };
    auto xempty = [&](int i) { return b0 + 8u * (SX + i); };
    auto afull = [&](int i) { return b0 + 8u * (2 * SX + i); };
    auto aempty = [&](int i) { return b0 + 8u * (2 * SX + SA + i); };
    auto pfull = [&](int i) { return b0 + 8u * (2 * SX + 2 * SA + i); };
    auto pempty = [&](int i) { return b0 + 8u * (2 * SX + 2 * SA + SP + i); };
    const uint32_t accum = b0 + 8u * (2 * SX + 2 * SA + 2 * SP);
    const uint32_t drain = accum + 8u;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles run m-fastest: CTAs resident together share each weight tile through L2
    const int m0 = static_cast<int>(blockIdx.x % args.m_tiles) * (2 * NX);
    const int n0 = static_cast<int>(blockIdx.x / args.m_tiles) * C::BW;
    const int nk = args.K / kBK;
    const int nst = (nk + kWdKs - 1) / kWdKs;
    const int nhalf = 2 * nk;   // activation half-slices

    if (threadIdx.x == 0) {
        for (int i = 0; i < SX; ++i) {
            mbar_init(xfull(i), 1);
            mbar_init(xempty(i), 1);
        }
        for (int i = 0; i < SA; ++i) {
            mbar_init(afull(i), kWdConvWarps);
            mbar_init(aempty(i), 1);
        }
        for (int i = 0; i < SP; ++i) {
            mbar_init(pfull(i), kPfullArrivals);
            mbar_init(pempty(i), kWdConvWarps);
        }
        mbar_init(accum, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the previous kernel on the stream has finished
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------- activation producer: half-slice q into slot q % SX
        // once the MMAs that read its previous contents completed
        if (lane == 0) {
            int issued = 0;
            for (int q = 0; q < nhalf; ++q) {
                const int x = q % SX;
                if (q >= SX &&
                    !mbar_wait(xempty(x), ((q / SX) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty))
                    break;
                if (*abort_flag) break;
                const uint32_t dst = smem_u32(smem + x * C::XH);
                mbar_arrive_expect_tx(xfull(x), C::XH);
                tma_load_2d(dst, &tm_x, xfull(x), q * 32, m0);
                tma_load_2d(dst + NX * 64, &tm_x, xfull(x), q * 32, m0 + NX);
                ++issued;
            }
            if (*abort_flag) drain_ring(xfull(0), SX, issued, args.err);
        }
    } else if (warp == kWdWprodWarp) {
        // ---------------- weight producer: stage st's packed bytes and scales
        // into slot st % SP once every converter warp has read it
        int issued = 0;
        for (int st = 0; st < nst; ++st) {
            const int p = st % SP;
            bool ok = true;
            if (st >= SP) ok = mbar_wait(pempty(p), ((st / SP) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            const int kb = st * kWdKs;
            uint8_t* ptile = smem + C::OFF_P + p * C::P_SLOT;
            produce_weights<C::BW, kWdKs, false>(pfull(p), lane, C::P_BYTES, &tm_w, smem_u32(ptile),
                                                 kb * kPackedRow, n0, 0, args.N, smem_u32(ptile + C::P_BYTES),
                                                 args.absmax, nk, kb);
            ++issued;
        }
        if (*abort_flag && lane == 0) drain_ring(pfull(0), SP, issued, args.err);
    } else if (warp == 1) {
        // ---------------- MMA issuer: per stage, wait for the expanded weights;
        // per activation half-slice, wait for it, 2 k-steps x 2 accumulators,
        // one commit that releases the half-slice; one commit per stage that
        // releases the weight slot
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16kind_f32<DT>(128, NX);
            const uint32_t a_base = smem_u32(smem + C::OFF_A);
            const uint32_t x_base = smem_u32(smem);
            bool ok = true;
            for (int st = 0; st < nst && ok; ++st) {
                const int a = st % SA;
                ok = mbar_wait(afull(a), (st / SA) & 1, args.err, abort_flag, kErrTimeoutConverted);
                if (!ok) break;
                const int kbs = min(kWdKs, nk - st * kWdKs);
                for (int h = 0; h < kbs && ok; ++h) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int q = 2 * (st * kWdKs + h) + half;
                        const int x = q % SX;
                        ok = mbar_wait(xfull(x), (q / SX) & 1, args.err, abort_flag, kErrTimeoutFull);
                        if (!ok) break;
                        tc_fence_after();
#pragma unroll
                        for (int j = 0; j < 2; ++j) {
                            // k-step 2 half + j of the K-slice: 32 bytes of each row
                            const uint64_t adesc =
                                smem_desc_sw128(a_base + a * C::A_SLOT + h * C::A_KS + 32 * (2 * half + j));
#pragma unroll
                            for (int acc = 0; acc < 2; ++acc) {
                                const uint64_t bdesc = smem_desc_sw64(x_base + x * C::XH + acc * NX * 64 + 32 * j);
                                const uint32_t first = (st == 0 && h == 0 && half == 0 && j == 0) ? 0u : 1u;
                                mma_bf16(tmem + acc * kWdAccStride, adesc, bdesc, idesc, first);
                            }
                        }
                        mma_commit(xempty(x));
                    }
                }
                if (ok) mma_commit(aempty(a));
            }
            if (ok) {
                mma_commit(accum);
            } else {
                int dummy = 0;
                mma_commit(drain);
                mbar_wait(drain, 0, args.err, &dummy, kErrTimeoutDrain);
            }
        }
    } else {
        // ---------------- converters: unit u = (warp - 2) / 4 expands half
        // `part` of K-slice h of each stage for weight rows 32 q .. 32 q + 31
        // (q = warp % 4, the TMEM lane quarter this warp reads in the epilogue)
        const int u = (warp - 2) >> 2;
        const int h = u % kWdKs;
        const int part = u / kWdKs;
        const int q = warp & 3;
        const int r = q * 32 + lane;   // weight row within the tile
        const CodebookRegs cb = codebook_regs<DT>();
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        bool ok = true;
        for (int st = 0; st < nst; ++st) {
            const int p = st % SP;
            const int a = st % SA;
            const bool got = mbar_wait(pfull(p), (st / SP) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint8_t* ptile = smem + C::OFF_P + p * C::P_SLOT;
            const bool live = st * kWdKs + h < nk;   // warp-uniform: the K-slice exists
            uint4 w4 = make_uint4(0, 0, 0, 0);
            float am = 0.0f;
            if (live) {
                am = reinterpret_cast<const float*>(ptile + C::P_BYTES)[h * C::BW + r];
                w4 = *reinterpret_cast<const uint4*>(ptile + C::packed_offset(r, 2 * h + part));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty(p));   // this warp is done with packed slot p
            // the expanded slot must be free: the MMAs of stage st - SA completed
            const bool free_slot = st < SA || mbar_wait(aempty(a), ((st / SA) - 1) & 1, args.err, abort_flag,
                                                        kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, free_slot)) {
                ok = false;
                break;
            }
            if (live) {
                // An absmax that is a DT value scales in one paired DT multiply
                // (exact product, one rounding); any other absmax scales each
                // value in fp32 and rounds once -- the dequantizer's value.
                const bool exact = exact_in<DT>(am);
                const uint32_t am2 = exact ? pack2<DT>(am, am) : pack2<DT>(1.0f, 1.0f);
                uint32_t v[16];
                expand8<DT>(w4.x, cb, am2, v + 0);
                expand8<DT>(w4.y, cb, am2, v + 4);
                expand8<DT>(w4.z, cb, am2, v + 8);
                expand8<DT>(w4.w, cb, am2, v + 12);
                if (!exact) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) v[i] = scale_entry<DT>(v[i], am);
                }
                // 32 values = 4 chunks of 16 bytes: chunks 4 part .. 4 part + 3 of
                // row r, each stored at chunk ^ (r % 8)
                const uint32_t row = a_base + a * C::A_SLOT + h * C::A_KS + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sts128(row + (((4 * part + c) ^ (r & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                           v[4 * c + 3]);
            }
            fence_proxy_async_smem();   // the MMAs read the slot through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(afull(a));
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = __all_sync(0xffffffffu, ok) && mbar_wait(accum, 0, args.err, abort_flag, kErrTimeoutAccum);
        if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            // accumulator acc: TMEM lane = weight row n0 + r, column c = activation
            // row m0 + acc NX + c; 16-column chunks round-robin over the 4 units
            const int n = n0 + r;
            const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
            constexpr int CHUNKS = NX / 16;
#pragma unroll 1
            for (int ci = u; ci < 2 * CHUNKS; ci += 4) {
                const int acc = ci / CHUNKS;
                const int c0 = 16 * (ci % CHUNKS);
                uint32_t v[16];
                tmem_ld16(lane_addr + acc * kWdAccStride + c0, v);
                tmem_ld_wait();
                if (n < args.N) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int m = m0 + acc * NX + c0 + i;
                        if (m < args.M) store_out<DT>(args.y, static_cast<int64_t>(m) * args.N + n, __uint_as_float(v[i]));
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ============================================================ host side

struct WdPlan {
    int nx;        // activation rows per accumulator (MMA N)
    int m_tiles;   // tiles of 2 nx activation rows
    int n_tiles;   // tiles of 128 weight rows
};

WdPlan make_wd_plan(int64_t M, int64_t N) {
    WdPlan p;
    p.m_tiles = static_cast<int>((M + 511) / 512);
    const int64_t rows = (M + p.m_tiles - 1) / p.m_tiles;   // balanced tiles of at most 512 rows
    p.nx = static_cast<int>(((rows + 1) / 2 + 15) / 16 * 16);
    p.n_tiles = static_cast<int>((N + 127) / 128);
    return p;
}

template <int NX, int DT>
cudaError_t launch_wd(const DeviceInfo& dev, const WdPlan& p, const void* x, int64_t M, int64_t K,
                      const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    using C = WdCfg<NX>;
    if (dev.smem_optin < C::SMEM) return cudaErrorInvalidConfiguration;
    auto kernel = wide_kernel<NX, DT>;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(kernel), C::SMEM, dev.ordinal); e != cudaSuccess)
        return e;
    CUtensorMap tm_x, tm_w;
    const CUtensorMapDataType xdt = DT == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    // activations: boxes of 32 values (64 bytes, the swizzle span) x NX rows;
    // packed weights: boxes of two K-slices (64 bytes) x 128 rows
    if (!make_map(&tm_x, x, xdt, 2, M, K, NX, 32, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, C::BW, kPackedRow * kWdKs,
                  CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (tiles > 0x7fffffff) return cudaErrorInvalidConfiguration;
    WdArgs a{absmax, y, static_cast<int>(M), static_cast<int>(N), static_cast<int>(K), p.m_tiles, dev.err_word};
    if (cudaError_t e = launch_pdl(kernel, dim3(static_cast<unsigned>(tiles)), dim3(kWdThreads), C::SMEM, s, tm_x,
                                   tm_w, a);
        e != cudaSuccess)
        return e;
    count_launches(1);
    return cudaGetLastError();
}

template <int DT>
cudaError_t dispatch_wd(const DeviceInfo& dev, const WdPlan& p, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    switch (p.nx) {
        case 144: return launch_wd<144, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 160: return launch_wd<160, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 176: return launch_wd<176, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 192: return launch_wd<192, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 208: return launch_wd<208, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 224: return launch_wd<224, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 240: return launch_wd<240, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 256: return launch_wd<256, DT>(dev, p, x, M, K, packed, absmax, N, y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// Whether the wide kernel takes this call, by the same shape-only estimate
// of both kernels' time: waves of one CTA per SM times the time per K-slice
// of a tile -- about 750 clocks for the tile kernel (128 x 256, bound by its
// converter warps) and 8 MMAs of N = nx for the wide one (about 127 clocks
// per N = 256 MMA; 128 x 2 nx, the same expansion work).
bool wide_applies(int dtype, int64_t M, int64_t N) {
    if ((dtype != kBF16 && dtype != kF16) || M <= 256) return false;
    const WdPlan p = make_wd_plan(M, N);
    if (p.nx < 144 || p.nx > 256) return false;
    constexpr double kSms = 152.0;
    const double n_tiles = static_cast<double>(p.n_tiles);
    const double ts_waves = std::ceil(n_tiles * std::ceil(M / 256.0) / kSms);
    const double wd_waves = std::ceil(n_tiles * p.m_tiles / kSms);
    const double wd_slice = std::max(750.0, 8.0 * 127.0 * p.nx / 256.0);
    return wd_waves * wd_slice < ts_waves * 750.0;
}

cudaError_t launch_gemm_wide(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                             const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    const WdPlan p = make_wd_plan(M, N);
    switch (dtype) {
        case kBF16: return dispatch_wd<kBF16>(dev, p, x, M, K, packed, absmax, N, y, s);
        case kF16: return dispatch_wd<kF16>(dev, p, x, M, K, packed, absmax, N, y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf4
