// nf4_gemm_wide.cu -- the fused NF4 GEMM for larger batches on CTA pairs:
// Y[M, N] = X[M, K] . deq(W)[N, K]^T at bf16, fp16 or fp32, fp32 accumulation
// in TMEM, tcgen05 kind::f16 (kind::tf32 for fp32) with cta_group::2 (one MMA
// spans the tensor cores of the two SMs of a CTA pair).
//
// This is the forward of the NF4 linear module of the diffuseR page "Gemma3
// NF4 on GPU" (#39, Summary: ltx23_nf4_linear) for the prompt batches of the
// text encoder.  Like the tile kernel (nf4_gemm.cu) it runs swap-AB -- the
// expanded weights are operand A, the activations operand B, the accumulator
// holds Y^T -- with two differences:
//   - the expanded weights go to shared memory (the K-major 128-byte-swizzle
//     layout the MMA descriptor reads), so all 512 TMEM columns hold two
//     accumulators of NX (<= 256) activation rows: every expanded 128 x 64
//     weight slab feeds 2 NX activation rows, half the expansion work per FLOP
//     of the tile kernel, whose converter warps set its pace;
//   - a pair of CTAs shares each MMA (M = 256): each CTA expands its own 128
//     weight rows and loads only its half of each accumulator's activation
//     rows, and each SM's tensor core reads the other half from the peer CTA's
//     shared memory.  A K-slice then costs each CTA 32 KB of activations
//     instead of 64, and its 4-slot activation ring spans 4 K-slices (a single
//     CTA this wide cannot hide the activation tiles' load latency within its
//     shared memory: its MMA issuer waited on them about a quarter of the time).
// The pair's tile is 256 weight rows x 2 NX activation rows over the whole K.
// A gate/up pair (GEGLU) takes 64 gate rows and the 64 up rows of the same
// outputs per CTA and writes gelu_tanh(gate) * up.
//
// Rings (per CTA): activations, SX slots of one ring slice (NX rows x 128
// bytes: the CTA's halves of both accumulators, TMA with the 128-byte
// swizzle); expanded weights, SA slots of one ring slice written by the
// converters; packed weights, SP slots of two K-slices of packed bytes and
// fp32 scales.  A ring slice is one K-slice (NF4 block) of a 16-bit type and
// half of one of fp32 -- 128 bytes of each row either way.
// Warps: 0 loads activations (both CTAs' copies complete on the even CTA's
// barrier); 1 allocates TMEM (both CTAs) and in the even CTA issues the first
// accumulator's MMAs; 2-17 are converters (both CTAs' arrive on the even
// CTA's barrier), then the epilogue; 18 loads packed weights; 19 (even CTA)
// issues the second accumulator's MMAs.  MMA completion is
// committed to the barriers of both CTAs.  Every wait is bounded
// (NF4_WAIT_LIMIT_NS); on expiry the CTA records an error code, drains what it
// has in flight and frees TMEM, and the peer's waits on it expire in turn.
// The odd CTA cannot observe its activation copies (they complete on the even
// CTA's barrier), so on that path it waits a fixed 1 ms -- orders of magnitude
// above a copy's latency -- before the pair's closing cluster barrier.
#include <algorithm>
#include <cmath>

#include <cudaTypedefs.h>

#include "nf4_convert.cuh"
#include "nf4_device.cuh"
#include "nf4_launch.h"

namespace nf4 {

namespace {

constexpr int kWdKs = 2;                               // K-slices per stage
constexpr int kWdConvWarps = 16;                       // 4 lane quarters x 2 K-slices x 2 halves
constexpr int kWdWprodWarp = 2 + kWdConvWarps;         // 18
constexpr int kWdIssuer1Warp = kWdWprodWarp + 1;       // 19: the second accumulator's MMA issuer
constexpr int kWdThreads = 32 * (kWdIssuer1Warp + 1);  // 640
constexpr int kWdIssuers = 2;                          // one MMA issuer thread per accumulator
constexpr uint64_t kWdSettleNs = 1000000;              // error path: time for copies in flight to land
constexpr int kWdSmemLimit = 232448;
constexpr int kWdAccStride = 256;                      // TMEM columns between the two accumulators

template <int NX>
struct WdCfg {
    static constexpr int BW = 128;                             // weight rows per CTA
    static constexpr int XS = NX * 128;                        // activation slot: NX rows (2 halves of NX / 2)
    static constexpr int A_KS = BW * 128;                      // one expanded ring slice (16 KB)
    static constexpr int P_BYTES = BW * kPackedRow * kWdKs;    // packed bytes of a stage
    static constexpr int AM_BYTES = BW * 4 * kWdKs;            // scales of a stage
    static constexpr int P_SLOT = (P_BYTES + AM_BYTES + 1023) / 1024 * 1024;
    static constexpr int SA = 4;                               // expanded-weight slots, one ring slice each
    static constexpr int SP = 3;
    static constexpr int BUDGET = kWdSmemLimit - 1024 - 512;   // alignment slack; barriers and flags
    static constexpr int SX_FIT = (BUDGET - SA * A_KS - SP * P_SLOT) / XS;
    static constexpr int SX = SX_FIT > 8 ? 8 : SX_FIT;
    static constexpr int OFF_A = SX * XS;
    static constexpr int OFF_P = OFF_A + SA * A_KS;
    static constexpr int OFF_BAR = OFF_P + SP * P_SLOT;
    // xfull, xempty (SX each); afull, aempty (SA each); pfull, pempty (SP
    // each); accum, drain
    static constexpr int NBAR = 2 * SX + 2 * SA + 2 * SP + 2;
    static constexpr size_t SMEM = 1024 + OFF_BAR + 8 * NBAR + 16;
    static_assert(NX % 32 == 0 && NX >= 32 && NX <= 256, "MMA N, two halves of a multiple of 16");
    static_assert(XS % 1024 == 0, "slot alignment");
    static_assert(SX >= 3, "activation ring depth");
    static_assert(SMEM <= kWdSmemLimit, "shared memory budget");
    // a gate/up pair's epilogue parks half of each CTA's accumulator columns,
    // [2 NX columns][64 pair rows] fp32, in the activation ring
    static_assert(SX * XS >= 2 * NX * (BW / 2) * 4, "gate/up exchange buffer");
    // packed tile: rows of 64 bytes loaded with the 64-byte swizzle (16-byte
    // chunk c of row r at c ^ ((r / 2) % 4)), so a warp's reads of one chunk
    // from 32 rows spread over all banks
    __device__ static uint32_t packed_offset(int row, int chunk) {
        const uint32_t o = static_cast<uint32_t>(row * kPackedRow * kWdKs + 16 * chunk);
        return o ^ (((o >> 7) & 3u) << 4);
    }
};

struct WdArgs {
    const float* absmax;   // [N, K / 64] ([2F, K / 64] for a gate/up pair)
    void* y;               // [M, N] ([M, F] for a gate/up pair)
    int M, N, K;           // N: output columns (F for a gate/up pair)
    int m_tiles;
    int64_t am_count;      // scales in absmax
    uint32_t* err;
};

__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of both CTAs of the cluster.
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Arrive (release, CTA scope) on the barrier at the same shared-memory offset
// in CTA `rank` of the cluster.
__device__ __forceinline__ void mbar_arrive_remote_cta(uint32_t local_bar, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_bar), "r"(rank));
    asm volatile("mbarrier.arrive.release.cta.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

// 2D TMA load into this CTA's shared memory whose completion (complete_tx)
// is signalled on the barrier at offset `bar` of the even CTA of the pair: the
// CTA-pair form of the copy, which may signal a barrier of the peer CTA.
__device__ __forceinline__ void tma_load_2d_pair_leader(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                                        int32_t x, int32_t y) {
    uint32_t leader_bar;
    asm volatile("mapa.shared::cluster.u32 %0, %1, 0;" : "=r"(leader_bar) : "r"(bar));
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(map), "r"(x), "r"(y), "r"(leader_bar)
        : "memory");
}

__device__ __forceinline__ void spin_ns(uint64_t ns) {
    const uint64_t t0 = globaltimer();
#pragma unroll 1
    while (globaltimer() - t0 < ns) {
    }
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait for a barrier the peer CTA arrives on (acquire at cluster scope).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity, uint32_t* err, volatile int* abort,
                                                  uint32_t code) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
        if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
#pragma unroll 1
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer() - t0 > NF4_WAIT_LIMIT_NS) {
            record_error(err, code);
            *abort = 1;
            return false;
        }
    }
}

// ---- tcgen05 in CTA-pair form (a kernel uses one form throughout)

__device__ __forceinline__ void tmem_alloc_pair(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D (+)= A . B^T over the pair: A's rows split between the two CTAs (128
// each, at the same shared-memory offset), B's columns likewise, D of each
// SM in its own TMEM at the same address.  kind::f16 for bf16 / fp16
// operands, kind::tf32 for fp32 ones (read as tf32).
template <int DT>
__device__ __forceinline__ void mma_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         uint32_t accumulate) {
    if constexpr (DT == kF32)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "setp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
            "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
            : "memory");
}

// The instruction descriptor of the pair's M = 256, N = NX MMAs.
template <int DT, int NX>
__host__ __device__ constexpr uint32_t wd_idesc() {
    if constexpr (DT == kF32)
        return idesc_tf32_f32(256, NX);
    else
        return idesc_f16kind_f32<DT>(256, NX);
}

// Arrive once on the barrier at this offset in both CTAs of the pair when
// every tcgen05 operation this thread issued so far has completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            bar),
        "h"(static_cast<uint16_t>(3))
        : "memory");
}

// GEGLU: the weight is a gate/up pair [2F, K] (gate rows first) and each
// CTA's 128 weight rows are 64 gate rows and the 64 up rows of the same
// outputs; the epilogue writes gelu_tanh(gate) * up, [M, F].
template <int NX, int DT, bool GEGLU>
__global__ void __launch_bounds__(kWdThreads, 1)
wide_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w, const WdArgs args) {
    using C = WdCfg<NX>;
    static_assert(DT == kBF16 || DT == kF16 || DT == kF32, "compute dtypes");
    constexpr int SX = C::SX, SA = C::SA, SP = C::SP;
    // A ring slice is 128 bytes of each row: one NF4 block (K-slice) of a
    // 16-bit type, half of one of fp32 (read by the MMAs as tf32).
    constexpr int SPB = DT == kF32 ? 2 : 1;                // ring slices per K-slice
    constexpr int kSliceVals = 128 / elem_bytes<DT>();     // values of a row in one ring slice
    constexpr int HX = NX / 2;   // activation rows of one accumulator held by each CTA
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
    const uint32_t rank = cluster_rank();   // 0: issues the pair's MMAs
    const int pair = static_cast<int>(blockIdx.x >> 1);
    // pairs run m-fastest: pairs resident together share each weight tile through L2
    const int m0 = (pair % args.m_tiles) * (2 * NX);
    // this CTA's first weight row (first gate row of a pair: the pair covers
    // 128 outputs, 64 per CTA)
    constexpr int kRowsOut = GEGLU ? C::BW / 2 : C::BW;
    const int n0 = (pair / args.m_tiles) * (2 * kRowsOut) + static_cast<int>(rank) * kRowsOut;
    const int nk = args.K / kBK;
    const int nks = nk * SPB;   // ring slices
    const int nst = (nk + kWdKs - 1) / kWdKs;

    if (threadIdx.x == 0) {
        // the MMA commits of both issuers release a slot, complete the
        // accumulators, drain
        for (int i = 0; i < SX; ++i) {
            mbar_init(xfull(i), 1);
            mbar_init(xempty(i), kWdIssuers);
        }
        for (int i = 0; i < SA; ++i) {
            // (even CTA) the warps of both CTAs that expand a ring slice: 8
            // per CTA for a 16-bit type, 4 for fp32
            mbar_init(afull(i), kWdConvWarps / SPB);
            mbar_init(aempty(i), kWdIssuers);
        }
        for (int i = 0; i < SP; ++i) {
            mbar_init(pfull(i), kPfullArrivals);
            mbar_init(pempty(i), kWdConvWarps);
        }
        mbar_init(accum, kWdIssuers);
        mbar_init(drain, kWdIssuers);
        *abort_flag = 0;
        fence_mbar_init();
    }
    const float* code_f32 = nullptr;   // fp32: the codebook, read by the converters
    if constexpr (DT == kF32) {
        __shared__ float s_code[16];
        if (threadIdx.x < 16) s_code[threadIdx.x] = c_code[threadIdx.x];
        code_f32 = s_code;
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // both CTAs' barriers exist before either signals the other
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();   // the previous kernel on the stream has finished
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------- activation producer: ring slice k into slot k % SX once
        // the pair's MMAs that read its previous contents completed.  Both
        // CTAs' copies complete on the even CTA's xfull barrier, which the even
        // CTA arms with the pair's bytes (the odd CTA's may land first: the
        // barrier's transaction count goes below zero until it is armed).
        if (lane == 0) {
            int issued = 0;
            for (int k = 0; k < nks; ++k) {
                const int x = k % SX;
                if (k >= SX &&
                    !mbar_wait_cluster(xempty(x), ((k / SX) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty))
                    break;
                if (*abort_flag) break;
                const uint32_t dst = smem_u32(smem + x * C::XS);
                // this CTA's halves of the two accumulators' activation rows
                const int r0 = m0 + static_cast<int>(rank) * HX;
                if (rank == 0) {
                    mbar_arrive_expect_tx(xfull(x), 2 * C::XS);
                    tma_load_2d(dst, &tm_x, xfull(x), k * kSliceVals, r0);
                    tma_load_2d(dst + HX * 128, &tm_x, xfull(x), k * kSliceVals, r0 + NX);
                } else {
                    tma_load_2d_pair_leader(dst, &tm_x, xfull(x), k * kSliceVals, r0);
                    tma_load_2d_pair_leader(dst + HX * 128, &tm_x, xfull(x), k * kSliceVals, r0 + NX);
                }
                ++issued;
            }
            if (*abort_flag) {
                if (rank == 0)
                    drain_ring(xfull(0), SX, issued, args.err);
                else   // its copies complete on the even CTA's barriers: give them time to land
                    spin_ns(kWdSettleNs);
            }
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
            produce_weights<C::BW, kWdKs, GEGLU>(pfull(p), lane, C::P_BYTES, &tm_w, smem_u32(ptile),
                                                 kb * kPackedRow, n0, args.N + n0, args.N,
                                                 smem_u32(ptile + C::P_BYTES), args.absmax, nk, kb, args.am_count,
                                                 args.err);
            ++issued;
        }
        if (*abort_flag && lane == 0) drain_ring(pfull(0), SP, issued, args.err);
    } else if (warp == 1 || warp == kWdIssuer1Warp) {
        if (lane == 0 && rank == 0) {
            // ---------------- MMA issuers of the pair, one thread per
            // accumulator (warp 1: activation rows m0 .. m0 + NX - 1, warp 19:
            // the next NX), each in a warp of its own: a single thread issuing
            // both accumulators' MMAs, with its two barrier checks per K-slice,
            // took about 0.7 us per K-slice against 0.5 us of tensor work.  Per
            // K-slice each waits until both CTAs expanded its weights and both
            // CTAs' activation halves landed, issues its 4 k-steps and commits
            // to both CTAs' barriers that release the K-slice's activation and
            // expanded-weight slots (each counts both issuers' commits).  For
            // fp32 the same per ring slice (half a K-slice, 4 tf32 k-steps of
            // 8 values: 32 bytes of each row, as for a 16-bit type).
            const int acc = warp == 1 ? 0 : 1;
            constexpr uint32_t idesc = wd_idesc<DT, NX>();
            // descriptors of slot 0, k-step 0; a slot or a k-step adds to the
            // 14-bit start-address field (address / 16), which never carries:
            // shared-memory addresses stay below 2^18
            const uint64_t a_desc0 = smem_desc_sw128(smem_u32(smem + C::OFF_A));
            const uint64_t b_desc0 = smem_desc_sw128(smem_u32(smem) + acc * HX * 128);
            const uint32_t d_tmem = tmem + acc * kWdAccStride;
            bool ok = true;
            for (int k = 0; k < nks; ++k) {
                const int a = k % SA;
                const int x = k % SX;
                ok = mbar_wait_cluster(afull(a), (k / SA) & 1, args.err, abort_flag, kErrTimeoutConverted) &&
                     mbar_wait_cluster(xfull(x), (k / SX) & 1, args.err, abort_flag, kErrTimeoutFull);
                if (!ok) break;
                tc_fence_after();
                const uint64_t ad = a_desc0 + static_cast<uint64_t>((a * C::A_KS) >> 4);
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((x * C::XS) >> 4);
#pragma unroll
                for (int j = 0; j < 4; ++j)   // k-step j of the ring slice: 32 bytes of each row
                    mma_pair<DT>(d_tmem, ad + 2 * j, bd + 2 * j, idesc, (k == 0 && j == 0) ? 0u : 1u);
                mma_commit_pair(xempty(x));
                mma_commit_pair(aempty(a));
            }
            if (ok) mma_commit_pair(accum);
            // On every path, the MMAs committed to both CTAs' drain barriers:
            // warp 1 of each CTA waits on it before releasing TMEM, so TMEM is
            // never freed under a running MMA (converters that gave up skip
            // their wait on accum).
            mma_commit_pair(drain);
        }
    } else {
        // ---------------- converters: unit u = (warp - 2) / 4 expands half
        // `part` of K-slice h of each stage for weight rows 32 q .. 32 q + 31
        // (q = warp % 4, the TMEM lane quarter this warp reads in the epilogue)
        const int u = (warp - 2) >> 2;
        const int h = u % kWdKs;
        const int part = u / kWdKs;
        const int q = warp & 3;
        const int r = q * 32 + lane;   // weight row within this CTA's 128
        const CodebookRegs cb = codebook_regs<DT == kF32 ? kBF16 : DT>();   // (unused for fp32)
        const uint32_t a_base = smem_u32(smem + C::OFF_A);
        bool ok = true;
        for (int st = 0; st < nst; ++st) {
            const int p = st % SP;
            const int k = st * kWdKs + h;
            const bool got = mbar_wait(pfull(p), (st / SP) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            const uint8_t* ptile = smem + C::OFF_P + p * C::P_SLOT;
            const bool live = k < nk;   // warp-uniform: the K-slice exists
            uint4 w4 = make_uint4(0, 0, 0, 0);
            float am = 0.0f;
            if (live) {
                am = reinterpret_cast<const float*>(ptile + C::P_BYTES)[h * C::BW + r];
                w4 = *reinterpret_cast<const uint4*>(ptile + C::packed_offset(r, 2 * h + part));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(pempty(p));   // this warp is done with packed slot p
            if (!live) continue;                      // the last stage of an odd number of K-slices
            // ring slice s: K-slice k, or (fp32) its half `part`; the expanded
            // slot must be free: the pair's MMAs of ring slice s - SA completed
            const int s = SPB * k + (SPB == 2 ? part : 0);
            const int a = s % SA;
            const bool free_slot = s < SA || mbar_wait_cluster(aempty(a), ((s / SA) - 1) & 1, args.err,
                                                               abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, free_slot)) {
                ok = false;
                break;
            }
            if constexpr (DT == kF32) {
                // 32 values of row r (this half of the K-slice) in fp32, rounded
                // to tf32: the whole 128-byte row of the slot, chunk c (4
                // values) stored at chunk c ^ (r % 8)
                uint32_t v[32];
                expand8_f32(w4.x, code_f32, am, v + 0);
                expand8_f32(w4.y, code_f32, am, v + 8);
                expand8_f32(w4.z, code_f32, am, v + 16);
                expand8_f32(w4.w, code_f32, am, v + 24);
                const uint32_t row = a_base + a * C::A_KS + r * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c)
                    sts128(row + ((c ^ (r & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            } else {
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
                const uint32_t row = a_base + a * C::A_KS + r * 128;
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    sts128(row + (((4 * part + c) ^ (r & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                           v[4 * c + 3]);
            }
            fence_proxy_async_smem();   // the MMAs read the slot through the async proxy
            __syncwarp();
            // Both CTAs' warps arrive on the even CTA's afull.  The odd CTA's
            // arrival is a CTA-scope release: the MMA that reads this slot runs
            // on this SM's tensor core through the async proxy, to which the
            // fence above has already made the stores visible, and it is issued
            // only after the arrival is observed (CUTLASS's cluster barrier
            // arrives from a peer CTA in the same default CTA-scope form).  A
            // cluster-scope release costs about 0.7 us per arrival (measured),
            // most of the converters' lead over the MMAs.
            if (lane == 0 && report_converted(st)) {
                if (rank == 0)
                    mbar_arrive(afull(a));
                else
                    mbar_arrive_remote_cta(afull(a), 0);
            }
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = __all_sync(0xffffffffu, ok) && mbar_wait_cluster(accum, 0, args.err, abort_flag, kErrTimeoutAccum);
        // accumulator acc: TMEM lane = weight row, column c = activation row
        // m0 + acc NX + c (both CTAs' halves); chunk ci = 16 columns of
        // accumulator ci / CHUNKS, chunks round-robin over the 4 units
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        constexpr int CHUNKS = NX / 16;
        auto load_chunk = [&](int ci, uint32_t (&v)[16]) {
            tmem_ld16(lane_addr + (ci / CHUNKS) * kWdAccStride + 16 * (ci % CHUNKS), v);
            tmem_ld_wait();
        };
        auto col_row = [&](int ci, int i) { return m0 + (ci / CHUNKS) * NX + 16 * (ci % CHUNKS) + i; };   // activation row
        if constexpr (GEGLU) {
            // Lanes 0-63 hold the gate rows n0 + r, lanes 64-127 the up rows of
            // the same outputs.  Of a unit's chunks u, u + 4, u + 8, ... the gate
            // warps (lane quarters 0-1) write u, u + 8, ... and the up warps
            // u + 4, u + 12, ...: first each side parks its raw values of the
            // chunks the other side writes in the activation ring (every TMA
            // load into it was read by an MMA that has completed, the peer's
            // included), then each side finishes its own chunks.  Every
            // converter thread reaches both named barriers on every path.
            constexpr int kConvThreads = 32 * kWdConvWarps;
            const bool all_ok = converters_and_all(__all_sync(0xffffffffu, ok), kConvThreads);
            float* xbuf = reinterpret_cast<float*>(smem);   // column c, pair row rr at c * 64 + rr
            const bool gate = q < 2;
            const int rr = gate ? r : r - C::BW / 2;
            if (all_ok) {
                tc_fence_after();
                fence_proxy_async_smem();   // the ring was last written by TMA
#pragma unroll 1
                for (int ci = u + (gate ? 4 : 0); ci < 2 * CHUNKS; ci += 8) {
                    uint32_t v[16];
                    load_chunk(ci, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) xbuf[(16 * ci + i) * (C::BW / 2) + rr] = __uint_as_float(v[i]);
                }
            }
            converters_sync(kConvThreads);
            if (all_ok) {
                const int n = n0 + rr;
#pragma unroll 1
                for (int ci = u + (gate ? 0 : 4); ci < 2 * CHUNKS; ci += 8) {
                    uint32_t v[16];
                    load_chunk(ci, v);
                    if (n < args.N) {
                        float o[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float mine = __uint_as_float(v[i]);
                            const float other = xbuf[(16 * ci + i) * (C::BW / 2) + rr];
                            o[i] = gate ? gelu_tanh(mine) * other : gelu_tanh(other) * mine;
                        }
                        store_col16<DT>(args.y, args.N, col_row(ci, 0), args.M, n, o, args.err);
                    }
                }
            }
        } else if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            const int n = n0 + r;
#pragma unroll 1
            for (int ci = u; ci < 2 * CHUNKS; ci += 4) {
                uint32_t v[16];
                load_chunk(ci, v);
                if (n < args.N) {
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = __uint_as_float(v[i]);
                    store_col16<DT>(args.y, args.N, col_row(ci, 0), args.M, n, o, args.err);
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync_all();   // the pair is done with both TMEMs before either frees them
    if (warp == 1) {
        int dummy = 0;   // bounded, whatever the abort flag says: the pair's MMAs have completed
        mbar_wait(drain, 0, args.err, &dummy, kErrTimeoutDrain);
        tc_fence_after();
        tmem_dealloc_pair(tmem, 512);
    }
}

// ============================================================ host side

struct WdPlan {
    int nx;        // activation rows per accumulator (MMA N), split between the pair
    int m_tiles;   // tiles of 2 nx activation rows
    int n_pairs;   // tiles of 256 weight rows
};

WdPlan make_wd_plan(int64_t M, int64_t N) {
    WdPlan p;
    p.m_tiles = static_cast<int>((M + 511) / 512);
    const int64_t rows = (M + p.m_tiles - 1) / p.m_tiles;   // balanced tiles of at most 512 rows
    p.nx = static_cast<int>(((rows + 1) / 2 + 31) / 32 * 32);
    p.n_pairs = static_cast<int>((N + 255) / 256);
    return p;
}

// N: rows of the weight (2F for a gate/up pair, whose output has F columns).
template <int NX, int DT, bool GEGLU>
cudaError_t launch_wd(const DeviceInfo& dev, const WdPlan& p, const void* x, int64_t M, int64_t K,
                      const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    using C = WdCfg<NX>;
    if (dev.smem_optin < C::SMEM) return cudaErrorInvalidConfiguration;
    auto kernel = wide_kernel<NX, DT, GEGLU>;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(kernel), C::SMEM, dev.ordinal); e != cudaSuccess)
        return e;
    CUtensorMap tm_x, tm_w;
    constexpr CUtensorMapDataType xdt = DT == kBF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : DT == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    constexpr int eb = elem_bytes<DT>();
    // activations: boxes of one ring slice (128 bytes of a row, the swizzle
    // span: 64 values of a 16-bit type, 32 of fp32) x NX / 2 rows; packed
    // weights: boxes of two K-slices x 128 rows (x 64 rows for a gate/up pair,
    // one box of gate rows and one of up rows)
    if (!make_map(&tm_x, x, xdt, eb, M, K, NX / 2, 128 / eb, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, GEGLU ? C::BW / 2 : C::BW,
                  kPackedRow * kWdKs, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;
    const int64_t ctas = 2 * static_cast<int64_t>(p.m_tiles) * p.n_pairs;
    if (ctas > 0x7fffffff) return cudaErrorInvalidConfiguration;
    const int64_t n_out = GEGLU ? N / 2 : N;
    WdArgs a{absmax, y, static_cast<int>(M), static_cast<int>(n_out), static_cast<int>(K), p.m_tiles, N * (K / kBK),
             dev.err_word};
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(ctas));
    cfg.blockDim = dim3(kWdThreads);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, tm_x, tm_w, a); e != cudaSuccess) return e;
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, bool GEGLU>
cudaError_t dispatch_wd(const DeviceInfo& dev, const WdPlan& p, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    switch (p.nx) {
        case 160: return launch_wd<160, DT, GEGLU>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 192: return launch_wd<192, DT, GEGLU>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 224: return launch_wd<224, DT, GEGLU>(dev, p, x, M, K, packed, absmax, N, y, s);
        case 256: return launch_wd<256, DT, GEGLU>(dev, p, x, M, K, packed, absmax, N, y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

// The tile kernel's time per K-slice and wave at fp32 (tf32 MMAs), in clocks.
constexpr double kTsSliceF32Clk = 1640.0;

// Whether the pair kernel takes this call, by a shape-only estimate of both
// kernels' time: waves of one CTA per SM times the time of a K-slice.  Measured
// on GB300 at M = 2048 (bf16, L2 flushed): about 0.52 us (1000 clocks) per
// K-slice for the tile kernel's 128 x 256 tile, and 0.53 us (1060 clocks, the
// slope of time over K) for a pair's 256 x 512 tile at nx = 256, the tensor
// rate -- its MMAs scale with nx, its converters and signalling do not, so
// smaller nx is not taken below the tile kernel's.
bool wide_applies(int dtype, int64_t M, int64_t N) {
    if ((dtype != kBF16 && dtype != kF16 && dtype != kF32) || M <= 256) return false;
    const WdPlan p = make_wd_plan(M, N);
    if (p.nx < 160 || p.nx > 256) return false;
    constexpr double kSms = 152.0;
    const double n_tiles = std::ceil(N / 128.0);
    const double ts_waves = std::ceil(n_tiles * std::ceil(M / 256.0) / kSms);
    const double wd_waves = std::ceil(2.0 * p.n_pairs * p.m_tiles / kSms);
    double wd_slice = std::max(1000.0, 1060.0 * p.nx / 256.0);
    double ts_slice = 1000.0;
    if (dtype == kF32) {   // two ring slices per K-slice; the tile kernel's tf32 K-slice
        wd_slice *= 2.0;
        ts_slice = kTsSliceF32Clk;
    }
    return wd_waves * wd_slice < ts_waves * ts_slice;
}

cudaError_t launch_gemm_wide(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                             const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s,
                             bool geglu) {
    if (geglu && N % 2 != 0) return cudaErrorInvalidValue;
    const WdPlan p = make_wd_plan(M, N);   // a pair of 256 weight rows = 128 gate/up row pairs
    switch (dtype) {
        case kBF16:
            return geglu ? dispatch_wd<kBF16, true>(dev, p, x, M, K, packed, absmax, N, y, s)
                         : dispatch_wd<kBF16, false>(dev, p, x, M, K, packed, absmax, N, y, s);
        case kF16:
            return geglu ? dispatch_wd<kF16, true>(dev, p, x, M, K, packed, absmax, N, y, s)
                         : dispatch_wd<kF16, false>(dev, p, x, M, K, packed, absmax, N, y, s);
        case kF32:
            return geglu ? dispatch_wd<kF32, true>(dev, p, x, M, K, packed, absmax, N, y, s)
                         : dispatch_wd<kF32, false>(dev, p, x, M, K, packed, absmax, N, y, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace nf4
