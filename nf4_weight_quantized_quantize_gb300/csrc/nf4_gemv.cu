// nf4_gemv.cu -- the NF4 linear for batches of at most 16 activation rows,
// Y[M, N] = X[M, K] . deq(W)[N, K]^T with M <= 16 (bf16 or fp16), the
// HBM-bound case: per weight element the kernel moves 0.5625 bytes and does
// only 2M flops, so it runs at the speed the packed weights stream in.
//
// This is the forward of the NF4 linear module of the diffuseR page "Gemma3
// NF4 on GPU" (#39, Summary: ltx23_nf4_linear) for a small batch.  As in the
// tile kernel, the weight is expanded in registers and never exists in the
// compute dtype in memory; here the expanded values go straight into the
// operand registers of warp-level tensor-core MMAs (mma.sync m16n8k16), so
// there is no hand-off between warps and nothing between expansion and MMA.
//
// Work split.  A CTA owns a tile of R = 128 or 256 weight rows and a range of
// K; a shape-only plan picks R and the number of K splits so that one wave of
// CTAs (one per SM) carries nearly equal work.  Stage i of the K range holds
// NF4 blocks BL i .. BL i + BL - 1 (BL = 8 for R = 128, 4 for R = 256), and
// the CTA's 16 consumer warps are 16 / BL sets of 4 row groups (16 rows each)
// x BL "block lanes": block lane b handles block BL i + b of every stage for
// its set's 4 row groups, so each warp reuses one block's activation fragments
// for 64 rows and its fixed costs per stage (the barrier wait, the fragment
// loads, the scale check) are spread over 4096 weights.  A 17th warp loads
// the stages: TMA boxes for the activations (16 rows x 64 values, 128-byte
// swizzle), the packed bytes (32 bytes x R rows per block) and the fp32
// block scales ([R rows][BL blocks]; 4-byte cp.async copies when K is not a
// multiple of 256).
//
// Fragments.  In an m16n8k16 MMA with A = 16 weight rows and B = 8 activation
// rows, lane (g = lane / 4, t = lane % 4) holds rows g and g + 8 and four
// values of the contraction index per step.  The contraction order inside an
// NF4 block is free as long as both operands use the same one, so lane t
// takes the block's physical k = 16t .. 16t + 15: for rows g and g + 8 that
// is one 8-byte packed read each, and for the activations two 16-byte reads
// per row.  Step s of the block uses the lane's packed bytes 2s and 2s + 1.
// The packed bytes arrive as 128-byte-wide boxes (4 blocks per row per TMA
// request: small boxes cap the request rate); fragment row g of a row group
// is weight row 2 (g % 4) + g / 4, which keeps those reads conflict-free
// under the 128-byte swizzle.
//
// Expansion.  A 64 KB byte table in shared memory holds, for every packed
// byte b and lane l, the two codebook values of b in the compute dtype (first
// element in the low half) at byte 256 b + 4 l: one byte permute builds the
// address (b in bits 8-15, 4 l in bits 0-7), one load fetches the pair, and
// one paired multiply scales it by the block absmax.  Every lane has its own
// copy, so a warp's 32 lookups never share a bank.  A product of two bf16 (or
// two fp16) values is exact in fp32 and the multiply rounds once, so the
// operand is DT_rne(float(DT(C[code])) * absmax): the dequantizer's value.
// When an absmax is not itself a DT value (a weight quantized at another
// dtype) the warp scales that block in fp32 instead, with the same result.
//
// K splits.  With more than one split, each CTA writes its fp32 partial tile
// to the workspace, and the last CTA of a tile to arrive (an atomic counter in
// the workspace header) sums all partials in split order -- the same order
// whichever CTA is last, so results are deterministic -- and writes Y.  It
// then returns the counter to zero, so every call leaves the header as it
// found it.  Gate/up pairs (GEGLU) put 8 gate rows and the 8 up rows of the
// same outputs in one row group, so a lane holds both and writes
// gelu_tanh(gate) * up directly.
//
// Every wait is bounded (NF4_WAIT_LIMIT_NS).  On expiry the CTA records an
// error code, stops loading, and still writes NaN partials and arrives on its
// tile's counter, so the counters stay consistent; Y is then undefined.
#include <algorithm>

#include <cudaTypedefs.h>

#include "nf4_device.cuh"
#include "nf4_launch.h"

namespace nf4 {

namespace {

constexpr int kGvRgw = 4;                        // row groups (16 rows) per consumer warp
constexpr int kGvWarps = 16;                     // consumer warps
constexpr int kGvThreads = 32 * (kGvWarps + 1);  // + the producer warp
constexpr int kGvLutBytes = 256 * 256;           // entry b of lane l at byte 256 b + 4 l
constexpr int kGvXBox = 16 * 128;                // 16 activation rows x 64 values x 2 bytes
constexpr int kGvSmemLimit = 232448;
constexpr int kGvSms = 152;                      // one wave on a GB300
constexpr int kGvMaxTiles = 1024;                // arrival counters in the workspace header
constexpr size_t kGvHeaderBytes = 4096;          // kGvMaxTiles 32-bit counters

// BL: NF4 blocks per stage = block lanes; the 16 consumer warps are
// 16 / BL sets of kGvRgw row groups x BL block lanes, so a tile has
// R = 16 * kGvRgw * 16 / BL rows: 256 for BL = 4, 128 for BL = 8.
template <int BL>
struct GvCfg {
    static constexpr int SETS = kGvWarps / BL;
    static constexpr int RG = SETS * kGvRgw;           // row groups (16 rows) per tile
    static constexpr int R = 16 * RG;                  // weight rows per tile
    // packed bytes: one TMA box per 4 blocks (128 bytes of each of R rows,
    // 128-byte swizzle), BL / 4 of them per stage
    static constexpr int W_GROUP = R * 128;
    static constexpr int AM_BYTES = R * 4 * BL;        // the stage's scales: [row][BL blocks] fp32
    // stage layout: BL activation boxes and BL / 4 packed boxes (each 1 KB
    // aligned for the 128-byte swizzle), the scales [R rows][BL blocks]
    static constexpr int OFF_W = BL * kGvXBox;
    static constexpr int OFF_AM = OFF_W + (BL / 4) * W_GROUP;
    static constexpr int STAGE = (OFF_AM + AM_BYTES + 1023) / 1024 * 1024;
    static constexpr int OFF_RING = kGvLutBytes;
    static constexpr int BUDGET = kGvSmemLimit - 1024 - 256;   // alignment slack; barriers and flags
    static constexpr int SP_FIT = (BUDGET - OFF_RING) / STAGE;
    static constexpr int SP = SP_FIT > 8 ? 8 : SP_FIT;        // ring depth
    static constexpr int OFF_BAR = OFF_RING + SP * STAGE;
    static constexpr size_t SMEM = 1024 + OFF_BAR + 16 * SP + 64;
    static_assert(SP >= 3, "ring depth");
    static_assert(BL == 4 || BL == 8, "block lanes");
    static_assert(SMEM <= kGvSmemLimit, "shared memory budget");
};

struct GvArgs {
    const float* absmax;   // [rows, K / 64]
    void* y;               // [M, n_out]
    float* partials;       // [n_tiles, splits, RG, NT, 32 lanes, 4] fp32 (splits > 1)
    uint32_t* counters;    // [n_tiles] arrival counters, zero between calls
    int M, K;
    int rows;              // weight rows: N, or 2F for a gate/up pair
    int n_out;             // output columns: N, or F for a pair
    int n_tiles, splits, kb_per_split;
    int scale_tma;         // the scales come by TMA (K % 256 == 0), else by 4-byte copies
    int64_t part_floats;   // fp32 values the partials area holds
    int counter_count;     // arrival counters in the header
    uint32_t* err;
};

// Shared-memory reads at a byte offset from a shared pointer: plain loads,
// so the compiler can schedule them (the barrier waits are compiler fences).
template <typename T>
__device__ __forceinline__ T lds(const uint8_t* base, uint32_t off) {
    return *reinterpret_cast<const T*>(base + off);
}

__device__ __forceinline__ float4 ldg_cg_f4(const float* p) {
    float4 v;
    asm volatile("ld.global.cg.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "l"(p));
    return v;
}

// D (+)= A . B, m16n8k16, A and B of type DT (both bf16 or both fp16), fp32 D.
template <int DT>
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
    if constexpr (DT == kBF16)
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    else
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
            "{%0, %1, %2, %3};"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Whether a consumer warp reports stage i as consumed.  Always true in the
// library.  A test build (-DNF4_TEST_DROP_CONSUMED_ARRIVE) withholds the
// report of warp 0 for stage 0 -- a flag that nothing sets -- so the producer's
// bounded wait for that ring slot runs out and the timeout path can be
// checked on a GPU without faulting or hanging it.
__device__ __forceinline__ bool report_consumed(int warp, int i) {
#ifdef NF4_TEST_DROP_CONSUMED_ARRIVE
    return !(warp == 0 && i == 0);
#else
    (void)warp;
    (void)i;
    return true;
#endif
}

// Named barrier 1 over the 16 consumer warps (the producer never joins it).
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"r"(32 * kGvWarps) : "memory");
}

// Accumulator sets per row group and activation octet: two (even and odd
// MMA steps) while registers allow, so consecutive MMAs of a warp rarely wait
// on each other's accumulator.
template <int RGW, int NT>
constexpr int acc_sets() {
    return RGW * NT <= 4 ? 2 : 1;
}

// One block of the stage for the warp's RGW row groups: expand rows lo and hi
// (8 packed bytes each, the lane's share: wl[j], wh[j]) and run the block's
// four MMA steps against the activation fragments xl (activation rows 0-7)
// and xh (rows 8-15).  Each step covers all row groups, so its table loads
// and multiplies are independent of the previous step's MMAs.  EXACT:
// every absmax of the block is a DT value (one paired DT multiply); else each
// value is scaled in fp32 and rounded once.
template <int DT, int NT, int RGW, bool EXACT>
__device__ __forceinline__ void stage_mma(float (&acc)[RGW][NT][acc_sets<RGW, NT>()][4], const uint2 (&wl)[RGW],
                                          const uint2 (&wh)[RGW], const float (&aml)[RGW], const float (&amh)[RGW],
                                          const uint32_t (&xl)[8], const uint32_t (&xh)[8], const uint8_t* lut,
                                          uint32_t lane4) {
    constexpr int AS = acc_sets<RGW, NT>();
    // table entry of byte k (0-3) of word w, at byte b << 8 | 4 lane
    auto at = [&](uint32_t w, uint32_t k) { return lds<uint32_t>(lut, prmt(w, lane4, 0x5504u | (k << 4))); };
    uint32_t sl[RGW], sh[RGW];
#pragma unroll
    for (int j = 0; j < RGW; ++j) {
        sl[j] = pack2<DT>(aml[j], aml[j]);
        sh[j] = pack2<DT>(amh[j], amh[j]);
    }
    auto scale = [&](uint32_t e, uint32_t s2, float am) {
        if constexpr (EXACT)
            return mul2<DT>(e, s2);
        else
            return scale_entry<DT>(e, am);
    };
    // Per step: every row group's table loads first, then the multiplies, then
    // the MMAs -- 16 independent loads in flight before the first use (about
    // 7 % faster on down_proj at M = 16 than one row group after another).
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        const uint32_t k = (2 * s) & 3;
        uint32_t e[RGW][4];   // A fragment registers a0..a3 of each row group
#pragma unroll
        for (int j = 0; j < RGW; ++j) {
            const uint32_t w0 = s < 2 ? wl[j].x : wl[j].y, w1 = s < 2 ? wh[j].x : wh[j].y;
            e[j][0] = at(w0, k);
            e[j][2] = at(w0, k + 1);
            e[j][1] = at(w1, k);
            e[j][3] = at(w1, k + 1);
        }
#pragma unroll
        for (int j = 0; j < RGW; ++j) {
            e[j][0] = scale(e[j][0], sl[j], aml[j]);
            e[j][2] = scale(e[j][2], sl[j], aml[j]);
            e[j][1] = scale(e[j][1], sh[j], amh[j]);
            e[j][3] = scale(e[j][3], sh[j], amh[j]);
        }
#pragma unroll
        for (int j = 0; j < RGW; ++j) {
            mma16816<DT>(acc[j][0][s % AS], e[j][0], e[j][1], e[j][2], e[j][3], xl[2 * s], xl[2 * s + 1]);
            if constexpr (NT == 2)
                mma16816<DT>(acc[j][1][s % AS], e[j][0], e[j][1], e[j][2], e[j][3], xh[2 * s], xh[2 * s + 1]);
        }
    }
}

// Write the finished values of one row group: rows lo (n_lo) and hi of the
// lane, activation rows nt * 8 + 2t and + 1.  A pair writes
// gelu_tanh(gate) * up for output n_lo (lo = gate row, hi = up row).
template <int DT, int NT, bool PAIR>
__device__ __forceinline__ void store_rows(const GvArgs& a, const float (&v)[NT][4], int n_lo, int t) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int m0 = nt * 8 + 2 * t;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int m = m0 + e;
            if (m >= a.M) continue;
            const int64_t i = static_cast<int64_t>(m) * a.n_out + n_lo;
            const int64_t count = static_cast<int64_t>(a.M) * a.n_out;
            if constexpr (PAIR) {
                if (n_lo < a.n_out && in_bounds(a.err, i, count))
                    store_out<DT>(a.y, i, gelu_tanh(v[nt][e]) * v[nt][2 + e]);
            } else {
                if (n_lo < a.n_out && in_bounds(a.err, i, count)) store_out<DT>(a.y, i, v[nt][e]);
                if (n_lo + 8 < a.n_out && in_bounds(a.err, i + 8, count)) store_out<DT>(a.y, i + 8, v[nt][2 + e]);
            }
        }
    }
}

// DT: bf16 or fp16.  BL: blocks per stage (tile R = 1024 / BL rows).
// NT: activation row octets (1: M <= 8, 2: M <= 16).  PAIR: gate/up pair.
template <int DT, int BL, int NT, bool PAIR>
__global__ void __launch_bounds__(kGvThreads, 1)
gemv_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
            const __grid_constant__ CUtensorMap tm_am, const GvArgs a) {
    using C = GvCfg<BL>;
    constexpr int SP = C::SP;
    constexpr int RGW = kGvRgw;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);   // 1 KB aligned
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bar_mem + 2 * SP);
    volatile int* last_flag = abort_flag + 1;
    const uint32_t bar0 = smem_u32(bar_mem);
    auto full = [&](int p) { return bar0 + 8u * p; };
    auto empty = [&](int p) { return bar0 + 8u * (SP + p); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tile = static_cast<int>(blockIdx.x % a.n_tiles);
    const int split = static_cast<int>(blockIdx.x / a.n_tiles);
    const int nk_total = a.K / kBlock;
    const int kb0 = split * a.kb_per_split;
    const int nkb = min(a.kb_per_split, nk_total - kb0);
    const int nst = (nkb + BL - 1) / BL;
    const int n0 = tile * (PAIR ? C::R / 2 : C::R);   // first weight row (gate row of a pair)

    if (threadIdx.x == 0) {
        for (int p = 0; p < SP; ++p) {
            // the expect-tx arrive (+ one cp.async arrive per producer lane when
            // the scales are copied without a tensor map)
            mbar_init(full(p), a.scale_tma ? 1 : 1 + 32);
            mbar_init(empty(p), kGvWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == kGvWarps && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
        if (a.scale_tma) tma_prefetch_desc(&tm_am);
    }
    __syncthreads();
    pdl_wait();   // the previous kernel on the stream has finished
    pdl_launch_dependents();
    // the producer starts loading at once; the consumers build the byte table
    // meanwhile (entry b of lane l at word 64 b + l: consumer thread c writes
    // the 16 copies of lanes 16 (c % 2) .. 16 (c % 2) + 15 of byte c / 2)
    if (warp < kGvWarps) {
        const uint32_t e = lut_entry<DT>(threadIdx.x >> 1);
        uint4* dst = reinterpret_cast<uint4*>(smem + 256 * (threadIdx.x >> 1) + 64 * (threadIdx.x & 1));
#pragma unroll
        for (int i = 0; i < 4; ++i) dst[i] = make_uint4(e, e, e, e);
        consumers_sync();
    }

    if (warp == kGvWarps) {
        // ---------------- producer: stage i into ring slot i % SP once every
        // consumer warp released what the slot held
        int issued = 0;
        for (int i = 0; i < nst; ++i) {
            const int p = i % SP;
            bool ok = true;
            if (i >= SP) ok = mbar_wait(empty(p), ((i / SP) - 1) & 1, a.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            const int kb = kb0 + BL * i;
            const int hv = min(BL, nkb - BL * i);   // blocks of this split in the stage
            uint8_t* st = smem + C::OFF_RING + p * C::STAGE;
            if (lane == 0) {
                const int ng = (hv + 3) / 4;   // packed boxes of 4 blocks
                mbar_arrive_expect_tx(full(p), static_cast<uint32_t>(hv * kGvXBox + ng * C::W_GROUP +
                                                                     (a.scale_tma ? C::AM_BYTES : 0)));
                if (a.scale_tma) {   // the stage's BL scales of every weight row
                    const uint32_t adst = smem_u32(st + C::OFF_AM);
                    tma_load_2d(adst, &tm_am, full(p), kb, n0);
                    if constexpr (PAIR) tma_load_2d(adst + (C::R / 2) * 4 * BL, &tm_am, full(p), kb, a.n_out + n0);
                }
                for (int h = 0; h < hv; ++h)
                    tma_load_2d(smem_u32(st + h * kGvXBox), &tm_x, full(p), (kb + h) * kBlock, 0);
                for (int gr = 0; gr < ng; ++gr) {
                    const uint32_t wdst = smem_u32(st + C::OFF_W + gr * C::W_GROUP);
                    const int xb = (kb + 4 * gr) * (kBlock / 2);
                    tma_load_2d(wdst, &tm_w, full(p), xb, n0);
                    if constexpr (PAIR) tma_load_2d(wdst + (C::R / 2) * 128, &tm_w, full(p), xb, a.n_out + n0);
                }
            }
            // scales without a tensor map (K not a multiple of 256): 4-byte
            // copies; rows at or past the weight's end copy a harmless in-range value
            for (int h = 0; h < hv && !a.scale_tma; ++h) {
                for (int row = lane; row < C::R; row += 32) {
                    int n;
                    bool in;
                    if constexpr (PAIR) {
                        const int half = row >= C::R / 2 ? 1 : 0;
                        const int j = row - half * (C::R / 2);
                        n = half * a.n_out + n0 + j;
                        in = n0 + j < a.n_out;
                    } else {
                        n = n0 + row;
                        in = n < a.rows;
                    }
                    const int64_t src = in ? static_cast<int64_t>(n) * nk_total + kb + h : 0;
                    if (in_bounds(a.err, src, static_cast<int64_t>(a.rows) * nk_total))
                        cp_async_4(smem_u32(st + C::OFF_AM + (row * BL + h) * 4), a.absmax + src);
                }
            }
            if (!a.scale_tma) cp_async_arrive_noinc(full(p));
            ++issued;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (*abort_flag && lane == 0) {
            // wait (bounded) for the loads still in flight before the CTA may exit
            int dummy = 0;
            for (int i = max(0, issued - SP); i < issued; ++i)
                if (!mbar_wait(full(i % SP), (i / SP) & 1, a.err, &dummy, kErrTimeoutDrain)) break;
        }
        return;
    }

    // ---------------- consumers
    const int bl = warp % BL;       // block lane: block BL i + bl of stage i
    const int set = warp / BL;      // row groups set * RGW .. set * RGW + RGW - 1
    const int g = lane >> 2;
    const int t = lane & 3;
    // fragment row g of a row group is weight row rho (and rho + 8) of it:
    // half-warp 0 takes the even rows 0, 2, 4, 6 and half-warp 1 the odd
    // ones, so each half-warp's 8-byte reads hit 8 different swizzled chunks
    const int rho = 2 * (g & 3) + (g >> 2);
    const uint32_t lane4 = static_cast<uint32_t>(lane) * 4u;

    constexpr int AS = acc_sets<RGW, NT>();
    float acc[RGW][NT][AS][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int c = 0; c < AS; ++c)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[j][nt][c][q] = 0.0f;

    bool ok = true;
    for (int i = 0; i < nst; ++i) {
        const int p = i % SP;
        const bool got = mbar_wait(full(p), (i / SP) & 1, a.err, abort_flag, kErrTimeoutFull);
        if (!__all_sync(0xffffffffu, got)) {
            ok = false;
            break;
        }
        if (BL * i + bl < nkb) {   // warp-uniform
            const uint8_t* st = smem + C::OFF_RING + p * C::STAGE;
            // activation rows g and g + 8, values 16t .. 16t + 15: 16-byte chunks
            // 2t and 2t + 1 of the row, stored at chunk ^ (row % 8)
            const uint8_t* xs = st + bl * kGvXBox;
            uint32_t xl[8], xh[8];
            {
                const uint4 v0 = lds<uint4>(xs, g * 128 + (((2 * t) ^ g) << 4));
                const uint4 v1 = lds<uint4>(xs, g * 128 + (((2 * t + 1) ^ g) << 4));
                xl[0] = v0.x; xl[1] = v0.y; xl[2] = v0.z; xl[3] = v0.w;
                xl[4] = v1.x; xl[5] = v1.y; xl[6] = v1.z; xl[7] = v1.w;
            }
            if constexpr (NT == 2) {
                const uint4 v0 = lds<uint4>(xs, (g + 8) * 128 + (((2 * t) ^ g) << 4));
                const uint4 v1 = lds<uint4>(xs, (g + 8) * 128 + (((2 * t + 1) ^ g) << 4));
                xh[0] = v0.x; xh[1] = v0.y; xh[2] = v0.z; xh[3] = v0.w;
                xh[4] = v1.x; xh[5] = v1.y; xh[6] = v1.z; xh[7] = v1.w;
            } else {
#pragma unroll
                for (int q = 0; q < 8; ++q) xh[q] = 0u;
            }
            // block bl: 32-byte column c0 of its 4-block box; row r's 16-byte
            // chunk c is stored at chunk c ^ (r % 8)
            const uint8_t* wsm = st + C::OFF_W + (bl >> 2) * C::W_GROUP;
            const int c0 = 2 * (bl & 3) + (t >> 1);
            auto wrow = [&](int r) { return lds<uint2>(wsm, r * 128 + ((c0 ^ (r & 7)) << 4) + ((t & 1) << 3)); };
            const float* am_s = reinterpret_cast<const float*>(st + C::OFF_AM) + bl;   // [row][BL blocks]
            // the lane's packed bytes and scales of every row group, loaded up front
            uint2 wl[RGW], wh[RGW];
            float aml[RGW], amh[RGW];
            bool exact = true;
#pragma unroll
            for (int j = 0; j < RGW; ++j) {
                const int rg = set * RGW + j;
                const int rlo = PAIR ? 8 * rg + rho : 16 * rg + rho;
                const int rhi = PAIR ? C::R / 2 + 8 * rg + rho : 16 * rg + 8 + rho;
                wl[j] = wrow(rlo);
                wh[j] = wrow(rhi);
                aml[j] = am_s[BL * rlo];
                amh[j] = am_s[BL * rhi];
                exact = exact && exact_in<DT>(aml[j]) && exact_in<DT>(amh[j]);
            }
            if (__all_sync(0xffffffffu, exact))
                stage_mma<DT, NT, RGW, true>(acc, wl, wh, aml, amh, xl, xh, smem, lane4);
            else
                stage_mma<DT, NT, RGW, false>(acc, wl, wh, aml, amh, xl, xh, smem, lane4);
        }
        __syncwarp();
        if (lane == 0 && report_consumed(warp, i)) mbar_arrive(empty(p));
    }
    ok = __all_sync(0xffffffffu, ok && !*abort_flag);
    // the accumulator sets of each row group and octet, summed (in set order)
    float res[RGW][NT][4];
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float v = acc[j][nt][0][q];
#pragma unroll
                for (int c = 1; c < AS; ++c) v += acc[j][nt][c][q];
                res[j][nt][q] = ok ? v : __uint_as_float(0x7fc00000u);
            }

    // ---------------- sum the BL block lanes of each set (fixed order) through
    // shared memory: the ring is idle once every consumer warp is here (each
    // waited for every stage, so every copy into it has landed)
    consumers_sync();
    float* red = reinterpret_cast<float*>(smem + C::OFF_RING);   // [set][bl][j][nt][q][lane]
#pragma unroll
    for (int j = 0; j < RGW; ++j)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) red[((((set * BL + bl) * RGW + j) * NT + nt) * 4 + q) * 32 + lane] = res[j][nt][q];
    consumers_sync();

    // warp (set, bl) finishes row group j = bl of its set (bl < RGW)
    const bool owner = bl < RGW;
    const int j = bl;
    const int rg = set * RGW + j;
    float v[NT][4];
    if (owner) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                float s = red[((((set * BL + 0) * RGW + j) * NT + nt) * 4 + q) * 32 + lane];
#pragma unroll
                for (int b = 1; b < BL; ++b) s += red[((((set * BL + b) * RGW + j) * NT + nt) * 4 + q) * 32 + lane];
                v[nt][q] = s;
            }
    }
    const int n_lo = n0 + (PAIR ? 8 * rg : 16 * rg) + rho;   // output column of row lo

    if (a.splits == 1) {
        if (owner) store_rows<DT, NT, PAIR>(a, v, n_lo, t);
        return;
    }

    // ---------------- split K: publish this CTA's partial; the last CTA of the
    // tile to arrive sums all of them in split order and writes Y
    constexpr int kRgFloats = NT * 128;   // one row group's partial: NT x 32 lanes x 4
    // partial of split s: float4 index part(s) / 4 + 32 nt of the partials area
    auto part = [&](int s) {
        return ((static_cast<int64_t>(tile) * a.splits + s) * C::RG + rg) * kRgFloats + lane * 4;
    };
    const int64_t part_f4 = a.part_floats / 4;
    if (owner) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
            if (in_bounds(a.err, part(split) / 4 + 32 * nt, part_f4))
                *reinterpret_cast<float4*>(a.partials + part(split) + nt * 128) =
                    make_float4(v[nt][0], v[nt][1], v[nt][2], v[nt][3]);
    }
    // The barrier orders every consumer's partial before thread 0's arrival,
    // whose acquire-release atomic publishes them (cumulatively) to the CTA
    // that arrives last and acquires the others' partials for it.
    consumers_sync();
    if (threadIdx.x == 0) {
        uint32_t before = 0;
        if (in_bounds(a.err, tile, a.counter_count))
            asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(before) : "l"(a.counters + tile) : "memory");
        const bool last = before == static_cast<uint32_t>(a.splits - 1);
        if (last && in_bounds(a.err, tile, a.counter_count))
            a.counters[tile] = 0u;   // ready for the next call: nothing else touches it in this one
        *last_flag = last ? 1 : 0;
    }
    consumers_sync();
    if (!*last_flag || !owner) return;
    // all partials of the tile, summed in split order; loads issued 8 splits at a time
    float sum[NT][4];
    for (int s0 = 0; s0 < a.splits; s0 += 8) {
        float4 w4[8][NT];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int s = s0 + i;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (s == split)
                    w4[i][nt] = make_float4(v[nt][0], v[nt][1], v[nt][2], v[nt][3]);
                else if (s < a.splits)
                    w4[i][nt] = in_bounds(a.err, part(s) / 4 + 32 * nt, part_f4) ? ldg_cg_f4(a.partials + part(s) + nt * 128)
                                                                                : make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (s0 + i >= a.splits) break;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (s0 + i == 0) {
                    sum[nt][0] = w4[i][nt].x; sum[nt][1] = w4[i][nt].y; sum[nt][2] = w4[i][nt].z; sum[nt][3] = w4[i][nt].w;
                } else {
                    sum[nt][0] += w4[i][nt].x; sum[nt][1] += w4[i][nt].y; sum[nt][2] += w4[i][nt].z; sum[nt][3] += w4[i][nt].w;
                }
            }
        }
    }
    store_rows<DT, NT, PAIR>(a, sum, n_lo, t);
}

// ============================================================ host side

struct GvPlan {
    bool ok = false;
    int bl = 0;             // blocks per stage (tile R = 1024 / bl rows)
    int n_tiles = 0;
    int splits = 0;
    int kb_per_split = 0;
    int nt = 0;             // activation row octets
};

// The plan is a pure function of the shape (so the workspace size needs no
// device): the tile height and split count whose heaviest CTA carries the
// least work when one CTA runs per SM, plus a small charge per split for the
// final reduction.
GvPlan make_gv_plan(int64_t M, int64_t rows, int64_t K) {
    GvPlan best;
    if (M < 1 || M > 16 || rows < 1 || K < kBlock) return best;
    const int64_t nk = K / kBlock;
    const int64_t groups = (rows + 15) / 16;
    double best_cost = 1e300;
    for (int bl : {4, 8}) {
        const int64_t rg = (kGvWarps / bl) * kGvRgw;
        const int64_t n_tiles = (groups + rg - 1) / rg;
        if (n_tiles > kGvMaxTiles) continue;
        const int64_t smax = std::max<int64_t>(1, kGvSms / n_tiles);
        for (int64_t s = 1; s <= std::min<int64_t>(smax, (nk + bl - 1) / bl); ++s) {
            const int64_t per = ((nk + s - 1) / s + bl - 1) / bl * bl;   // whole stages
            const int64_t s_eff = (nk + per - 1) / per;
            const int64_t waves = (n_tiles * s_eff + kGvSms - 1) / kGvSms;
            const double cost = static_cast<double>(waves * rg * per) + (s_eff > 1 ? 0.2 * s_eff * rg : 0.0);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.ok = true;
                best.bl = bl;
                best.n_tiles = static_cast<int>(n_tiles);
                best.splits = static_cast<int>(s_eff);
                best.kb_per_split = static_cast<int>(per);
            }
        }
    }
    best.nt = M <= 8 ? 1 : 2;
    return best;
}

template <int DT, int BL, int NT, bool PAIR>
cudaError_t launch_gv(const DeviceInfo& dev, const GvPlan& p, const void* x, int64_t M, int64_t K,
                      const uint8_t* packed, const float* absmax, int64_t rows, void* y, void* workspace,
                      size_t ws_bytes, cudaStream_t s) {
    using C = GvCfg<BL>;
    if (dev.smem_optin < C::SMEM) return cudaErrorInvalidConfiguration;
    auto kernel = gemv_kernel<DT, BL, NT, PAIR>;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(kernel), C::SMEM, dev.ordinal); e != cudaSuccess)
        return e;
    CUtensorMap tm_x, tm_w, tm_am;
    const bool scale_tma = (K / kBlock) % 4 == 0;   // the scale rows' pitch is a multiple of 16 bytes
    const CUtensorMapDataType xdt = DT == kBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (!make_map(&tm_x, x, xdt, 2, M, K, 16, kBlock, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, rows, K / 2, PAIR ? C::R / 2 : C::R, 128,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    if (scale_tma) {
        if (!make_map(&tm_am, absmax, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, rows, K / kBlock, PAIR ? C::R / 2 : C::R,
                      BL, CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    } else {
        tm_am = tm_w;   // unused
    }
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    GvArgs a{absmax,
             y,
             reinterpret_cast<float*>(ws + kGvHeaderBytes),
             reinterpret_cast<uint32_t*>(ws),
             static_cast<int>(M),
             static_cast<int>(K),
             static_cast<int>(rows),
             static_cast<int>(PAIR ? rows / 2 : rows),
             p.n_tiles,
             p.splits,
             p.kb_per_split,
             scale_tma ? 1 : 0,
             static_cast<int64_t>((ws_bytes - kGvHeaderBytes) / sizeof(float)),
             static_cast<int>(kGvHeaderBytes / sizeof(uint32_t)),
             dev.err_word};
    const unsigned grid = static_cast<unsigned>(p.n_tiles) * static_cast<unsigned>(p.splits);
    if (cudaError_t e = launch_pdl(kernel, dim3(grid), dim3(kGvThreads), C::SMEM, s, tm_x, tm_w, tm_am, a); e != cudaSuccess)
        return e;
    count_launches(1);
    return cudaGetLastError();
}

template <int DT, bool PAIR>
cudaError_t dispatch_gv(const DeviceInfo& dev, const GvPlan& p, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t rows, void* y, void* ws, size_t ws_bytes,
                        cudaStream_t s) {
    if (p.bl == 4)
        return p.nt == 1 ? launch_gv<DT, 4, 1, PAIR>(dev, p, x, M, K, packed, absmax, rows, y, ws, ws_bytes, s)
                         : launch_gv<DT, 4, 2, PAIR>(dev, p, x, M, K, packed, absmax, rows, y, ws, ws_bytes, s);
    if (p.bl == 8)
        return p.nt == 1 ? launch_gv<DT, 8, 1, PAIR>(dev, p, x, M, K, packed, absmax, rows, y, ws, ws_bytes, s)
                         : launch_gv<DT, 8, 2, PAIR>(dev, p, x, M, K, packed, absmax, rows, y, ws, ws_bytes, s);
    return cudaErrorInvalidValue;
}

}  // namespace

bool gemv_applies(int dtype, int64_t M, int64_t rows, int64_t K) {
    return (dtype == kBF16 || dtype == kF16) && make_gv_plan(M, rows, K).ok;
}

size_t gemv_workspace_bytes(int64_t M, int64_t rows, int64_t K) {
    const GvPlan p = make_gv_plan(M, rows, K);
    if (!p.ok) return 0;
    size_t bytes = kGvHeaderBytes;
    if (p.splits > 1)
        bytes += static_cast<size_t>(p.n_tiles) * p.splits * ((kGvWarps / p.bl) * kGvRgw) * p.nt * 128 * sizeof(float);
    return bytes;
}

size_t gemv_header_bytes() { return kGvHeaderBytes; }

cudaError_t launch_gemv(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t rows, void* y, void* workspace,
                        size_t ws_bytes, cudaStream_t s, bool pair) {
    const GvPlan p = make_gv_plan(M, rows, K);
    if (!p.ok || (pair && rows % 2 != 0) || ws_bytes < gemv_workspace_bytes(M, rows, K) || workspace == nullptr)
        return cudaErrorInvalidValue;
    switch (dtype) {
        case kBF16:
            return pair ? dispatch_gv<kBF16, true>(dev, p, x, M, K, packed, absmax, rows, y, workspace, ws_bytes, s)
                        : dispatch_gv<kBF16, false>(dev, p, x, M, K, packed, absmax, rows, y, workspace, ws_bytes, s);
        case kF16:
            return pair ? dispatch_gv<kF16, true>(dev, p, x, M, K, packed, absmax, rows, y, workspace, ws_bytes, s)
                        : dispatch_gv<kF16, false>(dev, p, x, M, K, packed, absmax, rows, y, workspace, ws_bytes, s);
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace nf4
