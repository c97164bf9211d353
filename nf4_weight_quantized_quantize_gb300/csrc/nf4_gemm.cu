// nf4_gemm.cu -- fused NF4 weight-only GEMM on the 5th-generation tensor
// cores: Y[M, N] = X[M, K] . deq(W)[N, K]^T with X, Y and the dequantized
// weight in the compute dtype -- bf16 or fp16 (tcgen05 kind::f16) or fp32
// (kind::tf32) -- and fp32 accumulation in TMEM.
//
// This is the forward of the NF4 linear module of the diffuseR page "Gemma3
// NF4 on GPU" (#39, Summary: ltx23_nf4_linear, dequantize then a dense matmul
// at the compute dtype).  Instead of dequantizing the whole weight to HBM and
// calling a dense GEMM, each CTA expands its packed weight tile in registers
// and writes it straight into tensor memory, where the MMA reads it, so the
// weight crosses HBM at 0.5625 bytes per element and never touches shared
// memory in expanded form.
//
// One kernel template, three uses:
//   direct (M >= 128): CTA tile = 128 weight rows x NX activation rows
//       (NX <= 256), the whole K range, Y written by the epilogue.
//   split (M < 128):  NX = M rounded up to 16, K split over CTAs so every SM
//       streams weights; fp32 partials to a workspace, then an ordered
//       reduction kernel writes Y.
//   gate/up pair (GEGLU, M >= 128): the weight is the Gemma3 MLP's gate and
//       up projections stacked into one [2F, K] tensor; a tile's 128 rows are
//       64 gate rows and the 64 up rows of the same outputs, and the epilogue
//       writes gelu_tanh(gate) * up, [M, F], instead of both projections.
//
// The MMA runs "swap-AB": the converted weight tile is operand A (M = 128,
// in TMEM), the activation tile is operand B (N = NX, in shared memory, 128-byte
// swizzle, loaded by TMA), and the accumulator holds Y^T (TMEM lane = weight
// row, column = activation row).
//
// Warp roles: warp 0 lane 0 loads the activation tiles (TMA); warp 1
// allocates TMEM and lane 0 issues the MMAs (narrow tiles add a second
// issuer warp); the last warp loads the packed-weight tiles (TMA, lane 0)
// and copies the block scales (cp.async, all lanes); the warps in between
// are converters, 4 x KS x RS of them: each K-slice of a stage has RS groups
// of 4 warps (one thread per weight row, each taking 64 / RS of the row's
// values).  A 16-bit converter looks each 4-bit code up in the codebook of
// the compute dtype -- held in registers (byte permutes) on the direct path,
// in a per-lane shared-memory byte table on the split path -- scales it by
// the block absmax with one paired multiply and stores the values into its
// TMEM lane with tcgen05.st; an fp32 converter uses a 16-entry fp32 table,
// an fp32 multiply and rounds to tf32.  The converters then run the
// epilogue.  Every wait is bounded (NF4_WAIT_LIMIT_NS); on expiry the CTA
// records an error code, drains what it has in flight and returns.
#include <algorithm>
#include <mutex>
#include <type_traits>

#include <cudaTypedefs.h>

#include "nf4_convert.cuh"
#include "nf4_device.cuh"
#include "nf4_launch.h"

namespace nf4 {

// ============================================================ shared pieces

// Barriers, in shared memory.  A stage is KS consecutive K-slices.  Three
// rings carry it, each as deep as its storage allows:
//   TMEM ring (ST slots): the stage's converted weights;
//   activation ring (SX <= ST slots of shared memory): its activation tiles;
//   weight ring (SP slots of shared memory): its packed bytes and scales,
//     free again as soon as the converters have read them.
// Stage st uses TMEM slot st % ST, activation slot st % SX, weight slot
// st % SP.
//   xfull[s]   the stage's activation tiles landed (TMA)
//   conv[t]    the converter warps wrote the stage's weights into TMEM slot t
//   done[t]    the stage's MMAs completed (one commit per MMA issuer): TMEM
//              slot t may be rewritten, and the activation slot of stage st
//              (st % SX) may be refilled
//   pfull[p]   the stage's packed tile landed (TMA) and its scales were copied;
//              the weight producer issues these loads only after done[] of the
//              stage's TMEM slot, so pfull also means "TMEM slot free"
//   pempty[p]  every converter warp has read weight slot p
// plus accum (the accumulators are final) and one drain barrier per MMA
// issuer (error path only).
struct Barriers {
    uint32_t base;
    int nx, nt, np;
    __device__ uint32_t xfull(int s) const { return base + 8u * s; }
    __device__ uint32_t conv(int t) const { return base + 8u * (nx + t); }
    __device__ uint32_t done(int t) const { return base + 8u * (nx + nt + t); }
    __device__ uint32_t pfull(int p) const { return base + 8u * (nx + 2 * nt + p); }
    __device__ uint32_t pempty(int p) const { return base + 8u * (nx + 2 * nt + np + p); }
    __device__ uint32_t accum() const { return base + 8u * (nx + 2 * nt + 2 * np); }
    __device__ uint32_t drain(int issuer) const { return base + 8u * (nx + 2 * nt + 2 * np + 1 + issuer); }
    __host__ __device__ static constexpr int count(int xs, int ts, int ps) { return xs + 2 * ts + 2 * ps + 3; }
};

__device__ __forceinline__ void init_barriers(const Barriers& bar, int conv_arrivals, int mma_issuers) {
    for (int s = 0; s < bar.nx; ++s) mbar_init(bar.xfull(s), 1);
    for (int t = 0; t < bar.nt; ++t) {
        mbar_init(bar.conv(t), conv_arrivals);
        mbar_init(bar.done(t), mma_issuers);
    }
    for (int p = 0; p < bar.np; ++p) {
        mbar_init(bar.pfull(p), kPfullArrivals);
        mbar_init(bar.pempty(p), conv_arrivals);
    }
    mbar_init(bar.accum(), mma_issuers);
    mbar_init(bar.drain(0), 1);
    mbar_init(bar.drain(1), 1);
}

// Exit of an MMA issuer: commit every MMA it issued to its drain barrier.
// The TMEM owner waits on it (bounded, whatever the CTA's abort flag says)
// before releasing TMEM, so TMEM is never freed under a running MMA, on any
// path (converters that gave up skip their wait on the accumulators).
__device__ __forceinline__ void drain_mma(const Barriers& bar, int issuer) { mma_commit(bar.drain(issuer)); }

// ============================================================ the kernel

// Compile-time layout of one kernel instance: NX activation rows per tile
// (MMA N), stages of KS K-slices, RS converter threads per weight row and
// K-slice (each expands 64 / RS of the row's values), EB bytes per element
// of X and of the converted weights (2: bf16 / fp16, 4: fp32 read as tf32).
template <int NX, int KS, int RS, int LUT, int EB = 2>
struct TsCfg {
    static constexpr int BW = 128;                      // weight rows per tile (MMA M)
    static constexpr int XB = NX * kBK * EB;            // activation tile of one K-slice
    // A K-slice row of X is kBK * EB bytes: EB / 2 sub-tiles of 128-byte rows
    // (the 128-byte swizzle's span), XSUB bytes apart; one MMA covers 32 bytes
    // of K, so a K-slice takes MMAS of them
    static constexpr int XHALVES = EB / 2;
    static constexpr int XSUB = NX * 128;
    static constexpr int MMAS = kBK * EB / 32;
    static constexpr int WK = KS;                       // K-slices per weight slot
    static constexpr int P_BYTES = BW * kPackedRow * WK;
    static constexpr int AM_BYTES = BW * 4 * WK;
    static constexpr int X_SLOT = KS * XB;                               // activation ring slot
    static constexpr int P_SLOT = (P_BYTES + AM_BYTES + 1023) / 1024 * 1024;   // weight ring slot
    static constexpr int TMEM_COLS = 512;
    // NACC independent accumulators of NX columns each (MMA j of a K-slice
    // goes to accumulator j % NACC; the epilogue sums them): a narrow MMA
    // finishes faster than the accumulate chain turns around, so a single
    // accumulator would serialise small-NX tiles.
    static constexpr int NACC = NX <= 32 ? 4 : (NX <= 64 ? 2 : 1);
    static constexpr int ACC_STRIDE = (NX + 31) / 32 * 32;        // accumulator a at column a * ACC_STRIDE
    static constexpr int A_COL0 = NACC * ACC_STRIDE;
    // MMA issuers: a narrow MMA costs its issuing thread about as much as a
    // wide one, so small-NX tiles issue from two threads.  Issuer i takes the
    // K-slices h = i (mod MI) of every stage into its own NACC / MI
    // accumulators, which keeps each accumulator's summation order fixed.
    static constexpr int MI = (NACC >= 2 && KS >= 2) ? 2 : 1;
    static constexpr int ACC_PER_MI = NACC / MI;
    static constexpr int A_COLS = kBK * EB / 4;         // TMEM columns of one K-slice row (32 or 64)
    static constexpr int A_SLOT = A_COLS * KS;
    static constexpr int TMEM_SLOTS = (TMEM_COLS - A_COL0) / A_SLOT;
    static constexpr int SMEM_LIMIT = 232448;
    // LUT == 1: the converters expand through a 256-entry byte table
    // replicated once per lane (entry b of lane l at word 32 b + l, so a
    // warp's lookups never share a bank); LUT == 0: through register permutes
    static constexpr int LUT_BYTES = LUT != 0 ? 256 * 32 * 4 : 0;
    static constexpr int BUDGET = SMEM_LIMIT - 2048 - LUT_BYTES;   // alignment slack, barriers
    static constexpr int cmin(int a, int b) { return a < b ? a : b; }
    static constexpr int ST = cmin(TMEM_SLOTS, 8);
    // activation slots, at most ST (so a wait on done[] never falls two
    // phases behind), leaving room for 3 weight slots
    static constexpr int SX = cmin(ST, (BUDGET - 3 * P_SLOT) / X_SLOT);
    static constexpr int SP = cmin(8, (BUDGET - SX * X_SLOT) / P_SLOT);
    static constexpr int OFF_P = SX * X_SLOT;           // weight slot p: packed, then scales
    static constexpr int OFF_LUT = OFF_P + SP * P_SLOT;
    static constexpr int OFF_BAR = OFF_LUT + LUT_BYTES;
    // At least 120 KB, so no two CTAs share an SM: a second CTA there would
    // wait in tcgen05.alloc for the first one's 512 TMEM columns while
    // another SM idles.
    // after the barriers: the TMEM address, the abort flag and (fp32) the
    // 16 fp32 codebook values
    static constexpr int OFF_CODE = OFF_BAR + Barriers::count(SX, ST, SP) * 8 + 16;
    static constexpr size_t USED = 1024 + OFF_CODE + 64;
    static constexpr size_t SMEM = USED > 120 * 1024 ? USED : 120 * 1024;
    // warps: 0 activation producer, 1 MMA issuer, 2 .. 2 + CONV_WARPS - 1
    // converters (warp 2 + 4u + q: unit u, TMEM lane quarter q), then the
    // second MMA issuer (MI == 2) and the weight producer
    static constexpr int CONV_WARPS = 4 * KS * RS;
    static constexpr int ISSUER1_WARP = 2 + CONV_WARPS;
    static constexpr int WPROD_WARP = 2 + CONV_WARPS + (MI - 1);
    static constexpr int THREADS = 32 * (WPROD_WARP + 1);
    static_assert(NX % 16 == 0 && NX >= 16 && NX <= 256, "MMA N");
    static_assert(XB % 1024 == 0, "128B-swizzle tiles need 1 KB alignment");
    static_assert(SX >= 2 && ST >= SX && SP >= 3, "ring depths");
    static_assert(SMEM <= SMEM_LIMIT, "shared memory budget");
    static_assert(WK == 1 || WK == 2 || WK == 4, "packed rows of 32, 64 or 128 bytes");
    static_assert(LUT == 0 || LUT == 1, "expansion through permutes or the byte table");
    static_assert(RS == 1 || RS == 2, "converter threads per row");
    static_assert(EB == 2 || (EB == 4 && LUT == 0), "fp32 expands through the 16-entry code table");
    // The packed tile is loaded with the TMA swizzle whose span equals its
    // row (32 * WK bytes): the 16-byte chunk at byte offset o lands at chunk
    // (o / 16) XOR ((o / 128) mod 2 WK).  A converter warp reads one chunk
    // from each of 32 consecutive rows; the swizzle spreads them over all 32
    // banks, where plain rows would put them on the same four.
    static constexpr uint32_t SWZ_MASK = 2 * WK - 1;
    __device__ static uint32_t packed_offset(int row, int chunk) {
        const uint32_t o = static_cast<uint32_t>(row * kPackedRow * WK + 16 * chunk);
        return o ^ (((o >> 7) & SWZ_MASK) << 4);
    }
    static_assert(THREADS <= 1024, "block size");
};

struct TsArgs {
    const float* absmax;  // [N, K/64] ([2N, K/64] for a gate/up pair)
    void* y;              // [M, N] of the compute dtype (direct, gate/up pair)
    float* ws;            // [splits, M, N] fp32 partials (split)
    int M, N, K;          // N: output columns (rows of one half of a gate/up pair)
    int kb_per_split;
    int m_tiles;
    int64_t am_count;     // scales in absmax
    int64_t ws_floats;    // fp32 values the workspace holds (split)
    uint32_t* err;
};

// DT: the compute dtype of X, Y and the converted weights: bf16 or fp16
// (kind::f16) or fp32 (kind::tf32).
template <int NX, int KS, int RS, int LUT, bool SPLIT, bool GEGLU, int DT>
__global__ void __launch_bounds__(TsCfg<NX, KS, RS, LUT, elem_bytes<DT>()>::THREADS, 1)
ts_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
          const TsArgs args) {
    using C = TsCfg<NX, KS, RS, LUT, elem_bytes<DT>()>;
    static_assert(DT == kBF16 || DT == kF16 || DT == kF32, "compute dtypes");
    static_assert(!(SPLIT && GEGLU), "a gate/up pair sums its split-K partials before the activation");
    // output columns per tile: 128 weight rows, or 64 gate/up row pairs
    constexpr int HW = GEGLU ? C::BW / 2 : C::BW;
    // the up half's accumulators go through the (idle) activation ring
    static_assert(!GEGLU || C::SX * C::X_SLOT >= NX * HW * 4, "gate/up exchange buffer");
    constexpr int SX = C::SX;
    constexpr int ST = C::ST;
    constexpr int SP = C::SP;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bar_mem = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bar_mem + Barriers::count(SX, ST, SP));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    const Barriers bar{smem_u32(bar_mem), SX, ST, SP};

    auto x_tile = [&](int s, int h) { return smem + (s * KS + h) * C::XB; };
    auto p_tile = [&](int p) { return smem + C::OFF_P + p * C::P_SLOT; };
    auto am_tile = [&](int p) { return reinterpret_cast<const float*>(smem + C::OFF_P + p * C::P_SLOT + C::P_BYTES); };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // tiles run m-fastest: CTAs resident together share each weight tile through L2
    const int m0 = static_cast<int>(blockIdx.x % args.m_tiles) * NX;
    const int n0 = static_cast<int>(blockIdx.x / args.m_tiles) * HW;
    const int split = blockIdx.y;
    const int nk_total = args.K / kBK;
    const int kb0 = split * args.kb_per_split;
    const int nk = min(args.kb_per_split, nk_total - kb0);
    const int nst = (nk + KS - 1) / KS;   // stages; the last may hold fewer than KS K-slices

    uint32_t* lut = reinterpret_cast<uint32_t*>(smem + C::OFF_LUT);
    if constexpr (LUT != 0) {
        for (int e = threadIdx.x; e < 256 * 32; e += C::THREADS) lut[e] = lut_entry<DT>(static_cast<uint32_t>(e >> 5));
    }
    float* code_f32 = reinterpret_cast<float*>(smem + C::OFF_CODE);
    if constexpr (DT == kF32) {
        if (threadIdx.x < 16) code_f32[threadIdx.x] = c_code[threadIdx.x];
    }
    if (threadIdx.x == 0) {
        init_barriers(bar, C::CONV_WARPS, C::MI);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tm_x);
        tma_prefetch_desc(&tm_w);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();                      // the previous kernel on the stream has finished
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------- activation producer: lane 0 refills activation slot
        // s with the stage's KS tiles once the MMAs that read it (stage st - SX)
        // completed
        if (lane == 0) {
            int issued = 0;
            for (int st = 0; st < nst; ++st) {
                const int s = st % SX;
                const int prev = st - SX;
                if (prev >= 0 &&
                    !mbar_wait(bar.done(prev % ST), (prev / ST) & 1, args.err, abort_flag, kErrTimeoutEmpty))
                    break;
                if (*abort_flag) break;
                const int kb = kb0 + st * KS;
                mbar_arrive_expect_tx(bar.xfull(s), C::X_SLOT);
#pragma unroll
                for (int h = 0; h < KS; ++h) {
#pragma unroll
                    for (int x = 0; x < C::XHALVES; ++x)   // 128-byte column blocks of the K-slice
                        tma_load_2d(smem_u32(x_tile(s, h) + x * C::XSUB), &tm_x, bar.xfull(s),
                                    (kb + h) * kBK + x * (kBK / C::XHALVES), m0);
                }
                ++issued;
            }
            if (*abort_flag) drain_ring(bar.xfull(0), SX, issued, args.err);
        }
    } else if (warp == C::WPROD_WARP) {
        // ---------------- weight producer: refills weight slot p with stage
        // st once every converter warp has read what the slot held and the MMAs
        // that last read the stage's TMEM slot completed -- so pfull alone
        // tells a converter warp it may go ahead (one barrier wait per stage).
        int issued = 0;
        for (int st = 0; st < nst; ++st) {
            const int p = st % SP;
            bool ok = true;
            if (st >= SP) ok = mbar_wait(bar.pempty(p), ((st / SP) - 1) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            const int prev = st - ST;   // MMAs of stage `prev` (same TMEM slot) must be done
            if (ok && prev >= 0)
                ok = mbar_wait(bar.done(prev % ST), (prev / ST) & 1, args.err, abort_flag, kErrTimeoutEmpty);
            if (!__all_sync(0xffffffffu, ok && !*abort_flag)) break;
            const int kb = kb0 + st * KS;
            produce_weights<C::BW, KS, GEGLU>(bar.pfull(p), lane, C::P_BYTES, &tm_w, smem_u32(p_tile(p)),
                                                 kb * kPackedRow, n0, args.N + n0, args.N, smem_u32(am_tile(p)),
                                                 args.absmax, nk_total, kb, args.am_count, args.err);
            ++issued;
        }
        if (*abort_flag && lane == 0) drain_ring(bar.pfull(0), SP, issued, args.err);
    } else if (warp == 1 || (C::MI == 2 && warp == C::ISSUER1_WARP)) {
        // ---------------- MMA issuer(s): per stage, wait for the converted
        // weights and the activation tiles, one fence, the MMAs, one commit
        const int issuer = warp == 1 ? 0 : 1;
        if (lane == 0) {
            constexpr uint32_t idesc = [] {
                if constexpr (DT == kF32)
                    return idesc_tf32_f32(128, NX);
                else
                    return idesc_f16kind_f32<DT>(128, NX);
            }();
            // the activation-tile descriptors differ only in the start-address
            // field (low 14 bits): one base plus a compile-time or per-stage offset
            const uint64_t xdesc0 = smem_desc_sw128(smem_u32(x_tile(0, 0)));
            const uint32_t x_lo0 = static_cast<uint32_t>(xdesc0);
            const uint32_t x_hi = static_cast<uint32_t>(xdesc0 >> 32);
            const uint32_t acc0 = tmem + issuer * C::ACC_PER_MI * C::ACC_STRIDE;
            bool ok = true;
            for (int st = 0; st < nst && ok; ++st) {
                const int s = st % SX;
                const int t = st % ST;
                ok = mbar_wait(bar.conv(t), (st / ST) & 1, args.err, abort_flag, kErrTimeoutConverted) &&
                     mbar_wait(bar.xfull(s), (st / SX) & 1, args.err, abort_flag, kErrTimeoutFull);
                if (!ok) break;
                tc_fence_after();
                const int kbs = min(KS, nk - st * KS);
                const uint32_t a_col = tmem + C::A_COL0 + t * C::A_SLOT;
                const uint32_t x_lo = x_lo0 + static_cast<uint32_t>((s * KS * C::XB) >> 4);
                const uint32_t first = st > 0 ? 1u : 0u;   // accumulate into what earlier stages left
#pragma unroll
                for (int h = 0; h < KS; ++h) {
                    if (h % C::MI == issuer && h < kbs) {
#pragma unroll
                        for (int j = 0; j < C::MMAS; ++j) {
                            // 32 bytes of K: 8 TMEM columns of A; B at byte 32 (j % 4)
                            // of the rows of sub-tile j / 4
                            const uint32_t d = acc0 + (j % C::ACC_PER_MI) * C::ACC_STRIDE;
                            const uint32_t a = a_col + C::A_COLS * h + 8 * j;
                            const uint32_t b = x_lo + static_cast<uint32_t>((h * C::XB + (j / 4) * C::XSUB + 32 * (j % 4)) >> 4);
                            const uint32_t acc = (h >= C::MI || j >= C::ACC_PER_MI) ? 1u : first;
                            if constexpr (DT == kF32)
                                mma_tf32_ts2(d, a, b, x_hi, idesc, acc);
                            else
                                mma_bf16_ts2(d, a, b, x_hi, idesc, acc);
                        }
                    }
                }
                mma_commit(bar.done(t));
            }
            if (ok) mma_commit(bar.accum());
            drain_mma(bar, issuer);   // on every path (see drain_mma)
        }
    } else {
        // ---------------- converters: unit u = (warp - 2) / 4 converts part
        // u / KS (of RS) of K-slice u % KS of each stage for TMEM lane quarter
        // q = warp % 4 (one thread per weight row and part); then epilogue
        const int u = (warp - 2) >> 2;
        const int h = u % KS;                    // K-slice within the stage
        const int part = u / KS;                 // which 64 / RS values of the row
        const int q = warp & 3;                  // TMEM lane quarter this warp may access
        const int r = q * 32 + lane;             // weight row within the tile = TMEM lane
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(q * 32) << 16);
        const CodebookRegs cb = codebook_regs<DT == kF32 ? kBF16 : DT>();
        constexpr int D16 = DT == kF32 ? kBF16 : DT;   // the 16-bit type (unused for fp32)
        bool ok = true;
        for (int st = 0; st < nst; ++st) {
            const int p = st % SP;
            const int t = st % ST;
            // the stage's packed tile and scales; the weight producer loaded
            // them only after the MMAs that last read TMEM slot t
            const bool got = mbar_wait(bar.pfull(p), (st / SP) & 1, args.err, abort_flag, kErrTimeoutFull);
            if (!__all_sync(0xffffffffu, got)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // read this thread's share of the stage, then free the weight slot
            const uint8_t* ptile = p_tile(p);
            const bool live = st * KS + h < nk;           // warp-uniform: the K-slice exists
            uint4 q0 = make_uint4(0, 0, 0, 0), q1 = make_uint4(0, 0, 0, 0);
            float am = 0.0f;
            if (live) {
                am = am_tile(p)[h * C::BW + r];
                if constexpr (RS == 1) {
                    q0 = *reinterpret_cast<const uint4*>(ptile + C::packed_offset(r, 2 * h));
                    q1 = *reinterpret_cast<const uint4*>(ptile + C::packed_offset(r, 2 * h + 1));
                } else {
                    q0 = *reinterpret_cast<const uint4*>(ptile + C::packed_offset(r, 2 * h + part));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar.pempty(p));   // this warp is done with weight slot p
            const uint32_t col = lane_addr + C::A_COL0 + t * C::A_SLOT + C::A_COLS * h;
            if (DT == kF32 && live) {
                // 64 fp32 values per row and K-slice: 64 TMEM columns
                uint32_t v[32];
                expand8_f32(q0.x, code_f32, am, v + 0);
                expand8_f32(q0.y, code_f32, am, v + 8);
                expand8_f32(q0.z, code_f32, am, v + 16);
                expand8_f32(q0.w, code_f32, am, v + 24);
                tmem_st32(col + 32 * (RS == 1 ? 0 : part), v);
                if constexpr (RS == 1) {
                    expand8_f32(q1.x, code_f32, am, v + 0);
                    expand8_f32(q1.y, code_f32, am, v + 8);
                    expand8_f32(q1.z, code_f32, am, v + 16);
                    expand8_f32(q1.w, code_f32, am, v + 24);
                    tmem_st32(col + 32, v);
                }
                tmem_st_wait();
            } else if (DT != kF32 && live) {
                const uint32_t* lut_lane = lut + lane;
                // An absmax that is a D16 value scales in one paired D16 multiply
                // (exact product, one rounding); any other absmax (a weight
                // quantized at another dtype) scales each value in fp32 and
                // rounds once -- the dequantizer's value either way.
                const bool exact = exact_in<D16>(am);
                const uint32_t am2 = exact ? pack2<D16>(am, am) : pack2<D16>(1.0f, 1.0f);
                auto expand = [&](uint32_t word, uint32_t* o) {
                    if constexpr (LUT == 1)
                        expand8_lut<D16>(word, lut_lane, am2, o);
                    else
                        expand8<D16>(word, cb, am2, o);
                    if (!exact) {
#pragma unroll
                        for (int i = 0; i < 4; ++i) o[i] = scale_entry<D16>(o[i], am);
                    }
                };
                if constexpr (RS == 1) {
                    uint32_t v[32];
                    expand(q0.x, v + 0);
                    expand(q0.y, v + 4);
                    expand(q0.z, v + 8);
                    expand(q0.w, v + 12);
                    expand(q1.x, v + 16);
                    expand(q1.y, v + 20);
                    expand(q1.z, v + 24);
                    expand(q1.w, v + 28);
                    tmem_st32(col, v);
                } else {
                    // 16 packed bytes = 32 values = 16 TMEM columns
                    uint32_t v[16];
                    expand(q0.x, v + 0);
                    expand(q0.y, v + 4);
                    expand(q0.z, v + 8);
                    expand(q0.w, v + 12);
                    tmem_st16(col + 16 * part, v);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0 && report_converted(st)) mbar_arrive(bar.conv(t));
        }
        // tcgen05.ld is warp-collective: decide for the whole warp
        ok = ok && mbar_wait(bar.accum(), 0, args.err, abort_flag, kErrTimeoutAccum);
        // accumulators of an issuer that had no K-slice were never written
        const int nacc = min(C::MI, min(KS, nk)) * C::ACC_PER_MI;
        // sum of the NACC accumulators of this lane's row at columns c0 .. c0 + 15
        auto load_acc = [&](int c0, uint32_t (&v)[16]) {
            tmem_ld16(lane_addr + c0, v);
            tmem_ld_wait();
#pragma unroll
            for (int a = 1; a < C::NACC; ++a) {
                if (a >= nacc) break;
                uint32_t w[16];
                tmem_ld16(lane_addr + a * C::ACC_STRIDE + c0, w);
                tmem_ld_wait();
#pragma unroll
                for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + __uint_as_float(w[i]));
            }
        };
        if constexpr (GEGLU) {
            // Lanes 0-63 hold the gate rows n0 + r, lanes 64-127 the up rows of
            // the same outputs.  A warp's 16-column chunks alternate between
            // its two halves of the work: the gate warps write the even chunks
            // of Y and the up warps the odd ones.  First each side parks its
            // raw accumulators of the chunks the other side writes in shared
            // memory (the activation ring: every load into it was read by an
            // MMA that has completed); then each side finishes its own chunks
            // with the other's values.  Every converter thread reaches both
            // barriers whatever happened before.
            constexpr int kConvThreads = 32 * C::CONV_WARPS;
            constexpr int kStride = 16 * KS * RS;           // between a warp's chunks
            const bool all_ok = converters_and_all(__all_sync(0xffffffffu, ok), kConvThreads);
            float* xbuf = reinterpret_cast<float*>(smem);   // [NX][64]: column c, pair row rr at c * 64 + rr
            const bool gate = q < 2;
            const int rr = gate ? r : r - HW;               // row within the 64 pairs
            if (all_ok) {
                tc_fence_after();
                fence_proxy_async_smem();   // the ring was last written by TMA, read by the MMAs
#pragma unroll 1
                for (int c0 = 16 * u + (gate ? kStride : 0); c0 < NX; c0 += 2 * kStride) {
                    uint32_t v[16];
                    load_acc(c0, v);
#pragma unroll
                    for (int i = 0; i < 16; ++i) xbuf[(c0 + i) * HW + rr] = __uint_as_float(v[i]);
                }
            }
            converters_sync(kConvThreads);
            if (all_ok) {
                const int n = n0 + rr;
#pragma unroll 1
                for (int c0 = 16 * u + (gate ? 0 : kStride); c0 < NX; c0 += 2 * kStride) {
                    uint32_t v[16];
                    load_acc(c0, v);
                    if (n < args.N) {
                        float o[16];
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float mine = __uint_as_float(v[i]);
                            const float other = xbuf[(c0 + i) * HW + rr];
                            o[i] = gate ? gelu_tanh(mine) * other : gelu_tanh(other) * mine;
                        }
                        store_col16<DT>(args.y, args.N, m0 + c0, args.M, n, o, args.err);
                    }
                }
            }
        } else if (__all_sync(0xffffffffu, ok)) {
            tc_fence_after();
            // accumulator: TMEM lane = weight row n, column c = activation row m0 + c;
            // 16-column chunks go round-robin over the KS * RS warps of each lane quarter
            const int n = n0 + r;
#pragma unroll 1
            for (int c0 = 16 * u; c0 < NX; c0 += 16 * KS * RS) {
                uint32_t v[16];
                load_acc(c0, v);
                if (n < args.N) {
                    float o[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] = __uint_as_float(v[i]);
                    if constexpr (SPLIT) {   // this split's fp32 partial, [splits][M][N]
                        const int64_t plane = static_cast<int64_t>(args.M) * args.N;
                        if (in_bounds(args.err, (split + 1) * plane - 1, args.ws_floats))
                            store_col16<kF32>(args.ws + split * plane, args.N, m0 + c0, args.M, n, o, args.err);
                    } else {
                        store_col16<DT>(args.y, args.N, m0 + c0, args.M, n, o, args.err);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        // every MMA of the CTA has completed (each issuer committed to its drain)
        int dummy = 0;
        for (int i = 0; i < C::MI; ++i) mbar_wait(bar.drain(i), 0, args.err, &dummy, kErrTimeoutDrain);
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Sum the split-K partials in split order and store once in DT.  ws holds
// ws_floats values.
template <int DT>
__global__ void splitk_reduce_kernel(const float* __restrict__ ws, int splits, int64_t mn, void* __restrict__ y,
                                     int64_t ws_floats, uint32_t* err) {
    pdl_wait();
    pdl_launch_dependents();
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < mn;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        auto at = [&](int64_t j) { return in_bounds(err, j, ws_floats) ? ws[j] : 0.0f; };
        float acc = at(i);
        for (int s = 1; s < splits; ++s) acc += at(static_cast<int64_t>(s) * mn + i);
        if (in_bounds(err, i, mn)) store_out<DT>(y, i, acc);
    }
}

// Gate/up pair, M < 128: the split-K partials cover all 2F rows
// ([splits, M, 2F]); sum the gate and the up partials in split order, then
// write DT(gelu(gate) * up), [M, F].
template <int DT>
__global__ void splitk_geglu_reduce_kernel(const float* __restrict__ ws, int splits, int64_t M, int64_t F,
                                           void* __restrict__ y, int64_t ws_floats, uint32_t* err) {
    pdl_wait();
    pdl_launch_dependents();
    const int64_t mn2 = M * 2 * F;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M * F;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t m = i / F, n = i - m * F;
        const int64_t g0 = m * 2 * F + n;   // gate partial of split 0; the up partial is F further
        const float* g = ws + g0;
        auto at = [&](int64_t j) { return in_bounds(err, g0 + j, ws_floats) ? g[j] : 0.0f; };
        float gs = at(0), us = at(F);
        for (int s = 1; s < splits; ++s) {
            gs += at(s * mn2);
            us += at(s * mn2 + F);
        }
        if (in_bounds(err, i, M * F)) store_out<DT>(y, i, gelu_tanh(gs) * us);
    }
}

// ============================================================ host helpers shared with the other kernels

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

}  // namespace

// 2-D row-major tensor [rows, cols] of `elem` bytes per element, box
// {box_cols, box_rows}, the given shared-memory swizzle; out-of-range reads fill 0.
bool make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elem, uint64_t rows,
              uint64_t cols, uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * static_cast<cuuint64_t>(elem)};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle,
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

// ============================================================ host side

namespace {

constexpr int kTargetCtas = 152;             // one wave on a GB300 (152 SMs)
constexpr int kBW = 128;            // weight rows per tile
constexpr int kKsDirect = 2;        // K-slices per stage, M >= 128
constexpr int kKsSplit = 4;         // K-slices per stage, M < 128
constexpr int kRsDirect = 2;        // converter threads per weight row, M >= 128
constexpr int kRsSplit = 1;         // converter threads per weight row, M < 128
constexpr int kLutDirect = 0;       // M >= 128: register permutes (the byte table costs an activation slot)
constexpr int kLutSplit = 1;        // M < 128: the per-lane byte table (shared memory is idle there)
// fp32 (tf32 MMA): activation tiles twice as large, so fewer K-slices per
// stage; the 16-entry fp32 code table instead of the byte tables.
constexpr int kKsDirectF32 = 1, kRsDirectF32 = 2;
constexpr int kKsSplitF32 = 2, kRsSplitF32 = 1;
static_assert(kKsSplit % kKsSplitF32 == 0, "split-K ranges are whole stages at every dtype");

// How a call is cut into CTAs: a pure function of the shape, so the
// workspace size needs no device query.
struct Plan {
    int nx;            // activation rows per tile (MMA N)
    int m_tiles, n_tiles;
    int splits, kb_per_split;
    bool split;        // fp32 partials + reduction (M < 128)
};

Plan make_plan(int64_t M, int64_t N, int64_t K) {
    Plan p;
    const int nk = static_cast<int>(K / kBK);
    p.n_tiles = static_cast<int>((N + kBW - 1) / kBW);
    if (M >= 128) {
        p.split = false;
        p.m_tiles = static_cast<int>((M + 255) / 256);
        const int64_t rows = (M + p.m_tiles - 1) / p.m_tiles;   // balanced tiles, at most 256 rows
        p.nx = static_cast<int>(((rows + 15) / 16) * 16);
        p.splits = 1;
        p.kb_per_split = nk;
    } else {
        p.split = true;
        p.m_tiles = 1;
        p.nx = static_cast<int>(((M + 15) / 16) * 16);
        int splits = std::max(1, kTargetCtas / std::max(1, p.n_tiles));
        splits = std::min(splits, nk);
        const int per = (nk + splits - 1) / splits;
        p.kb_per_split = (per + kKsSplit - 1) / kKsSplit * kKsSplit;   // whole stages
        p.splits = (nk + p.kb_per_split - 1) / p.kb_per_split;          // no empty split
    }
    return p;
}

template <int NX, int KS, int RS, int LUT, bool SPLIT, bool GEGLU, int DT>
cudaError_t launch_ts(const DeviceInfo& dev, const Plan& p, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                      const TsArgs& a, cudaStream_t s) {
    using C = TsCfg<NX, KS, RS, LUT, elem_bytes<DT>()>;
    if (dev.smem_optin < C::SMEM) return cudaErrorInvalidConfiguration;
    auto kernel = ts_kernel<NX, KS, RS, LUT, SPLIT, GEGLU, DT>;
    if (cudaError_t e = set_smem(reinterpret_cast<const void*>(kernel), C::SMEM, dev.ordinal); e != cudaSuccess)
        return e;
    const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
    if (tiles > 0x7fffffff || p.splits > 65535) return cudaErrorInvalidConfiguration;
    dim3 grid(static_cast<unsigned>(tiles), static_cast<unsigned>(p.splits));
    if (cudaError_t e = launch_pdl(kernel, grid, dim3(C::THREADS), C::SMEM, s, tm_x, tm_w, a); e != cudaSuccess)
        return e;
    count_launches(1);
    return cudaGetLastError();
}

template <bool SPLIT, int KS, int RS, int LUT, bool GEGLU, int DT>
cudaError_t dispatch_nx(const DeviceInfo& dev, const Plan& p, const CUtensorMap& tm_x, const CUtensorMap& tm_w,
                        const TsArgs& a, cudaStream_t s) {
    if constexpr (SPLIT) {
        switch (p.nx) {   // M < 128
            case 16: return launch_ts<16, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 32: return launch_ts<32, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 48: return launch_ts<48, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 64: return launch_ts<64, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 80: return launch_ts<80, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 96: return launch_ts<96, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 112: return launch_ts<112, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            case 128: return launch_ts<128, KS, RS, LUT, SPLIT, false, DT>(dev, p, tm_x, tm_w, a, s);
            default: return cudaErrorInvalidValue;
        }
    } else {
        switch (p.nx) {   // 128 <= rows per tile <= 256
            case 128: return launch_ts<128, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 144: return launch_ts<144, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 160: return launch_ts<160, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 176: return launch_ts<176, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 192: return launch_ts<192, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 208: return launch_ts<208, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 224: return launch_ts<224, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 240: return launch_ts<240, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            case 256: return launch_ts<256, KS, RS, LUT, SPLIT, GEGLU, DT>(dev, p, tm_x, tm_w, a, s);
            default: return cudaErrorInvalidValue;
        }
    }
}

// N: rows of the weight.  pair: the weight is a gate/up pair ([2F, K], N = 2F)
// and the GEGLU epilogue writes [M, F] (direct path only).
template <int DT>
cudaError_t launch_plan(const DeviceInfo& dev, const Plan& p, bool pair, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t N, void* y, float* ws,
                        int64_t ws_floats, cudaStream_t s) {
    if (pair && (p.split || N % 2 != 0)) return cudaErrorInvalidValue;
    CUtensorMap tm_x, tm_w;
    constexpr bool F32 = DT == kF32;
    const int ks = p.split ? (F32 ? kKsSplitF32 : kKsSplit) : (F32 ? kKsDirectF32 : kKsDirect);   // K-slices per stage
    // the packed box row is 32 * ks bytes; its swizzle span matches (TsCfg::packed_offset)
    const CUtensorMapSwizzle wsw = ks == 1 ? CU_TENSOR_MAP_SWIZZLE_32B
                                 : ks == 2 ? CU_TENSOR_MAP_SWIZZLE_64B
                                           : CU_TENSOR_MAP_SWIZZLE_128B;
    constexpr CUtensorMapDataType xdt = DT == kBF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                        : DT == kF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    constexpr int eb = elem_bytes<DT>();
    // one box = 128 bytes of a row (the swizzle span): 64 16-bit or 32 fp32 values
    if (!make_map(&tm_x, x, xdt, eb, M, K, p.nx, 128 / eb, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&tm_w, packed, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, N, K / 2, pair ? kBW / 2 : kBW,
                  kPackedRow * ks, wsw))
        return cudaErrorInvalidValue;
    TsArgs a{absmax, y, ws, static_cast<int>(M), static_cast<int>(pair ? N / 2 : N), static_cast<int>(K),
             p.kb_per_split, p.m_tiles, N * (K / kBlock), ws_floats, dev.err_word};
    if constexpr (F32) {
        if (p.split)
            return dispatch_nx<true, kKsSplitF32, kRsSplitF32, 0, false, DT>(dev, p, tm_x, tm_w, a, s);
        return pair ? dispatch_nx<false, kKsDirectF32, kRsDirectF32, 0, true, DT>(dev, p, tm_x, tm_w, a, s)
                    : dispatch_nx<false, kKsDirectF32, kRsDirectF32, 0, false, DT>(dev, p, tm_x, tm_w, a, s);
    } else {
        if (p.split)
            return dispatch_nx<true, kKsSplit, kRsSplit, kLutSplit, false, DT>(dev, p, tm_x, tm_w, a, s);
        return pair ? dispatch_nx<false, kKsDirect, kRsDirect, kLutDirect, true, DT>(dev, p, tm_x, tm_w, a, s)
                    : dispatch_nx<false, kKsDirect, kRsDirect, kLutDirect, false, DT>(dev, p, tm_x, tm_w, a, s);
    }
}

// The element type at run time -> the kernels' compile-time DT.
template <typename Fn>
cudaError_t with_dt(int dtype, Fn&& fn) {
    switch (dtype) {
        case kBF16: return fn(std::integral_constant<int, kBF16>{});
        case kF16: return fn(std::integral_constant<int, kF16>{});
        case kF32: return fn(std::integral_constant<int, kF32>{});
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_gemm(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                        const uint8_t* packed, const float* absmax, int64_t N, void* y, cudaStream_t s) {
    if (wide_applies(dtype, M, N)) return launch_gemm_wide(dev, dtype, x, M, K, packed, absmax, N, y, s);
    const Plan p = make_plan(M, N, K);
    if (p.split) return cudaErrorInvalidValue;
    return with_dt(dtype, [&](auto dt) {
        return launch_plan<decltype(dt)::value>(dev, p, false, x, M, K, packed, absmax, N, y, nullptr, 0, s);
    });
}

cudaError_t launch_gemm_geglu(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                              const uint8_t* packed, const float* absmax, int64_t F, void* y, cudaStream_t s) {
    if (wide_applies(dtype, M, 2 * F)) return launch_gemm_wide(dev, dtype, x, M, K, packed, absmax, 2 * F, y, s, true);
    // ceil(2F / 128) tiles of 128 weight rows = ceil(F / 64) tiles of 64 gate/up row pairs
    const Plan p = make_plan(M, 2 * F, K);
    if (p.split) return cudaErrorInvalidValue;
    return with_dt(dtype, [&](auto dt) {
        return launch_plan<decltype(dt)::value>(dev, p, true, x, M, K, packed, absmax, 2 * F, y, nullptr, 0, s);
    });
}

// The tcgen05 split-K path's fp32 partials, [splits, M, N].
static size_t split_partials_bytes(int64_t M, int64_t N, int64_t K) {
    const Plan p = make_plan(M, N, K);
    return static_cast<size_t>(p.splits) * M * N * sizeof(float);
}

// Every skinny workspace starts with the warp-MMA kernel's arrival counters
// (gemv_header_bytes(), zero between calls); the split-K partials of either
// path follow, so one workspace serves every dtype.
size_t skinny_workspace_bytes(const DeviceInfo*, int64_t M, int64_t N, int64_t K) {
    const size_t gv = gemv_workspace_bytes(M, N, K);
    const size_t split = gemv_header_bytes() + split_partials_bytes(M, N, K);
    return gv > split ? gv : split;
}

// N: rows of the weight; geglu: the weight is a gate/up pair (N = 2F) and
// the reduction writes gelu(gate) * up, [M, F].
cudaError_t launch_skinny(const DeviceInfo& dev, int dtype, const void* x, int64_t M, int64_t K,
                          const uint8_t* packed, const float* absmax, int64_t N, void* y, void* workspace,
                          size_t ws_bytes, cudaStream_t s, bool geglu) {
    if (ws_bytes < skinny_workspace_bytes(&dev, M, N, K) || (geglu && N % 2 != 0)) return cudaErrorInvalidValue;
    if (gemv_applies(dtype, M, N, K))   // M <= 16, bf16 or fp16: warp-MMA kernel, reduction fused
        return launch_gemv(dev, dtype, x, M, K, packed, absmax, N, y, workspace, ws_bytes, s, geglu);
    const Plan p = make_plan(M, N, K);
    if (!p.split) return cudaErrorInvalidValue;
    workspace = static_cast<uint8_t*>(workspace) + gemv_header_bytes();   // the counters stay untouched
    const int64_t ws_floats = static_cast<int64_t>((ws_bytes - gemv_header_bytes()) / sizeof(float));
    return with_dt(dtype, [&](auto dtc) {
        constexpr int DT = decltype(dtc)::value;
        if (cudaError_t e = launch_plan<DT>(dev, p, false, x, M, K, packed, absmax, N, y,
                                            static_cast<float*>(workspace), ws_floats, s);
            e != cudaSuccess)
            return e;
        const int64_t mn = geglu ? M * (N / 2) : M * N;   // outputs
        const int threads = 256;
        const int grid =
            static_cast<int>(std::min<int64_t>((mn + threads - 1) / threads, 4 * static_cast<int64_t>(dev.sm_count)));
        const float* wsf = static_cast<const float*>(workspace);
        cudaError_t e = geglu ? launch_pdl(splitk_geglu_reduce_kernel<DT>, grid, threads, 0, s, wsf, p.splits, M, N / 2,
                                           y, ws_floats, dev.err_word)
                              : launch_pdl(splitk_reduce_kernel<DT>, grid, threads, 0, s, wsf, p.splits, mn, y, ws_floats,
                                           dev.err_word);
        if (e != cudaSuccess) return e;
        count_launches(1);
        return cudaGetLastError();
    });
}

}  // namespace nf4
