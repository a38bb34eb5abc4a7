// matmul_tc.cu -- IQ4_XS x Q8_1 matmul on the 5th-generation tensor cores.
//
// Method (V100TPS engine page, new-kernel table and the tile-geometry passage
// after it): per 32-weight sub-block, an integer dot product of decoded
// codebook values with Q8_1 codes, scaled by d_w*(ls-32)*d_x into fp32.
//
// GB300 design.  sm_103a has no integer tcgen05 kind, so both operands
// travel as fp16 holding small integers exactly: the codebook values kv and
// the Q8_1 codes q.  Two MMAs (K = 16 each) per sub-block accumulate into
// the sub-block's own fp32 TMEM accumulator; every product and every partial
// sum is an integer below 2^24, so the accumulator holds the exact integer
// dot P of the sub-block.  The epilogue scales it in: acc += (P*d_x)*Sw with
// Sw = d_w*(ls-32).  One CTA owns 128 weight rows (= 128 TMEM lanes = UMMA M)
// and an activation tile of MT rows (= UMMA N); K is split over a cluster
// whose CTAs reduce their partial tiles through distributed shared memory.
// The kernel reads the Q8_1 arrays (qs, ds) as the quantizer wrote them.
//
// Warp-specialized roles, each a loop over the CTA's work, decoupled by
// mbarrier rings (kNP slots of tensor memory: the decoded A operand, 16
// columns per sub-block; the accumulators, MT columns per sub-block; the row
// scales, one column per sub-block).  Warp numbers are for two decoder
// groups; at MT = 16 a third group takes warps 8-11 and the others move up:
//   warps 0-7 (decoders)   G groups of four; group g takes units g, g+G,
//                          ....  Warp w decodes rows 32(w%4)..+31 from the
//                          staged W bytes to exact fp16 (one shared-memory
//                          table lookup per qs byte) and stores them with
//                          tcgen05.st straight into the A slot (row i in
//                          TMEM lane i), plus d_w*(ls-32) into the scale
//                          column, then arrives on the slot's a_full.
//   warps 8, 11 (MMA)      warp-uniform loops over even / odd units: the
//                          warp builds its unit's B operand from the staged
//                          Q8_1 codes (exact fp16, canonical K-major layout,
//                          K-permuted like the decoded weights), then one
//                          elected lane issues two tcgen05.mma 128 x MT x 16
//                          (A from tensor memory, B from shared memory) per
//                          sub-block and commits.
//   warp 9 (producer)      TMA: W stages of 512 weights per row (2D tensor
//                          map: one 128 x 272 B box of two IQ4_XS
//                          super-blocks, or two 128 x 144 B boxes of eight
//                          18-byte Q4_0 / IQ4_NL blocks each -- 144-byte rows
//                          keep the decoders' shared-memory reads at 4-way
//                          bank conflicts where 288-byte rows would be
//                          8-way); Q8_1 code stages of 4 sub-blocks (2D
//                          tensor map over qs, MT rows x 128 B, 128-byte
//                          swizzle, rows past M read as zeros).
//   warp 10                allocates and frees tensor memory, and turns each
//                          stage's activation scales d_x (fp16 in ds) into
//                          fp32 for the epilogue.
//   warps 12- (epilogue)   thread t reads row t's integer dots and scale,
//                          releases the slot, and accumulates
//                          (P*d_x)*d_w*(ls-32) in fp32 registers.
// Every mbarrier wait is bounded (2 s); a timeout sets the device error word
// and an abort flag that releases every other wait, the CTA drains its copies
// and frees its tensor memory, and the call's output is undefined.
#include <cuda.h>

#include <type_traits>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kTmemCols = 512;        // whole TMEM; one CTA per SM (see kMinSmem)
constexpr int kMaxCluster = 8;
constexpr int kMinSmem = 120 * 1024;  // > half of the SM's shared memory: one CTA per SM
constexpr int kACols = kSub / 2;      // 16 TMEM columns of fp16 pairs per sub-block
constexpr int kCoreSbo = 128;         // 8 rows x 16 B core matrices, contiguous along N
constexpr int kBStagesPerW = kSubPerPair / kBStageSubs;  // activation stages per W stage

template <int R>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

// Rows of other ranks' slices a rank receives in the split-K reduction, at
// most: max over S = 2..kMaxCluster of (S - 1) * ceil(128 / S).
constexpr int recv_rows_max() {
    int r = 0;
    for (int s = 2; s <= kMaxCluster; ++s) {
        const int v = (s - 1) * ((kTileN + s - 1) / s);
        r = v > r ? v : r;
    }
    return r;
}

// kPrep selects the activation operand: false -- the Q8_1 arrays, staged by
// TMA and turned into exact fp16 codes by the MMA warps, d_x applied in the
// epilogue (two MMAs per sub-block); true -- the prepared operand (each
// q*d_x as an exact hi / lo pair of fp16, written by the quantizer), loaded
// by bulk copies, d_x already inside the products (four MMAs per sub-block,
// one FMA per element in the epilogue, no per-CTA conversion).
template <int MT, int WT, bool kPrep>
struct TcCfg {
    static_assert(MT % 16 == 0 && MT >= 16 && MT <= kMaxMTile, "UMMA N for M=128");
    // W stage: 512 weights of each of the 128 rows, as kWBoxes TMA boxes of
    // kTileN rows x kWBoxBytes (each box a dense block of shared memory).
    static constexpr int kWBoxes = (WT == kWtIQ4XS) ? 1 : 2;
    static constexpr int kWBoxBytes = (WT == kWtIQ4XS) ? kPairBytes : kB18GroupBytes;
    static constexpr int kWRowBytes = kWBoxes * kWBoxBytes;  // bytes of one row per stage
    static constexpr int kWStage = kTileN * kWRowBytes;
    static_assert(kWBoxBytes % 16 == 0 && kWBoxBytes / 4 <= 256, "TMA box inner extent");
    // Warp roles.  Decoders: kDecGroups groups of four warps (warpgroups
    // 0..G-1); more groups hide more of the decode's latency where the
    // epilogue is light (three at MT = 16).  Then one control warpgroup
    // (MMA issuers, TMA producer, tensor-memory owner) and the epilogue
    // warpgroups.
    static constexpr int kDecGroups = (MT <= 16) ? 3 : 2;
    static constexpr int kDecWarps = 4 * kDecGroups;
    static constexpr int kMmaWarp0 = kDecWarps;       // MMA issuers (even / odd units)
    static constexpr int kProducerWarp = kDecWarps + 1;
    static constexpr int kTmemWarp = kDecWarps + 2;
    static constexpr int kMmaWarp1 = kDecWarps + 3;
    static constexpr int kEpiWarp0 = kDecWarps + 4;
    // Epilogue warpgroups: from MT = 48 on two, each owning half of the
    // activation rows (columns of every accumulator): the per-unit read and
    // scale-in of 128 x MT results then takes half as long, which matters
    // because only two to four units fit in tensor memory at once.
    static constexpr int kEpiGroups = (MT >= 48) ? 2 : 1;
    static constexpr int kMH = MT / kEpiGroups;  // activation rows of one epilogue group
    static constexpr int kWarps = kEpiWarp0 + 4 * kEpiGroups;
    static constexpr int kThreads = 32 * kWarps;
    // Per-warpgroup register budgets (setmaxnreg).  The block launches with
    // the registers of 65536 / kThreads per thread (rounded down to 8); the
    // budgets, 128 threads each, must sum within that.
    static constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;
    static constexpr int kRegsDecode = (kEpiGroups == 2) ? 72 : (kDecGroups == 3) ? 88 : 96;
    static constexpr int kRegsControl = 64;
    static constexpr int kRegsEpiFree =
        ((kWarps / 4) * kRegsLaunch - kDecGroups * kRegsDecode - kRegsControl) / kEpiGroups / 8 * 8;
    static constexpr int kRegsEpilogue = kRegsEpiFree < 248 ? kRegsEpiFree : 248;
    static_assert(kDecGroups * kRegsDecode + kRegsControl + kEpiGroups * kRegsEpilogue <=
                      (kWarps / 4) * kRegsLaunch,
                  "register split fits the launch allocation");
    // Work unit: kU consecutive sub-blocks, decoded, multiplied and scaled
    // together (one barrier handshake per unit between the roles).
    static constexpr int kU = (MT <= 96) ? 2 : 1;
    // Tensor-memory slots per unit: accumulators (kU*MT columns), A (kU*16),
    // scales (kU).  kNP units are in flight.
    static constexpr int kUnitCols = kU * (MT + kACols + 1);
    static constexpr int kNP = (kTmemCols / kUnitCols < 8) ? kTmemCols / kUnitCols : 8;
    static constexpr int kColD = 0;
    static constexpr int kColA = kNP * kU * MT;
    static constexpr int kColS = kColA + kNP * kU * kACols;
    static_assert(kColS + kNP * kU <= kTmemCols, "slots fit tensor memory");
    static_assert(kNP >= 2, "at least two units in flight");
    static_assert(kBStageSubs % kU == 0 && kSubPerBlock % kU == 0, "units tile stages and super-blocks");
    // Byte-table decode: each qs byte (two nibbles) is looked up in shared
    // memory as the fp16x2 word of the A operand.  32 copies of each of the
    // 256 entries, copy l in bank l, so a warp's 32 lookups never conflict.
    // At MT = 16 entry j starts at byte 256 j: one byte permute of the qs
    // word and the lane's offset 4l builds the whole lookup address (the
    // byte as bits 8-15), one instruction less per lookup than a shift and
    // add (measured 6-15% faster).  Larger tiles keep entries 128 bytes
    // apart and give the 32 KB saved to a deeper activation ring (measured
    // as fast or faster from MT = 32 on).
    // Activation stage slot: the staged codes (Q8_1 form: MT rows x 128 B,
    // swizzled) and the B operand of 4 sub-blocks (kBSubBytes each: one fp16
    // plane, or hi and lo planes of the prepared form).
    static constexpr int kQRawBytes = kPrep ? 0 : kQRowBytes * MT;
    static constexpr int kBSubBytes = (kPrep ? kPlanes : 1) * kChunksPerSub * MT * 16;
    static constexpr int kBSlotBytes = kQRawBytes + kBStageSubs * kBSubBytes;
    static constexpr int usage(int nw, int nb, int lut_stride) {
        const int nx0 = nb + (kNP * kU + kBStageSubs - 1) / kBStageSubs + 1;
        const int nx = kPrep ? 1 : (nx0 < 8 ? nx0 : 8);
        return nw * kWStage + 256 * lut_stride + nb * kBSlotBytes + (kPrep ? 0 : nx * kBStageSubs * MT * 4) +
               8 * (2 * nw + 2 * nb + 2 * nx + 3 * kNP + 2) + 32 + (kPrep ? 4 * MT * 4 : 0);
    }
    static constexpr int kSmemLimit = 226 * 1024;
    static constexpr bool kWideLut = MT <= 16 && usage(2, 2, 256) <= kSmemLimit;
    // Without room for even the 32 KB table (the prepared form at MT = 128)
    // the decoders use register tables (byte permutes, ~15 integer
    // instructions per 8 weights).
    static constexpr bool kLut = kWideLut || usage(2, 2, 128) <= kSmemLimit;
    static constexpr int kLutStride = kWideLut ? 256 : kLut ? 128 : 0;
    static constexpr int kLutBytes = 256 * kLutStride;
    // Ring depths before the fit.  An activation stage's slot stays busy
    // until the MMAs of its units complete, a unit or two behind the
    // decoders, so the activation ring is the deep one: 6 stages instead of
    // 3 at MT = 16 measured 11-12% faster on K ranges of 5120 and more.  A W
    // stage holds 8 units of work, so three (two from MT = 64) suffice.
    static constexpr int kNW0 = (MT <= 48) ? 3 : 2;
    static constexpr int kNB0 = (MT <= 16) ? 6 : (MT <= 32) ? 5 : (MT <= 64) ? 4 : 3;
    static constexpr int fit(bool want_nb) {
        int nw = kNW0, nb = kNB0;
        while (usage(nw, nb, kLutStride) > kSmemLimit) { if (nb > 2) --nb; else --nw; }
        return want_nb ? nb : nw;
    }
    static constexpr int kNW = fit(false);
    static constexpr int kNB = fit(true);
    static_assert(kNW >= 2 && kNB >= 2, "rings of at least two stages");
    // Activation scales: fp32 [4 sub-blocks][MT] per stage, in a ring the
    // epilogue releases (it runs behind the MMAs by up to kNP units).
    static constexpr int kNX0 = kNB + (kNP * kU + kBStageSubs - 1) / kBStageSubs + 1;
    static constexpr int kNX = kPrep ? 1 : (kNX0 < 8 ? kNX0 : 8);  // (unused by the prepared form)
    static constexpr int kXStageBytes = kBStageSubs * MT * 4;
    static constexpr int kXItems = (kBStageSubs * MT + 31) / 32;  // scales per lane and stage
    static constexpr int kOffW = 0;
    static constexpr int kOffLut = kOffW + kNW * kWStage;
    static constexpr int kOffB = kOffLut + kLutBytes;
    static constexpr int kOffX = kOffB + kNB * kBSlotBytes;
    static constexpr int kOffBar = kOffX + (kPrep ? 0 : kNX * kXStageBytes);
    // Barriers, in this order: W full / empty, code stage landed, code
    // stage consumed (its MMAs complete), scales built / consumed, and per
    // unit slot A full / MMA done / accumulators free; then drain and
    // split-K rows received.
    static constexpr int kNumBars = 2 * kNW + 2 * kNB + 2 * kNX + 3 * kNP + 2;
    static constexpr int kBarDrain = kNumBars - 2;
    static constexpr int kBarRecv = kNumBars - 1;
    __host__ __device__ static constexpr uint32_t bar_count(int i) {
        if (i < kNW) return 1;                       // w_full: producer, + tx
        if ((i -= kNW) < kNW) return kDecWarps;      // w_empty
        if ((i -= kNW) < kNB) return 1;              // q_full: producer, + tx
        if ((i -= kNB) < kNB) return 2;              // b_empty: the MMA warps' commits
        if ((i -= kNB) < kNX) return 1;              // x_full: the scale warp
        if ((i -= kNX) < kNX) return 4 * kEpiGroups; // x_empty
        if ((i -= kNX) < kNP) return 4;              // a_full: a decoder group
        if ((i -= kNP) < kNP) return 1;              // mma_done: commit
        if ((i -= kNP) < kNP) return 4 * kEpiGroups; // d_free: epilogue warps
        if ((i -= kNP) == 0) return 2;               // drain: MMA warps
        return 1;                                    // recv: expect_tx
    }
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;  // tmem base, abort flag
    static constexpr int kOffSpan = (kOffMisc + 16 + 15) / 16 * 16;  // prepared form: the span's 2^e
    // Split-K reduction.  Each rank stages its partial tile (128 rows of
    // MT fp32, kRedStride apart) in its own activation ring, which is free
    // once its last MMA has completed, and bulk-copies the rows every other
    // rank owns into that rank's W ring and byte table, which are free once
    // that rank's decoders are done: S - 1 slices of ceil(128 / S) rows.
    static constexpr int kRedStride = MT + 4;  // fp32 words per row (16-byte rows, no bank conflicts)
    static constexpr int kOffStage = kOffB;
    static constexpr int kOffRecv = kOffW;
    static_assert(kTileN * kRedStride * 4 <= kNB * kBSlotBytes, "staged partial tile fits the activation ring");
    static_assert(recv_rows_max() * kRedStride * 4 <= kOffB - kOffW, "received slices fit the W ring and table");
    static constexpr int kUsed = kOffSpan + (kPrep ? 4 * MT * 4 : 0);
    static_assert(kUsed <= usage(kNW, kNB, kLutStride), "the ring fit counts every region");
    static_assert(kUsed <= 226 * 1024, "stages fit shared memory");
    static constexpr int kSmem = (kUsed > kMinSmem) ? kUsed : kMinSmem;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kOffB % 1024 == 0 && kBSlotBytes % 1024 == 0 && kQRawBytes % 1024 == 0,
                  "128-byte-swizzled code stages start on 1024-byte boundaries");
    static_assert(kOffLut % 128 == 0 && kOffX % 16 == 0 && kOffBar % 8 == 0, "alignment");
    static_assert(kNumBars <= 96, "barriers initialised three per producer lane");
    static_assert(kRegsControl >= 56, "the MMA warps also build the B operand");
};

constexpr int kEpilogueBarrier = 1;  // named barriers 1, 2: the 4 warps of epilogue group 0, 1
__device__ volatile int g_never_abort = 0;  // an abort flag that is never set
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int MT, int WT, bool kPrep, bool kGrouped = false>
__global__ void __launch_bounds__(TcCfg<MT, WT, kPrep>::kThreads, 1)
    matmul_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const __grid_constant__ CUtensorMap tmap_q, const __half* __restrict__ ds,
                     const uint8_t* __restrict__ tc_op, int64_t M, int N, int K,
                     float* __restrict__ y, int64_t ldy, int* err, int skip_w_stage,
                     const int32_t* __restrict__ row_offsets, int G) {
    using C = TcCfg<MT, WT, kPrep>;
    constexpr int kDecGroups = C::kDecGroups, kDecWarps = C::kDecWarps;
    constexpr int kMmaWarp0 = C::kMmaWarp0, kMmaWarp1 = C::kMmaWarp1;
    constexpr int kProducerWarp = C::kProducerWarp, kTmemWarp = C::kTmemWarp, kEpiWarp0 = C::kEpiWarp0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw;
    // The layout assumes the 1024-byte alignment the declaration asks for
    // (128-byte-swizzled copies); anything else is reported, not run.
    if (smem_u32(smem_raw) & 1023u) {
        if (threadIdx.x == 0) atomicExch(err, kDevErrLayout);
        return;
    }
    const Bc bc = bc_open(err);
    if (!bc_range(bc, 0, C::kSmem, dyn_smem_bytes(), kBcTcSmem)) return;  // every CTA alike
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + C::kNW;
    uint64_t* q_full = w_empty + C::kNW;   // a code stage has landed (TMA)
    uint64_t* b_empty = q_full + C::kNB;   // its MMAs are complete (slot reusable)
    uint64_t* x_full = b_empty + C::kNB;   // a stage's activation scales are built
    uint64_t* x_empty = x_full + C::kNX;   // ... and read by the epilogue
    // a_full[p]: unit slot p holds a decoded unit (A and scale columns);
    // mma_done[p]: its MMAs are complete (accumulators readable);
    // d_free[p]: the epilogue has read the accumulators and scales, so the
    // whole slot may be reused.  Every use of slot p waits, directly or
    // through this chain, for the previous use's d_free, so none of the
    // three barriers ever runs two phases ahead of a waiter.
    uint64_t* a_full = x_empty + C::kNX;
    uint64_t* mma_done = a_full + C::kNP;
    uint64_t* d_free = mma_done + C::kNP;
    uint64_t* drain = bars + C::kBarDrain;
    uint64_t* recv_bar = bars + C::kBarRecv;  // split-K: the other ranks' slices have landed
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = gridDim.y;  // K splits = cluster size
    const uint32_t rank = (S > 1) ? cluster_ctarank() : 0;
    const int n0 = blockIdx.x * kTileN;
    const int z = blockIdx.z;  // activation tile
    // Activation rows [row_lo, row_hi) of this CTA's tile (the tile holds
    // the first MT of them).  Grouped form (kGrouped, mixture of experts, the
    // Q8_1 form, no K split): tile z of the layer is tile t of expert g, the
    // experts with rows taken in order and each covering ceil(rows / MT)
    // tiles; W is expert g's matrix (a 3D tensor map), the rows its own.
    // CTAs past the last tile return before any set-up.
    static_assert(!kGrouped || (!kPrep && WT == kWtIQ4XS), "grouped: IQ4_XS codes in the Q8_1 form");
    int gexp = 0;
    using RowT = typename std::conditional<kGrouped, int, int64_t>::type;  // M <= 32768 rows
    RowT row_lo = (RowT)z * MT, row_hi = (RowT)M;
    if constexpr (kGrouped) {
        int* grp = reinterpret_cast<int*>(smem + C::kOffMisc + 8);
        if (warp == 0) {
            griddep_wait();  // the offsets may come from the preceding grid
            int found = -1, found_t = 0, before = 0;  // tiles of the experts already passed
            for (int e0 = 0; e0 < G && found < 0; e0 += 32) {
                const int e = e0 + lane;
                int tiles = 0;
                if (e < G && bc_global(bc, row_offsets + e, 8, row_offsets, (int64_t)(G + 1) * 4, kBcTcRows)) {
                    const int lo = __ldg(row_offsets + e), hi = __ldg(row_offsets + e + 1);
                    tiles = hi > lo ? (hi - lo + MT - 1) / MT : 0;
                }
                int incl = tiles;  // inclusive prefix sum over the 32 experts
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += v;
                }
                const int zz = z - before;
                const uint32_t mask = __ballot_sync(0xffffffffu, tiles > 0 && zz >= incl - tiles && zz < incl);
                if (mask) {
                    const int src = __ffs(mask) - 1;
                    found = e0 + src;
                    found_t = __shfl_sync(0xffffffffu, zz - (incl - tiles), src);
                }
                before += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) {
                grp[0] = found;
                grp[1] = found_t;
            }
        }
        __syncthreads();
        gexp = grp[0];
        if (gexp < 0) return;  // past the layer's last tile (whole CTA; no cluster)
        row_lo = __ldg(row_offsets + gexp) + grp[1] * MT;
        row_hi = __ldg(row_offsets + gexp + 1);
        if (!bc_range(bc, row_lo, row_hi - row_lo, M, kBcTcRows)) return;  // offsets outside the rows of y
    }
    const int pairs = K / kPairK;
    const int p0 = (int)((int64_t)pairs * rank / S);
    const int p1 = (int)((int64_t)pairs * (rank + 1) / S);
    const int nsub = (p1 - p0) * kSubPerPair;
    const int nunits = nsub / C::kU;
    const int nbst = nsub / kBStageSubs;

    // W stage ps (pair index within this CTA's K range) into ring slot `slot`.
    // Stage skip_w_stage is not issued at all (a test of the bounded waits:
    // its consumers' wait runs out; -1 in every ordinary launch).
    auto load_w_stage = [&](int slot, int ps) {
        if (ps == skip_w_stage) return;
        mbar_arrive_expect_tx(&w_full[slot], C::kWStage);
#pragma unroll
        for (int b = 0; b < C::kWBoxes; ++b) {
            const int x = (p0 + ps) * (C::kWRowBytes / 4) + b * (C::kWBoxBytes / 4);
            if (!bc_tma(bc, x, 4, C::kWBoxBytes / 4, wt_row_bytes(WT, K) / 4, n0, N, kBcTcWAlign, kBcTcW)) continue;
            if constexpr (kGrouped)
                tma_load_3d(smem + C::kOffW + slot * C::kWStage + b * (kTileN * C::kWBoxBytes), &tmap_w, x, n0, gexp,
                            &w_full[slot]);
            else
                tma_load_2d(smem + C::kOffW + slot * C::kWStage + b * (kTileN * C::kWBoxBytes), &tmap_w, x, n0,
                            &w_full[slot]);
        }
    };
    if (warp == kProducerWarp) {
        // Lane i initialises barriers i, i + 32, i + 64; lane 0 then starts
        // the first W copy at once (W is read-only model state).
#pragma unroll
        for (int h = 0; h < 3; ++h) {
            const int i = lane + 32 * h;
            if (i < C::kNumBars) mbar_init(&bars[i], C::bar_count(i));
        }
        fence_barrier_init();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            *abort_flag = 0;
            prefetch_tmap(&tmap_w);
            if constexpr (!kPrep) prefetch_tmap(&tmap_q);
            load_w_stage(0, 0);
            // Split-K: this rank's rows arrive from the S - 1 other ranks.
            // Posted now, before any rank can send (sends wait for a cluster
            // barrier phase that needs this CTA's threads past set-up).
            if (S > 1) {
                const int rows = (int)(kTileN * (rank + 1) / S) - (int)(kTileN * rank / S);
                mbar_arrive_expect_tx(recv_bar, (uint32_t)((S - 1) * rows * C::kRedStride * 4));
            }
        }
    }
    if constexpr (C::kLut) {
        // Row j of the byte table: 32 copies of entry j (one per bank).
        for (int i = threadIdx.x; i < 256 * 8; i += C::kThreads) {
            const uint32_t e = f16x2_byte_entry<WT>(i >> 3);
            *reinterpret_cast<uint4*>(smem + C::kOffLut + (i >> 3) * C::kLutStride + (i & 7) * 16) =
                make_uint4(e, e, e, e);
        }
    }
    if (warp == kTmemWarp) tmem_alloc(tmem_base_ptr, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_ptr;
    // Split-K clusters use three phases of the cluster barrier, each thread
    // arriving and waiting once per phase: 0 (now) -- every rank has started;
    // 1 -- every rank's decoders are done with their W ring and byte table
    // (the other roles arrive at once); 2 -- every rank has received its
    // slices, so no copy still reads a rank's staged rows when it exits.
    if (S > 1) cluster_arrive_relaxed();
    // Let the next kernel in the stream begin its launch; it waits for this
    // grid's completion before touching anything this grid reads or writes.
    griddep_launch_dependents();

    // Activation scales (tensor-memory warp, running ahead of the epilogue
    // by up to kNX stages): d_x of each stage's four sub-blocks, fp16 in
    // ds, to fp32 [sub-block][row] for the epilogue; rows past M get 0.
    auto build_scales = [&]() {
        bool ok = true;
        const int64_t K32 = K / kSub;
        const uint32_t* ds32 = reinterpret_cast<const uint32_t*>(ds);  // {d, s} pairs
        griddep_wait();  // ds comes from the preceding grid
        for (int bs = 0; bs < nbst; ++bs) {
            const int xs = bs % C::kNX;
            const int64_t sub0 = (int64_t)p0 * kSubPerPair + (int64_t)bs * kBStageSubs;
            // Item e = 4 * row + sub-block: four consecutive lanes read one
            // row's 16 contiguous bytes.
            uint32_t dsv[C::kXItems];
#pragma unroll
            for (int k = 0; k < C::kXItems; ++k) {
                const int e = lane + 32 * k;
                const int64_t row = row_lo + e / kBStageSubs;
                const uint32_t* dp = ds32 + row * K32 + sub0 + e % kBStageSubs;
                dsv[k] = (e < kBStageSubs * MT && row < row_hi && bc_global(bc, dp, 4, ds, M * K32 * 4, kBcTcDs))
                             ? __ldg(dp)
                             : 0u;
            }
            if (ok && bs >= C::kNX)
                ok = mbar_wait(&x_empty[xs], ((bs / C::kNX) - 1) & 1, abort_flag, err, kDevErrTimeoutX);
            if (!ok) break;
            float* xr = reinterpret_cast<float*>(smem + C::kOffX + xs * C::kXStageBytes);
#pragma unroll
            for (int k = 0; k < C::kXItems; ++k) {
                const int e = lane + 32 * k;
                if (e < kBStageSubs * MT)
                    xr[(e % kBStageSubs) * MT + e / kBStageSubs] =
                        __half2float(__ushort_as_half((unsigned short)(dsv[k] & 0xFFFFu)));
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&x_full[xs]);
        }
    };

    if (warp < kDecWarps) {
        // ------------------------------------------------------------ decoders
        reg_dealloc<C::kRegsDecode>();
        const int g = warp >> 2;                // decoder group: units g, g+G, ...
        const int t = (warp & 3) * 32 + lane;   // row within the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        bool ok = true;
        // A unit is kU consecutive sub-blocks of one super-block of one W
        // stage.
        int sp = g, sphase = 0;                     // unit slot of v (v % kNP, v / kNP)
        int prev_ps = -1;                           // W stage of this group's previous unit
        for (int v = g; v < nunits; v += kDecGroups) {
            const int l0 = v * C::kU;
            const int ps = l0 / kSubPerPair, jj = l0 % kSubPerPair;
            const int wslot = ps % C::kNW;
            if (ok && ps != prev_ps)  // this group's first unit of the stage
                ok = mbar_wait(&w_full[wslot], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutW);
            prev_ps = ps;
            const uint8_t* stage = smem + C::kOffW + wslot * C::kWStage;
            uint32_t q[C::kU][4];
            float Sw[C::kU];
            if constexpr (WT == kWtIQ4XS) {
                const uint8_t* blk = stage + t * kPairBytes + (jj / kSubPerBlock) * kBlockBytes;
                const int j = jj % kSubPerBlock;
                const uint2 hdr = *reinterpret_cast<const uint2*>(blk);
                if (MT >= 80 && jj >= kSubPerBlock) {
                    // Second super-block of the stage row: its qs start at
                    // byte 144, 16-byte aligned, so one 16-byte load per
                    // sub-block (half the shared-memory wavefronts of two
                    // 8-byte loads at this row stride; measured 1-4% faster
                    // at MT = 80 and 96, no gain at smaller tiles).
#pragma unroll
                    for (int u = 0; u < C::kU; ++u) {
                        const uint4 a = *reinterpret_cast<const uint4*>(blk + 8 + 16 * (j + u));
                        q[u][0] = a.x; q[u][1] = a.y; q[u][2] = a.z; q[u][3] = a.w;
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < C::kU; ++u) {
                        const uint2 a = *reinterpret_cast<const uint2*>(blk + 8 + 16 * (j + u));
                        const uint2 b = *reinterpret_cast<const uint2*>(blk + 16 + 16 * (j + u));
                        q[u][0] = a.x; q[u][1] = a.y; q[u][2] = b.x; q[u][3] = b.y;
                    }
                }
#pragma unroll
                for (int u = 0; u < C::kU; ++u) Sw[u] = iq4xs_scale(hdr.x, hdr.y, j + u);
            } else {
                // 18-byte block jq of the stage: box jq / 8, row t (144 bytes,
                // 16-byte aligned), block jq % 8 at byte 18 * (jq % 8); its
                // five aligned words stay inside the row.
#pragma unroll
                for (int u = 0; u < C::kU; ++u) {
                    const int jq = jj + u, b = jq % kSubPerBlock;
                    const uint32_t* a = reinterpret_cast<const uint32_t*>(
                        stage + (jq / kSubPerBlock) * (kTileN * kB18GroupBytes) + t * kB18GroupBytes +
                        kB18Bytes * b - 2 * (b & 1));
                    uint32_t raw[5];
#pragma unroll
                    for (int k = 0; k < 5; ++k) raw[k] = a[k];
                    Sw[u] = b18_unpack(raw, (b & 1) != 0, q[u]);
                }
            }
            uint32_t h[C::kU][kACols];
            {
                // Byte k of word c holds elements 4c+k (low nibble) and
                // 16+4c+k (high nibble): table row = the byte (moved to the
                // low byte by one byte permute, measured faster than a
                // shift and mask).
                if constexpr (C::kWideLut) {
                    // address = table + (byte << 8) + 4 lane: one byte
                    // permute of the qs word and the lane's offset.
                    const uint32_t lut = smem_u32(smem_raw) + C::kOffLut;
                    const uint32_t lane4 = (uint32_t)lane * 4u;
#pragma unroll
                    for (int u = 0; u < C::kU; ++u)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                h[u][4 * c + k] = lds_u32(lut + __byte_perm(q[u][c], lane4, 0x5504u | (k << 4)));
                } else if constexpr (C::kLut) {
                    const uint32_t lut = smem_u32(smem + C::kOffLut) + (uint32_t)lane * 4u;
#pragma unroll
                    for (int u = 0; u < C::kU; ++u)
#pragma unroll
                        for (int c = 0; c < 4; ++c)
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                h[u][4 * c + k] = lds_u32(lut + (__byte_perm(q[u][c], 0u, 0x4440u + k) << 7));
                } else {
#pragma unroll
                    for (int u = 0; u < C::kU; ++u)
#pragma unroll
                        for (int c = 0; c < 4; ++c) decode_f16x2<WT>(q[u][c], h[u] + 4 * c);
                }
            }
            // The stage's bytes are consumed (in registers) once this warp's
            // last unit of it is decoded.
            if (v + kDecGroups >= nunits || (l0 + kDecGroups * C::kU) / kSubPerPair != ps) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&w_empty[wslot]);
            }
            if (ok && v >= C::kNP)
                ok = mbar_wait(&d_free[sp], sphase ^ 1, abort_flag, err, kDevErrTimeoutFree);
            tc_fence_after();
#pragma unroll
            for (int u = 0; u < C::kU; ++u) {
                tmem_st16(tmem + lane_off + (uint32_t)(C::kColA + (sp * C::kU + u) * kACols), h[u]);
                tmem_st1(tmem + lane_off + (uint32_t)(C::kColS + sp * C::kU + u), __float_as_uint(Sw[u]));
            }
            // Signal at once: a tensor-memory store lands within tens of
            // cycles, while holding the signal until the group's next unit
            // is decoded lengthens every slot's round trip by a decode
            // (measured: 3-11% slower, most at large MT).
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&a_full[sp]);
            sp += kDecGroups;
            while (sp >= C::kNP) { sp -= C::kNP; sphase ^= 1; }
        }
        if (S > 1) {  // phase 1: this warp's reads of the W ring and table are done
            __syncwarp();
            cluster_wait();
            cluster_arrive_release();
        }
    } else if (warp < kEpiWarp0) {
        reg_dealloc<C::kRegsControl>();
        if (S > 1) {
            cluster_wait();
            cluster_arrive_relaxed();
        }
        if (warp == kMmaWarp0 || warp == kMmaWarp1) {
            // ---------------------------------------------------------- MMA
            // Warp-uniform loop with incremental indices (the warp shares its
            // SM sub-partition's integer pipe with decoders); one elected
            // lane issues.  Warp k takes units k, k+2, ... (those of decoder
            // group k).
            constexpr uint32_t idesc = idesc_f16_m128(MT);
            const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffB + C::kQRawBytes), MT * 16, kCoreSbo);
            const int k = (warp == kMmaWarp0) ? 0 : 1;
            const int r8 = lane & 7, c = lane >> 3;
            bool ok = true;
            int sp = k, sphase = 0;
            for (int v = k, l0 = k * C::kU; v < nunits; v += 2, l0 += 2 * C::kU) {
                const int lb = l0 % kBStageSubs;  // first sub-block's position in its B stage
                const int bs = l0 / kBStageSubs, bslot = bs % C::kNB, bphase = (bs / C::kNB) & 1;
                // B operand of this unit's sub-blocks, built from the staged
                // codes (MT rows x 128 B, 128-byte swizzled: 16-byte unit u
                // of row r sits at unit u ^ (r % 8)).  Lane (r8, c) of
                // item (sub-block s, rows 8rb..8rb+7) builds chunk c of row
                // 8rb + r8 from code words c and 4 + c: the 32 lanes read 32
                // distinct banks and store 4 x 128 contiguous bytes.
                if (ok) ok = mbar_wait(&q_full[bslot], bphase, abort_flag, err, kDevErrTimeoutQ);
                if (!kPrep && ok) {
                    const uint8_t* raw = smem + C::kOffB + bslot * C::kBSlotBytes;
                    uint8_t* bop = smem + C::kOffB + bslot * C::kBSlotBytes + C::kQRawBytes;
#pragma unroll 4
                    for (int wi = 0; wi < C::kU * (MT / 8); ++wi) {
                        const int s = lb + wi / (MT / 8), r = (wi % (MT / 8)) * 8 + r8;
                        const uint8_t* row = raw + r * kQRowBytes + 4 * c;
                        const uint32_t lo4 = *reinterpret_cast<const uint32_t*>(row + (((2 * s) ^ r8) << 4));
                        const uint32_t hi4 = *reinterpret_cast<const uint32_t*>(row + (((2 * s + 1) ^ r8) << 4));
                        *reinterpret_cast<uint4*>(bop + s * C::kBSubBytes + c * MT * 16 + r * 16) =
                            q8x8_to_f16(lo4, hi4);
                    }
                    fence_proxy_async_smem();  // the tensor core reads what was stored
                }
                __syncwarp();
                if (ok) ok = mbar_wait(&a_full[sp], sphase, abort_flag, err, kDevErrTimeoutA);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (elect_one()) {
                    if (ok) {
                        const uint32_t boff = (uint32_t)(bslot * C::kBSlotBytes + lb * C::kBSubBytes);
                        // per K step of 16: kv*q (Q8_1 form), or kv*hi and kv*lo
                        constexpr int kPl = kPrep ? kPlanes : 1;
#pragma unroll
                        for (int u = 0; u < C::kU; ++u)
#pragma unroll
                            for (int i = 0; i < kMmaPerSub; ++i)
#pragma unroll
                                for (int pl = 0; pl < kPl; ++pl)
                                    tc_mma_f16_ta(
                                        tmem + (uint32_t)(C::kColD + (sp * C::kU + u) * MT),
                                        tmem + (uint32_t)(C::kColA + (sp * C::kU + u) * kACols + i * (kUmmaK / 2)),
                                        bdesc0 + ((boff + u * C::kBSubBytes + (pl * kChunksPerSub + 2 * i) * MT * 16) >> 4),
                                        idesc, (i | pl) != 0);
                    }
                    // Commits are made even after an abort so that every
                    // waiter's barrier still completes.
                    tc_commit(&mma_done[sp]);
                    // this warp's last unit of the B stage
                    if (lb + 2 * C::kU >= kBStageSubs) tc_commit(&b_empty[bslot]);
                }
                __syncwarp();
                sp += 2;
                if (sp >= C::kNP) { sp -= C::kNP; sphase ^= 1; }
            }
            if (elect_one()) tc_commit(drain);
            __syncwarp();
        } else if (warp == kProducerWarp) {
            if (lane == 0) {
                // ------------------------------------------------- producer
                // The first W stage was started during set-up, before the
                // preceding kernel (which produces the activations) has
                // finished.  The other stages follow once it has landed, so
                // that at launch, when every CTA requests at once, first
                // stages are served first.
                auto load_q_stage = [&](int slot, int bs) {
                    if constexpr (kPrep) {
                        // one contiguous bulk copy of the stage's hi / lo planes
                        const int64_t sub0 = (int64_t)p0 * kSubPerPair + (int64_t)bs * kBStageSubs;
                        const uint8_t* src = tc_op + ((int64_t)z * (K / kSub) + sub0) * C::kBSubBytes;
                        mbar_arrive_expect_tx(&q_full[slot], C::kBSlotBytes);
                        if (bc_global_async(bc, src, C::kBSlotBytes, tc_op, tc_qh_bytes(M, K), kBcTcOp))
                            bulk_load(smem + C::kOffB + slot * C::kBSlotBytes, src, C::kBSlotBytes, &q_full[slot]);
                    } else {
                        const int x = (p0 * kSubPerPair + bs * kBStageSubs) * kSub;
                        mbar_arrive_expect_tx(&q_full[slot], C::kQRawBytes);
                        if (bc_tma(bc, x, 1, kBStageSubs * kSub, K, row_lo, M, kBcTcQAlign, kBcTcQ))
                            tma_load_2d(smem + C::kOffB + slot * C::kBSlotBytes, &tmap_q, x, (int)row_lo,
                                        &q_full[slot]);
                    }
                };
                // At most three activation stages go out before the W stages
                // after the first (when every CTA requests at once, the first
                // units' operands are served first); the rest follow in the
                // loop, into slots that need no wait.
                constexpr int kFirstQ = (C::kNB < 3) ? C::kNB : 3;
                int issued_w = 1, issued_q = 0;
                bool ok = true;
                const int pre = (C::kNW < (p1 - p0)) ? C::kNW : (p1 - p0);
                griddep_wait();  // the codes come from the preceding grid
                for (int bs = 0; bs < kFirstQ && bs < nbst; ++bs) {
                    load_q_stage(bs, bs);
                    ++issued_q;
                }
                if (pre > 1) ok = mbar_wait(&w_full[0], 0, abort_flag, err, kDevErrTimeoutW);
                for (int ps = 1; ps < pre && ok; ++ps) {
                    load_w_stage(ps, ps);
                    ++issued_w;
                }
                for (int bs = issued_q; bs < nbst && ok; ++bs) {
                    if (bs % kBStagesPerW == 0) {
                        const int ps = bs / kBStagesPerW;
                        if (ps >= pre) {
                            const int slot = ps % C::kNW;
                            ok = mbar_wait(&w_empty[slot], ((ps / C::kNW) - 1) & 1, abort_flag, err,
                                           kDevErrTimeoutW);
                            if (!ok) break;
                            load_w_stage(slot, ps);
                            ++issued_w;
                        }
                    }
                    // The slot's previous stage is consumed: its MMAs are
                    // complete, so its codes have been read too.
                    const int slot = bs % C::kNB;
                    ok = mbar_wait(&b_empty[slot], ((bs / C::kNB) - 1) & 1, abort_flag, err, kDevErrTimeoutB);
                    if (!ok) break;
                    load_q_stage(slot, bs);
                    ++issued_q;
                }
                // Drain: the last copies issued into each ring slot have
                // landed (earlier ones were consumed before their slot was
                // reused).  These waits do not stop on an abort (bounded all
                // the same): no copy may land after the CTA exits.
                for (int ps = (issued_w > C::kNW ? issued_w - C::kNW : 0); ps < issued_w; ++ps)
                    if (ps != skip_w_stage)
                        mbar_wait(&w_full[ps % C::kNW], (ps / C::kNW) & 1, &g_never_abort, err,
                                  kDevErrTimeoutDrain);
                for (int bs = (issued_q > C::kNB ? issued_q - C::kNB : 0); bs < issued_q; ++bs)
                    mbar_wait(&q_full[bs % C::kNB], (bs / C::kNB) & 1, &g_never_abort, err,
                              kDevErrTimeoutDrain);
            }
        } else if (warp == kTmemWarp) {
            if constexpr (!kPrep) build_scales();
            // Every MMA issued has completed before tensor memory is freed
            // (the MMA warps commit this after their loops, abort or not).
            mbar_wait(drain, 0, &g_never_abort, err, kDevErrTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ epilogue
        reg_alloc<C::kRegsEpilogue>();
        if (S > 1) {
            cluster_wait();
            cluster_arrive_relaxed();
        }
        const int t = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        constexpr int kMH = C::kMH;            // activation rows of this epilogue group
        const int eg = (warp - kEpiWarp0) / 4;  // epilogue group
        const int c0 = eg * kMH;                // its first activation row (accumulator column)
        float acc[kMH];
#pragma unroll
        for (int m = 0; m < kMH; ++m) acc[m] = 0.f;
        // Scale-in of n columns from m0: Q8_1 form acc += (P * d_x) * sw (the
        // scales of four columns per shared-memory load, the same address
        // across the warp: a broadcast); prepared form acc += P * sw (d_x is
        // inside P).  Two columns per instruction.
        auto scale_in = [&](const uint32_t* r, int n, int m0, float sw, const float* xrow) {
#pragma unroll
            for (int i = 0; i < n; i += 4) {
                float2 p0 = make_float2(__uint_as_float(r[i]), __uint_as_float(r[i + 1]));
                float2 p1 = make_float2(__uint_as_float(r[i + 2]), __uint_as_float(r[i + 3]));
                if constexpr (!kPrep) {
                    const float4 d = *reinterpret_cast<const float4*>(xrow + m0 + i);
                    p0 = __fmul2_rn(p0, make_float2(d.x, d.y));
                    p1 = __fmul2_rn(p1, make_float2(d.z, d.w));
                }
                const float2 a0 = __ffma2_rn(p0, make_float2(sw, sw), make_float2(acc[m0 + i], acc[m0 + i + 1]));
                const float2 a1 = __ffma2_rn(p1, make_float2(sw, sw), make_float2(acc[m0 + i + 2], acc[m0 + i + 3]));
                acc[m0 + i] = a0.x;
                acc[m0 + i + 1] = a0.y;
                acc[m0 + i + 2] = a1.x;
                acc[m0 + i + 3] = a1.y;
            }
        };
        // Prepared form: the partial sums are kept in units of the current
        // span's 2^-e (the operand's per-row power of two, from the preceding
        // grid) and rescaled by exact powers of two where the span changes
        // (every 32 sub-blocks); the current span's scales are staged in
        // shared memory, each group's own entries by that group.
        const float* span_scale = nullptr;
        // [2][MT] the current span's 2^e (two buffers), then [2][MT] the
        // ratios old / new 2^e of a switch (two buffers)
        float* s_span = reinterpret_cast<float*>(smem + C::kOffSpan) + c0;
        int cur_span = (p0 * kSubPerPair) / kSubPerSpan;
        const int last_span = (p1 * kSubPerPair - 1) / kSubPerSpan;
        float cur_e = 1.f, next_e = 1.f;  // thread t < kMH: its column's 2^e, this span and the next
        int nswitch = 0;
        if constexpr (kPrep) {
            griddep_wait();
            span_scale = reinterpret_cast<const float*>(tc_op + tc_qh_bytes(M, K)) +
                         (int64_t)z * tc_num_spans(K) * MT + c0;
            if (t < kMH) {
                const void* sbase = tc_op + tc_qh_bytes(M, K);
                const int64_t sext = tc_operand_total_bytes(M, K) - tc_qh_bytes(M, K);
                const float* sp0 = span_scale + (int64_t)cur_span * MT + t;
                if (bc_global(bc, sp0, 4, sbase, sext, kBcTcSpan)) cur_e = *sp0;
                if (cur_span < last_span && bc_global(bc, sp0 + MT, 4, sbase, sext, kBcTcSpan)) next_e = sp0[MT];
                s_span[t] = cur_e;
            }
            named_barrier_sync(kEpilogueBarrier + eg, kTileN);
        }
        bool ok = true;
        int sp = 0, sphase = 0;
        for (int v = 0; v < nunits; ++v) {
            const int l0 = v * C::kU, bs = l0 / kBStageSubs, jj = l0 % kBStageSubs, xs = bs % C::kNX;
            if constexpr (kPrep) {
                const int span = (p0 * kSubPerPair + l0) / kSubPerSpan;
                if (span != cur_span) {  // span == cur_span + 1
                    // The new span's 2^e was loaded a span ahead (a load at
                    // the switch itself stalled the epilogue ~1,700 cycles,
                    // measured).  Thread t publishes its column's ratio, an
                    // exact power of two, and the new 2^e, each in the
                    // buffer of this switch's parity: a thread reads switch
                    // k's buffers between barriers k and k + 1, and the
                    // buffers are rewritten at switch k + 2, so one barrier
                    // per switch suffices.
                    float* ratio = s_span + (2 + (nswitch & 1)) * MT;
                    if (t < kMH) {
                        ratio[t] = cur_e / next_e;
                        cur_e = next_e;
                        s_span[((nswitch + 1) & 1) * MT + t] = cur_e;
                        if (span < last_span) next_e = span_scale[(int64_t)(span + 1) * MT + t];
                    }
                    named_barrier_sync(kEpilogueBarrier + eg, kTileN);
                    const float4* f = reinterpret_cast<const float4*>(ratio);
#pragma unroll
                    for (int m = 0; m < kMH; m += 4) {
                        const float4 a = f[m / 4];
                        acc[m] *= a.x;
                        acc[m + 1] *= a.y;
                        acc[m + 2] *= a.z;
                        acc[m + 3] *= a.w;
                    }
                    ++nswitch;
                    cur_span = span;
                }
            } else if (ok && jj == 0) {  // the stage's scales
                ok = mbar_wait(&x_full[xs], (bs / C::kNX) & 1, abort_flag, err, kDevErrTimeoutX);
            }
            if (ok) ok = mbar_wait(&mma_done[sp], sphase, abort_flag, err, kDevErrTimeoutMma);
            tc_fence_after();
            const uint32_t dcol = tmem + lane_off + (uint32_t)(C::kColD + sp * C::kU * MT + c0);
            const uint32_t scol = tmem + lane_off + (uint32_t)(C::kColS + sp * C::kU);
            const float* xst = reinterpret_cast<const float*>(smem + C::kOffX + xs * C::kXStageBytes) + c0;
            uint32_t swb[C::kU];
            if constexpr (C::kEpiGroups == 1) {
                // this group's columns of both sub-blocks are contiguous
                constexpr int kCols = C::kU * MT;
                static_assert(kCols <= 64, "one load per unit");
                uint32_t r[kCols];
                if constexpr (C::kU == 2) {
                    if constexpr (kCols == 64) tmem_ld64_s2_wait(dcol, scol, r, swb);
                    else tmem_ld32_s2_wait(dcol, scol, r, swb);
                } else {
                    if constexpr (kCols == 64) tmem_ld64_s1_wait(dcol, scol, r, swb);
                    else if constexpr (kCols == 32) tmem_ld32_s1_wait(dcol, scol, r, swb);
                    else tmem_ld16_s1_wait(dcol, scol, r, swb);
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&d_free[sp]);
#pragma unroll
                for (int u = 0; u < C::kU; ++u)
                    scale_in(r + u * MT, MT, 0, __uint_as_float(swb[u]), xst + (jj + u) * MT);
            } else {
                // kMH columns of each sub-block u, at u * MT + c0, in at most
                // two loads (the first with the scale columns)
                constexpr int kP0 = (kMH <= 40) ? kMH : 32;
                constexpr int kP1 = kMH - kP0;
                static_assert(kP1 == 0 || kP1 == 16 || kP1 == 24 || kP1 == 32, "load widths");
#pragma unroll
                for (int u = 0; u < C::kU; ++u) {
                    const uint32_t col = dcol + (uint32_t)(u * MT);
                    const float* xrow = xst + (jj + u) * MT;
                    {
                        uint32_t r[kP0];
                        if (u == 0) tmem_ld_cols_wait<kP0, C::kU>(col, scol, r, swb);
                        else tmem_ld_cols_wait<kP0, 0>(col, scol, r, swb);
                        if (kP1 == 0 && u == C::kU - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&d_free[sp]);
                        }
                        scale_in(r, kP0, 0, __uint_as_float(swb[u]), xrow);
                    }
                    if constexpr (kP1 > 0) {
                        uint32_t r[kP1 > 0 ? kP1 : 1];
                        tmem_ld_cols_wait<kP1, 0>(col + kP0, scol, r, swb);
                        if (u == C::kU - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&d_free[sp]);
                        }
                        scale_in(r, kP1, kP0, __uint_as_float(swb[u]), xrow);
                    }
                }
            }
            if (!kPrep && jj + C::kU >= kBStageSubs) {  // the stage's last unit: its scales are read
                __syncwarp();
                if (lane == 0) mbar_arrive(&x_empty[xs]);
            }
            if (++sp == C::kNP) { sp = 0; sphase ^= 1; }
        }
        if constexpr (kPrep) {  // back to true units: times the last span's 2^e (exact)
            // (written before the last barrier this thread passed)
            const float4* f = reinterpret_cast<const float4*>(s_span + (nswitch & 1) * MT);
#pragma unroll
            for (int m = 0; m < kMH; m += 4) {
                const float4 a = f[m / 4];
                acc[m] *= a.x;
                acc[m + 1] *= a.y;
                acc[m + 2] *= a.z;
                acc[m + 3] *= a.w;
            }
        }
        // Partial tile -> y (one CTA), or staged in this CTA's activation
        // ring (free: every MMA has completed) for the split-K reduction.
        const int64_t mrows = row_hi - row_lo;
        if (S == 1) {
            griddep_wait();
#pragma unroll
            for (int m = 0; m < kMH; ++m)
                if (c0 + m < mrows && n0 + t < N &&
                    bc_global(bc, y + (row_lo + c0 + m) * ldy + n0 + t, 4, y, ((M - 1) * ldy + N) * 4, kBcTcY))
                    y[(row_lo + c0 + m) * ldy + n0 + t] = acc[m];
        } else {
            float* st = reinterpret_cast<float*>(smem + C::kOffStage) + t * C::kRedStride + c0;
#pragma unroll
            for (int m = 0; m < kMH; m += 4)
                *reinterpret_cast<float4*>(st + m) = make_float4(acc[m], acc[m + 1], acc[m + 2], acc[m + 3]);
            fence_proxy_async_smem();  // the staged rows are read by bulk copies
        }
    }

    if (S > 1) {
        // Split-K reduction.  Rank r owns rows [128 r / S, 128 (r + 1) / S)
        // of the tile.  Once every rank's decoders are done (phase 1), one
        // thread of each rank bulk-copies the staged rows every other rank
        // owns into that rank's W ring (slot of sender q: q, or q - 1 past
        // the owner), completing on the owner's recv barrier.  The owner
        // then sums its rows over the S slices in rank order (deterministic)
        // and writes them; decoder and epilogue warps share the sums.
        __syncthreads();  // staged rows written
        __syncwarp();
        cluster_wait();   // phase 1
        const int cap = (kTileN + S - 1) / S;
        if (warp == kEpiWarp0 && lane == 0) {
            const uint32_t stage0 = smem_u32(smem + C::kOffStage);
            const uint32_t recv0 = smem_u32(smem + C::kOffRecv);
            const int slot_base = (int)rank;
            for (int q = 0; q < S; ++q) {
                if (q == (int)rank) continue;
                const int q0 = kTileN * q / S, q1 = kTileN * (q + 1) / S;
                const int slot = slot_base < q ? slot_base : slot_base - 1;
                // the slice inside this CTA's staging area and the owner's receive area
                if (!bc_range(bc, (int64_t)q1 * C::kRedStride * 4, 0, (int64_t)C::kNB * C::kBSlotBytes, kBcTcRecv) ||
                    !bc_range(bc, (int64_t)slot * cap * C::kRedStride * 4, (int64_t)(q1 - q0) * C::kRedStride * 4,
                              (int64_t)(C::kOffB - C::kOffRecv), kBcTcRecv))
                    continue;
                bulk_copy_to_rank(recv0 + (uint32_t)(slot * cap * C::kRedStride * 4),
                                  stage0 + (uint32_t)(q0 * C::kRedStride * 4),
                                  (uint32_t)((q1 - q0) * C::kRedStride * 4), smem_u32(recv_bar), (uint32_t)q);
            }
        }
        // Every rank sends its slices whatever its state, so this wait does
        // not stop early on an abort (bounded all the same): no copy may
        // land in this CTA's shared memory after it exits.
        mbar_wait(recv_bar, 0, &g_never_abort, err, kDevErrTimeoutRecv);
        __syncwarp();
        cluster_arrive_relaxed();  // phase 2: this rank's slices have landed
        if (warp < kDecWarps || warp >= kEpiWarp0) {
            griddep_wait();
            const int idx = (warp < kDecWarps) ? threadIdx.x : threadIdx.x - (kEpiWarp0 - kDecWarps) * 32;
            const int64_t mrows = row_hi - row_lo;
            const float* stg = reinterpret_cast<const float*>(smem + C::kOffStage);
            const float* recv = reinterpret_cast<const float*>(smem + C::kOffRecv);
            const int r0 = (int)(kTileN * rank / S), r1 = (int)(kTileN * (rank + 1) / S);
            const int rows = r1 - r0;
            // element e = (row, 4 columns); consecutive threads take
            // consecutive rows, so the stores to y coalesce
            for (int e = idx; e < rows * (MT / 4); e += (kDecWarps + 4 * C::kEpiGroups) * 32) {
                const int lr = e % rows, m = 4 * (e / rows);
                float4 sum = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int q = 0; q < S; ++q) {
                    const float* src = (q == (int)rank)
                                           ? stg + (r0 + lr) * C::kRedStride
                                           : recv + ((q < (int)rank ? q : q - 1) * cap + lr) * C::kRedStride;
                    const float4 v = *reinterpret_cast<const float4*>(src + m);
                    if (q == 0) {
                        sum = v;
                    } else {
                        sum.x += v.x;
                        sum.y += v.y;
                        sum.z += v.z;
                        sum.w += v.w;
                    }
                }
                const int row = r0 + lr;
                // rows m .. last of y (the checked build checks the first and the last)
                const int64_t y_ext = ((M - 1) * ldy + N) * 4, last = (m + 3 < mrows) ? m + 3 : mrows - 1;
                if (n0 + row < N && m < mrows &&
                    bc_global(bc, y + (row_lo + m) * ldy + n0 + row, 4, y, y_ext, kBcTcY) &&
                    bc_global(bc, y + (row_lo + last) * ldy + n0 + row, 4, y, y_ext, kBcTcY)) {
                    float* yp = y + (row_lo + m) * ldy + n0 + row;
                    if (m < mrows) yp[0] = sum.x;
                    if (m + 1 < mrows) yp[ldy] = sum.y;
                    if (m + 2 < mrows) yp[2 * ldy] = sum.z;
                    if (m + 3 < mrows) yp[3 * ldy] = sum.w;
                }
            }
        }
        __syncwarp();
        cluster_wait();  // phase 2: no copy still reads this CTA's staged rows
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kTmemWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// K splits per tile (= cluster size): the S in 1..kMaxCluster (and at most
// the K pairs) with the least modelled time
//     waves(S) x (F + ceil(pairs / S)),
// in units of one K pair's streaming time per CTA.  A wave is as many
// clusters as the device runs at once for this kernel and cluster size
// (cudaOccupancyMaxActiveClusters, queried once per device and S; clusters
// stay inside one GPC, so on GB300 at most 152 / 76 / 46 / 36 / 28 / 23 /
// 15 / 15 clusters of 1..8 run at once -- the query agrees with a probe of
// CTA start times).  F is a CTA's fixed cost (launch ramp, first W stage,
// reduction), ~4.5 us on GB300 against 2.4 / 4.6 / 6.7 us per pair at
// MT = 16 / 64 / 96.  Ties keep the smaller split.  Examples: 48 row tiles
// take S = 2 (one wave) instead of S = 3 (48 clusters of 3 need two waves):
// 27.2 -> 18.4 us at 6144 x 5120, M = 16; 96 tiles stay at S = 1.
// `fallback` (the largest split that fits one wave on the SM count) stands
// if a query fails.
template <int MT, int WT, bool kPrep>
int choose_split(int dev, int fallback, int units, int pairs) {
    using C = TcCfg<MT, WT, kPrep>;
    constexpr double kFixed = MT <= 32 ? 1.9 : (MT <= 64 ? 1.1 : 0.66);
    static int max_clusters[64][kMaxCluster + 1] = {};  // per instantiation
    if (dev < 0 || dev >= 64) return fallback;
    int best = fallback;
    double best_t = 0.0;
    for (int s = 1; s <= kMaxCluster && s <= pairs; ++s) {
        int& mc = max_clusters[dev][s];
        if (mc == 0) {
            cudaLaunchConfig_t q = {};
            q.gridDim = dim3(1, (unsigned)s, 1);
            q.blockDim = dim3(C::kThreads);
            q.dynamicSmemBytes = C::kSmem;
            cudaLaunchAttribute a[1];
            a[0].id = cudaLaunchAttributeClusterDimension;
            a[0].val.clusterDim.x = 1;
            a[0].val.clusterDim.y = (unsigned)s;
            a[0].val.clusterDim.z = 1;
            q.attrs = a;
            q.numAttrs = 1;
            int n = 0;
            if (cudaOccupancyMaxActiveClusters(&n, matmul_tc_kernel<MT, WT, kPrep>, &q) != cudaSuccess ||
                n < 1) {
                cudaGetLastError();
                n = -1;
            }
            mc = n;
        }
        if (mc < 1) return fallback;
        const int waves = (units + mc - 1) / mc;
        const double t = waves * (kFixed + (double)((pairs + s - 1) / s));
        if (s == 1 || t < best_t * 0.999) {
            best = s;
            best_t = t;
        }
    }
    return best;
}

// Grouped launch of the <MT> Q8_1-form kernel: grid (row tiles, 1, tiles)
// with `tiles` an upper bound of the layer's expert tiles.
template <int MT>
cudaError_t launch_grouped_mt(const CUtensorMap& tmap_w, const CUtensorMap& tmap_q, const __half* ds,
                              const int32_t* row_offsets, int G, int64_t total_rows, int N, int K, float* y,
                              int64_t ldy, int* err, int ntiles, int tiles, cudaStream_t stream) {
    using C = TcCfg<MT, kWtIQ4XS, false>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(matmul_tc_kernel<MT, kWtIQ4XS, false, true>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles, 1, (unsigned)tiles);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matmul_tc_kernel<MT, kWtIQ4XS, false, true>, tmap_w, tmap_q, ds,
                              static_cast<const uint8_t*>(nullptr), total_rows, N, K, y, ldy, err, -1, row_offsets,
                              G);
}

template <int MT, int WT, bool kPrep>
cudaError_t launch_mt(const CUtensorMap& tmap_w, const CUtensorMap& tmap_q, const __half* ds,
                      const uint8_t* op, int64_t M, int N, int K, float* y, int64_t ldy, int* err, int S,
                      int ntiles, int mtiles, int skip, cudaStream_t stream) {
    using C = TcCfg<MT, WT, kPrep>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(matmul_tc_kernel<MT, WT, kPrep>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    S = choose_split<MT, WT, kPrep>(dev, S, ntiles * mtiles, K / kPairK);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles, (unsigned)S, (unsigned)mtiles);
    cfg.blockDim = dim3(C::kThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, matmul_tc_kernel<MT, WT, kPrep>, tmap_w, tmap_q, ds, op, M, N, K, y,
                              ldy, err, skip, static_cast<const int32_t*>(nullptr), 0);
}

template <int WT, bool kPrep>
cudaError_t launch_wt(const CUtensorMap& tw, const CUtensorMap& tq, const __half* ds, const uint8_t* op,
                      int64_t M, int N, int K, float* y, int64_t ldy, int* err, int S, int ntiles,
                      int mtiles, int skip, cudaStream_t stream) {
#define IQ4XS_TC_CASE(mt)                                                                           \
    case mt:                                                                                        \
        return launch_mt<mt, WT, kPrep>(tw, tq, ds, op, M, N, K, y, ldy, err, S, ntiles, mtiles, skip, \
                                        stream);
    switch (tc_mtile(M)) {
        IQ4XS_TC_CASE(16)
        IQ4XS_TC_CASE(32)
        IQ4XS_TC_CASE(48)
        IQ4XS_TC_CASE(64)
        IQ4XS_TC_CASE(80)
        IQ4XS_TC_CASE(96)
        IQ4XS_TC_CASE(112)
        IQ4XS_TC_CASE(128)
        default: return cudaErrorInvalidValue;
    }
#undef IQ4XS_TC_CASE
}

template <int WT>
cudaError_t launch_form(const CUtensorMap& tw, const CUtensorMap& tq, const __half* ds, const uint8_t* op,
                        int64_t M, int N, int K, float* y, int64_t ldy, int* err, int S, int ntiles,
                        int mtiles, int skip, cudaStream_t stream) {
    if (op) return launch_wt<WT, true>(tw, tq, ds, op, M, N, K, y, ldy, err, S, ntiles, mtiles, skip, stream);
    return launch_wt<WT, false>(tw, tq, ds, op, M, N, K, y, ldy, err, S, ntiles, mtiles, skip, stream);
}

}  // namespace

cudaError_t launch_matmul_tc(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs,
                             const void* ds, const void* tc_operand, int64_t M, float* y,
                             int64_t ldy, void* encode, int* err, int num_sms, int skip_w_stage,
                             cudaStream_t stream) {
    if (wt != kWtIQ4XS && wt != kWtQ4_0 && wt != kWtIQ4NL) return cudaErrorInvalidValue;
    const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(encode);
    const int64_t row_bytes = wt_row_bytes(wt, K);
    // W: one TMA box = 128 rows x (two super-blocks, or eight 18-byte blocks)
    const int box_bytes = (wt == kWtIQ4XS) ? kPairBytes : kB18GroupBytes;
    CUtensorMap tmap_w;
    {
        const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
        const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 4), (cuuint32_t)kTileN};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // Q8_1 codes: one TMA box = MT rows x 128 codes (4 sub-blocks), 128-byte
    // swizzle (conflict-free reads when the B operand is built); rows past M
    // read as 0.  The prepared form does not read them (the W map stands in).
    const int MT = tc_mtile(M);
    CUtensorMap tmap_q = tmap_w;
    if (!tc_operand) {
        const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
        const cuuint64_t gstride[1] = {(cuuint64_t)K};
        const cuuint32_t box[2] = {(cuuint32_t)kQRowBytes, (cuuint32_t)MT};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(qs), gdim, gstride, box,
                estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }

    const int mtiles = (int)tc_num_mtiles(M);
    const int ntiles = (int)((N + kTileN - 1) / kTileN);
    const int pairs = (int)(K / kPairK);
    int S = num_sms / (ntiles * mtiles);
    if (S > kMaxCluster) S = kMaxCluster;
    if (S > pairs) S = pairs;
    if (S < 1) S = 1;
    const __half* dsh = reinterpret_cast<const __half*>(ds);
    const int Ni = (int)N, Ki = (int)K;
    const int skip = skip_w_stage;
    const uint8_t* op = reinterpret_cast<const uint8_t*>(tc_operand);
    if (wt == kWtQ4_0)
        return launch_form<kWtQ4_0>(tmap_w, tmap_q, dsh, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, skip,
                                    stream);
    if (wt == kWtIQ4NL)
        return launch_form<kWtIQ4NL>(tmap_w, tmap_q, dsh, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, skip,
                                     stream);
    return launch_form<kWtIQ4XS>(tmap_w, tmap_q, dsh, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, skip,
                                 stream);
}

cudaError_t launch_matmul_tc_grouped(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                                     const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                     int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                     cudaStream_t stream) {
    const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(encode);
    const int64_t row_bytes = wt_row_bytes(kWtIQ4XS, K);
    // W of expert g: a 3D map (row words x rows x experts, expert_stride
    // bytes apart), one box = 128 rows x one super-block pair of one expert.
    CUtensorMap tmap_w;
    {
        const cuuint64_t gdim[3] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N, (cuuint64_t)G};
        const cuuint64_t gstride[2] = {(cuuint64_t)row_bytes, (cuuint64_t)expert_stride};
        const cuuint32_t box[3] = {(cuuint32_t)(kPairBytes / 4), (cuuint32_t)kTileN, 1};
        const cuuint32_t estride[3] = {1, 1, 1};
        if (enc(&tmap_w, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // at most min(G, rows) experts have rows; the tile height from the mean
    // rows per such expert
    const int64_t slots = G < total_rows ? G : total_rows;
    const int64_t mean = (total_rows + slots - 1) / slots;
    const int MT = tc_mtile(mean);
    CUtensorMap tmap_q;
    {
        const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)total_rows};
        const cuuint64_t gstride[1] = {(cuuint64_t)K};
        const cuuint32_t box[2] = {(cuuint32_t)kQRowBytes, (cuuint32_t)MT};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&tmap_q, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(qs), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    // an expert with r rows takes ceil(r / MT) <= r / MT + 1 tiles
    const int64_t tiles = (total_rows + MT - 1) / MT + slots;
    if (tiles > 65535) return cudaErrorInvalidValue;
    const int ntiles = (int)((N + kTileN - 1) / kTileN);
    const __half* dsh = reinterpret_cast<const __half*>(ds);
    const int Ni = (int)N, Ki = (int)K, Gi = (int)G, Ti = (int)tiles;
#define IQ4XS_TC_G(mt)                                                                                     \
    case mt:                                                                                              \
        return launch_grouped_mt<mt>(tmap_w, tmap_q, dsh, row_offsets, Gi, total_rows, Ni, Ki, y, ldy, err, \
                                     ntiles, Ti, stream);
    switch (MT) {
        IQ4XS_TC_G(16)
        IQ4XS_TC_G(32)
        IQ4XS_TC_G(48)
        IQ4XS_TC_G(64)
        IQ4XS_TC_G(80)
        IQ4XS_TC_G(96)
        IQ4XS_TC_G(112)
        IQ4XS_TC_G(128)
        default: return cudaErrorInvalidValue;
    }
#undef IQ4XS_TC_G
}

}  // namespace iq4xs
