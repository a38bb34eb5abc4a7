// matmul_tc.cu -- IQ4_XS x Q8_1 matmul on the 5th-generation tensor cores.
//
// Method (V100TPS engine page, new-kernel table and the tile-geometry passage
// after it): per 32-weight sub-block, a dot product of decoded codebook
// values with Q8_1 codes, scaled by d_w*(ls-32)*d_x into fp32.
//
// GB300 design.  sm_103a has no integer tcgen05 kind, so the operands travel
// as fp16: the codebook values kv (exact), and each activation's q*d_x as an
// exact pair of fp16 values hi + lo (written by the quantizer).  Per K step
// of 16 two MMAs accumulate kv*hi and kv*lo into the fp32 TMEM accumulator:
// every product is exact (at most 8 + 11 significant bits), so a sub-block's
// result d_x*sum(kv*q) differs from the exact one only by fp32 accumulation
// rounding, and the epilogue needs no activation scale (one fp32 FMA per
// element with d_w*(ls-32)).  One CTA owns 128 weight rows (= 128 TMEM lanes
// = UMMA M) and an activation tile of MT rows (= UMMA N); K is split over a
// cluster whose CTAs reduce their partial tiles through distributed shared
// memory.
//
// Warp-specialized roles, each a loop over the CTA's units of kU sub-blocks,
// decoupled by mbarrier rings (kNP slots of tensor memory: the decoded A
// operand, 16 columns per sub-block; the accumulators, MT columns per
// sub-block; the row scales, one column per sub-block).  Warp numbers below
// are for two decoder groups (MT > 16); at MT = 16 a third group takes warps
// 8-11 and the others move up by four:
//   warps 0-7 (decoders)   G groups of four; group g takes units g, g+G,
//                          ....  Warp w decodes rows 32(w%4)..+31 from
//                          the staged W bytes to exact fp16 (one shared-
//                          memory table lookup per qs byte for MT <= 96)
//                          and stores them with tcgen05.st straight into
//                          the A slot (row i in TMEM lane i), plus
//                          d_w*(ls-32) into the scale column, then arrives
//                          on the slot's a_full.
//   warps 8, 11 (MMA)      warp-uniform loops over even / odd units; one
//                          elected lane issues four tcgen05.mma 128 x MT x 16
//                          (A from tensor memory, B hi / lo planes from
//                          shared memory) per sub-block and commits.  Two
//                          issuers keep the tensor pipe fed between their
//                          own handshakes.
//   warp 9 (producer)      TMA: W stages of 512 weights per row (2D tensor
//                          map: one 128 x 272 B box of two IQ4_XS
//                          super-blocks, or two 128 x 144 B boxes of eight
//                          18-byte Q4_0 / IQ4_NL blocks each -- 144-byte rows
//                          keep the decoders' shared-memory reads at 4-way
//                          bank conflicts where 288-byte rows would be
//                          8-way); activation stages of 4 sub-blocks (one
//                          bulk copy of the pre-tiled fp16 hi / lo pairs).
//   warp 10                allocates and frees tensor memory.
//   warps 12-15 (epilogue) thread t reads row t's integer results and scale,
//                          releases the slot, and accumulates
//                          d_w*(ls-32)*(d_x*dot) in fp32 registers.
// Every mbarrier wait is bounded (2 s); a timeout sets the device error word
// and an abort flag that releases every other wait, the CTA drains its copies
// and frees its tensor memory, and the call's output is undefined.
#include <cuda.h>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kTmemCols = 512;        // whole TMEM; one CTA per SM (see kMinSmem)
constexpr int kMaxCluster = 8;
constexpr int kMinSmem = 120 * 1024;  // > half of the SM's shared memory: one CTA per SM
constexpr int kACols = kSub / 2;      // 16 TMEM columns of fp16 pairs per sub-block
constexpr int kCoreSbo = 128;         // 8 rows x 16 B core matrices, contiguous along N

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

template <int MT, int WT>
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
    // epilogue is light (small tiles).  Then one control warpgroup (MMA
    // issuers, TMA producer, tensor-memory owner) and the epilogue warpgroup.
    // Three groups at MT = 16 (more independent decode streams per SM
    // sub-partition: the decoders are latency-bound there; measured 4-11%
    // faster) and at MT = 48 (1-3% faster); at MT = 32 and MT >= 64 a third
    // group measured 9-15% slower, and a fourth at MT = 16 2% slower.
    static constexpr int kDecGroups = (MT <= 16 || MT == 48) ? 3 : 2;
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
    // Measured on GB300: 10-25% faster at MT = 48..128; at MT = 32 mixed
    // (3% slower on 4096 x 4096, 3-5% faster on larger shapes), so one group.
    static constexpr int kEpiGroups = (MT >= 48) ? 2 : 1;
    static constexpr int kMH = MT / kEpiGroups;  // activation rows of one epilogue group
    static constexpr int kThreads = 32 * (kDecWarps + 4 + 4 * kEpiGroups);
    // Per-warpgroup register budgets (setmaxnreg).  The block launches with
    // the registers of 65536 / kThreads per thread (rounded down to 8); the
    // budgets, 128 threads each, must sum within that.
    static constexpr int kRegsLaunch = (65536 / kThreads) / 8 * 8;
    static constexpr int kRegsDecode = (kEpiGroups == 2) ? ((MT >= 64 || kDecGroups == 3) ? 72 : 80) : (kDecGroups == 3) ? 88 : 96;
    static constexpr int kRegsControl = 56;
    static constexpr int kRegsEpiFree =
        ((kThreads / 128) * kRegsLaunch - kDecGroups * kRegsDecode - kRegsControl) / kEpiGroups / 8 * 8;
    static constexpr int kRegsEpilogue = kRegsEpiFree < 248 ? kRegsEpiFree : 248;
    static_assert(kDecGroups * kRegsDecode + kRegsControl + kEpiGroups * kRegsEpilogue <=
                      (kThreads / 128) * kRegsLaunch,
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
    // Byte-table decode (MT <= 96): each qs byte (two nibbles) is looked up
    // in shared memory as the fp16x2 word of the A operand, one load in
    // place of the register-table decode's integer instructions.  32
    // copies of the 256-entry table, copy l in bank l: entry j for lane l
    // at 4 * (32 * j + l), so a warp's 32 lookups never conflict.  Larger
    // tiles keep the register tables (their activation stages leave no
    // room).
    static constexpr bool kLut = MT <= 96;
    static constexpr int kLutBytes = kLut ? 256 * 32 * 4 : 0;
    static constexpr int kNW = kLut ? ((MT <= 16) ? 4 : (MT <= 48) ? 3 : (MT <= 64) ? 2 : (MT <= 80) ? 3 : 2)
                                    : ((MT <= 16) ? 5 : (MT <= 48) ? 4 : (MT <= 96) ? 3 : 2);  // W stages
    static constexpr int kNB = (MT <= 32) ? 4 : (MT <= 64) ? 3 : 2;                               // activation stages
    static constexpr int kBSubBytes = kPlanes * kChunksPerSub * MT * 16;  // hi + lo of one sub-block
    static constexpr int kBQhBytes = kBStageSubs * kBSubBytes;            // one bulk copy per stage
    static constexpr int kBStageBytes = kBQhBytes;
    static constexpr int kOffW = 0;
    static constexpr int kOffLut = kOffW + kNW * kWStage;
    static constexpr int kOffB = kOffLut + kLutBytes;
    static constexpr int kOffBar = kOffB + kNB * kBStageBytes;
    // W full/empty, B full/empty, A full / MMA done / accumulator free per
    // unit slot, drain, split-K rows received
    static constexpr int kNumBars = 2 * kNW + 2 * kNB + 3 * kNP + 2;
    static constexpr int kBarDrain = 2 * kNW + 2 * kNB + 3 * kNP;
    static constexpr int kBarRecv = kBarDrain + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;   // tmem base, abort flag
    static constexpr int kOffSpan = (kOffMisc + 16 + 15) / 16 * 16;  // current span's scales (MT fp32)
    static_assert(kOffSpan % 16 == 0, "span scales are read as 16-byte vectors");
    // Split-K reduction.  Each rank stages its partial tile (128 rows of
    // MT fp32, kRedStride apart) in its own activation ring, which is free
    // once its last MMA has completed, and bulk-copies the rows every other
    // rank owns into that rank's W ring and byte table, which are free once
    // that rank's decoders are done: S - 1 slices of ceil(128 / S) rows.
    static constexpr int kRedStride = MT + 4;  // fp32 words per row (16-byte rows, no bank conflicts)
    static constexpr int kOffStage = kOffB;
    static constexpr int kOffRecv = kOffW;
    static_assert(kTileN * kRedStride * 4 <= kNB * kBStageBytes, "staged partial tile fits the activation ring");
    static_assert(recv_rows_max() * kRedStride * 4 <= kOffB - kOffW, "received slices fit the W ring and table");
    static constexpr int kUsed = kOffSpan + MT * 4;
    static_assert(kUsed <= 226 * 1024, "stages fit shared memory");
    static constexpr int kSmem = (kUsed + 1024 > kMinSmem) ? kUsed + 1024 : kMinSmem;
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kOffB % 1024 == 0 && kBStageBytes % 16 == 0 && kOffLut % 128 == 0, "alignment");
};

constexpr int kEpilogueBarrier = 1;  // named barriers 1, 2: the 4 warps of epilogue group 0, 1
__device__ volatile int g_never_abort = 0;  // an abort flag that is never set
__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int MT, int WT>
__global__ void __launch_bounds__(TcCfg<MT, WT>::kThreads, 1)
    matmul_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const uint8_t* __restrict__ tc_op, int64_t M, int N, int K,
                     float* __restrict__ y, int64_t ldy, int* err) {
    using C = TcCfg<MT, WT>;
    constexpr int kDecGroups = C::kDecGroups, kDecWarps = C::kDecWarps;
    constexpr int kMmaWarp0 = C::kMmaWarp0, kMmaWarp1 = C::kMmaWarp1;
    constexpr int kProducerWarp = C::kProducerWarp, kTmemWarp = C::kTmemWarp, kEpiWarp0 = C::kEpiWarp0;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + C::kNW;
    uint64_t* b_full = w_empty + C::kNW;
    uint64_t* b_empty = b_full + C::kNB;
    // a_full[p]: unit slot p holds a decoded unit (A and scale columns);
    // mma_done[p]: its MMAs are complete (accumulators readable);
    // d_free[p]: the epilogue has read the accumulators and scales, so the
    // whole slot may be reused.  Every use of slot p waits, directly or
    // through this chain, for the previous use's d_free, so none of the
    // three barriers ever runs two phases ahead of a waiter.
    uint64_t* a_full = b_empty + C::kNB;
    uint64_t* mma_done = a_full + C::kNP;
    uint64_t* d_free = mma_done + C::kNP;
    uint64_t* drain = d_free + C::kNP;
    uint64_t* recv_bar = bars + C::kBarRecv;  // split-K: the other ranks' slices have landed
    uint32_t* tmem_base_ptr = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int S = gridDim.y;  // K splits = cluster size
    const uint32_t rank = (S > 1) ? cluster_ctarank() : 0;
    const int n0 = blockIdx.x * kTileN;
    const int z = blockIdx.z;  // activation tile
    const int pairs = K / kPairK;
    const int p0 = (int)((int64_t)pairs * rank / S);
    const int p1 = (int)((int64_t)pairs * (rank + 1) / S);
    const int nsub = (p1 - p0) * kSubPerPair;
    const int nunits = nsub / C::kU;
    const int nbst = nsub / kBStageSubs;
    const int64_t K32 = K / kSub;
    const uint8_t* qh_tile = tc_op + (int64_t)z * K32 * C::kBSubBytes;

    static_assert(C::kNumBars <= 64, "barriers initialised two per producer lane");
    // W stage ps (pair index within this CTA's K range) into ring slot `slot`.
    auto load_w_stage = [&](int slot, int ps) {
        mbar_arrive_expect_tx(&w_full[slot], C::kWStage);
#pragma unroll
        for (int b = 0; b < C::kWBoxes; ++b)
            tma_load_2d(smem + C::kOffW + slot * C::kWStage + b * (kTileN * C::kWBoxBytes), &tmap_w,
                        (p0 + ps) * (C::kWRowBytes / 4) + b * (C::kWBoxBytes / 4), n0,
                        &w_full[slot]);
    };
    if (warp == kProducerWarp) {
        // Lane i initialises barriers i and i + 32; lane 0 then starts the
        // first W copy at once (W is read-only model state).
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            uint32_t count = 0;
            if (i < C::kNW) count = 1;                                           // w_full
            else if (i < 2 * C::kNW) count = kDecWarps;                          // w_empty
            else if (i < 2 * C::kNW + C::kNB) count = 1;                         // b_full
            else if (i < 2 * C::kNW + 2 * C::kNB) count = 2;                     // b_empty: the MMA warps' commits
            else if (i < 2 * C::kNW + 2 * C::kNB + C::kNP) count = 4;            // a_full: a decoder group
            else if (i < 2 * C::kNW + 2 * C::kNB + 2 * C::kNP) count = 1;        // mma_done
            else if (i < 2 * C::kNW + 2 * C::kNB + 3 * C::kNP) count = 4 * C::kEpiGroups;  // d_free: epilogue warps
            else if (i == C::kBarDrain) count = 2;                               // drain: MMA warps
            else if (i == C::kBarRecv) count = 1;                                // recv: expect_tx below
            if (count) mbar_init(&bars[i], count);
        }
        fence_barrier_init();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            *abort_flag = 0;
            prefetch_tmap(&tmap_w);
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
        uint4* lut = reinterpret_cast<uint4*>(smem + C::kOffLut);
        for (int i = threadIdx.x; i < 256 * 8; i += C::kThreads) {
            const uint32_t e = f16x2_byte_entry<WT>(i >> 3);
            lut[i] = make_uint4(e, e, e, e);
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
                if (C::kLut && MT >= 80 && jj >= kSubPerBlock) {
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
            if constexpr (C::kLut) {
                // Byte k of word c holds elements 4c+k (low nibble) and
                // 16+4c+k (high nibble): table row = the byte (moved to the
                // low byte by one byte permute, measured faster than a
                // shift and mask).
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
                for (int u = 0; u < C::kU; ++u) {
                    decode_f16x2<WT>(q[u][0], h[u]);
                    decode_f16x2<WT>(q[u][1], h[u] + 4);
                    decode_f16x2<WT>(q[u][2], h[u] + 8);
                    decode_f16x2<WT>(q[u][3], h[u] + 12);
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
            const uint64_t bdesc0 = smem_desc(smem_u32(smem + C::kOffB), MT * 16, kCoreSbo);
            const int k = (warp == kMmaWarp0) ? 0 : 1;
            bool ok = true;
            int sp = k, sphase = 0;
            for (int v = k, l0 = k * C::kU; v < nunits; v += 2, l0 += 2 * C::kU) {
                const int lb = l0 % kBStageSubs;  // first sub-block's position in its B stage
                const int bs = l0 / kBStageSubs, bslot = bs % C::kNB, bphase = (bs / C::kNB) & 1;
                if (ok && lb < 2 * C::kU)  // this warp's first unit of the B stage
                    ok = mbar_wait(&b_full[bslot], bphase, abort_flag, err, kDevErrTimeoutB);
                if (ok) ok = mbar_wait(&a_full[sp], sphase, abort_flag, err, kDevErrTimeoutA);
                ok = __all_sync(0xffffffffu, ok);
                tc_fence_after();
                if (elect_one()) {
                    if (ok) {
                        const uint32_t boff = (uint32_t)(bslot * C::kBStageBytes + lb * C::kBSubBytes);
#pragma unroll
                        for (int u = 0; u < C::kU; ++u)
#pragma unroll
                            for (int i = 0; i < kMmaPerSub; ++i)
#pragma unroll
                                for (int pl = 0; pl < kPlanes; ++pl)
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
        } else if (warp == kProducerWarp && lane == 0) {
            // ----------------------------------------------------- producer
            // The first W stage was started during set-up, before the
            // preceding kernel (which produces the activations) has finished.
            // The other stages follow once it has landed, so that at launch,
            // when every CTA requests at once, first stages are served first.
            int issued_w = 1, issued_b = 0;
            bool ok = true;
            const int pre = (C::kNW < (p1 - p0)) ? C::kNW : (p1 - p0);
            griddep_wait();
            for (int bs = 0; bs < C::kNB && bs < nbst; ++bs) {
                uint8_t* dst = smem + C::kOffB + bs * C::kBStageBytes;
                const int64_t sub0 = (int64_t)p0 * kSubPerPair + (int64_t)bs * kBStageSubs;
                mbar_arrive_expect_tx(&b_full[bs], C::kBQhBytes);
                bulk_load(dst, qh_tile + sub0 * C::kBSubBytes, C::kBQhBytes, &b_full[bs]);
                ++issued_b;
            }
            if (pre > 1) ok = mbar_wait(&w_full[0], 0, abort_flag, err, kDevErrTimeoutW);
            for (int ps = 1; ps < pre && ok; ++ps) {
                load_w_stage(ps, ps);
                ++issued_w;
            }
            for (int bs = issued_b; bs < nbst && ok; ++bs) {
                if (bs % (kSubPerPair / kBStageSubs) == 0) {
                    const int ps = bs / (kSubPerPair / kBStageSubs);
                    if (ps >= pre) {
                        const int slot = ps % C::kNW;
                        ok = mbar_wait(&w_empty[slot], ((ps / C::kNW) - 1) & 1, abort_flag, err,
                                       kDevErrTimeoutW);
                        if (!ok) break;
                        load_w_stage(slot, ps);
                        ++issued_w;
                    }
                }
                const int slot = bs % C::kNB;
                if (bs >= C::kNB)
                    ok = mbar_wait(&b_empty[slot], ((bs / C::kNB) - 1) & 1, abort_flag, err,
                                   kDevErrTimeoutB);
                if (!ok) break;
                uint8_t* dst = smem + C::kOffB + slot * C::kBStageBytes;
                const int64_t sub0 = (int64_t)p0 * kSubPerPair + (int64_t)bs * kBStageSubs;
                mbar_arrive_expect_tx(&b_full[slot], C::kBQhBytes);
                bulk_load(dst, qh_tile + sub0 * C::kBSubBytes, C::kBQhBytes, &b_full[slot]);
                ++issued_b;
            }
            // Drain: the last copies issued into each ring slot have landed.
            for (int ps = (issued_w > C::kNW ? issued_w - C::kNW : 0); ps < issued_w; ++ps)
                mbar_wait(&w_full[ps % C::kNW], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutDrain);
            for (int bs = (issued_b > C::kNB ? issued_b - C::kNB : 0); bs < issued_b; ++bs)
                mbar_wait(&b_full[bs % C::kNB], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutDrain);
        } else if (warp == kTmemWarp) {
            // Every MMA issued has completed before tensor memory is freed.
            mbar_wait(drain, 0, abort_flag, err, kDevErrTimeoutDrain);
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
        // Activation span scales (from the preceding grid): the partial sums
        // are kept in units of the current span's 2^-e and rescaled by exact
        // powers of two where the span changes (every 32 sub-blocks).  The
        // current span's scales are staged in shared memory, each group's
        // own entries by that group (named barrier 1 + group).
        griddep_wait();
        const float* span_scale = reinterpret_cast<const float*>(tc_op + tc_qh_bytes(M, K)) +
                                  (int64_t)z * tc_num_spans(K) * MT + c0;
        float* s_span = reinterpret_cast<float*>(smem + C::kOffSpan) + c0;
        int cur_span = (p0 * kSubPerPair) / kSubPerSpan;
        if (t < kMH) s_span[t] = span_scale[(int64_t)cur_span * MT + t];
        named_barrier_sync(kEpilogueBarrier + eg, kTileN);
        bool ok = true;
        int sp = 0, sphase = 0;
        for (int v = 0; v < nunits; ++v) {
            const int span = (p0 * kSubPerPair + v * C::kU) / kSubPerSpan;
            if (span != cur_span) {
                const float4* fo = reinterpret_cast<const float4*>(s_span);
                const float4* fn = reinterpret_cast<const float4*>(span_scale + (int64_t)span * MT);
#pragma unroll
                for (int m = 0; m < kMH; m += 4) {
                    const float4 a = fo[m / 4], b = fn[m / 4];
                    acc[m] *= a.x / b.x;
                    acc[m + 1] *= a.y / b.y;
                    acc[m + 2] *= a.z / b.z;
                    acc[m + 3] *= a.w / b.w;
                }
                named_barrier_sync(kEpilogueBarrier + eg, kTileN);  // every thread has read the old scales
                if (t < kMH) s_span[t] = span_scale[(int64_t)span * MT + t];
                named_barrier_sync(kEpilogueBarrier + eg, kTileN);
                cur_span = span;
            }
            if (ok) ok = mbar_wait(&mma_done[sp], sphase, abort_flag, err, kDevErrTimeoutMma);
            tc_fence_after();
            const uint32_t dcol = tmem + lane_off + (uint32_t)(C::kColD + sp * C::kU * MT + c0);
            const uint32_t scol = tmem + lane_off + (uint32_t)(C::kColS + sp * C::kU);
            uint32_t swb[C::kU];
            if constexpr (C::kEpiGroups == 1) {
                // this group's columns of both sub-blocks are contiguous
                constexpr int kCols = C::kU * MT;
#pragma unroll
                for (int part = 0; part < kCols; part += 64) {
                    const int w = (kCols - part < 64) ? kCols - part : 64;
                    uint32_t r[64];
                    if (part == 0) {
                        if (C::kU == 2) {
                            if (w == 64) tmem_ld64_s2_wait(dcol, scol, r, swb);
                            else if (w == 48) tmem_ld48_s2_wait(dcol, scol, r, swb);
                            else if (w == 32) tmem_ld32_s2_wait(dcol, scol, r, swb);
                            else tmem_ld16_s2_wait(dcol, scol, r, swb);
                        } else {
                            if (w == 64) tmem_ld64_s1_wait(dcol, scol, r, swb);
                            else if (w == 48) tmem_ld48_s1_wait(dcol, scol, r, swb);
                            else if (w == 32) tmem_ld32_s1_wait(dcol, scol, r, swb);
                            else tmem_ld16_s1_wait(dcol, scol, r, swb);
                        }
                    } else {
                        if (w == 64) tmem_ld64_wait(dcol + part, r);
                        else if (w == 48) tmem_ld48_wait(dcol + part, r);
                        else if (w == 32) tmem_ld32_wait(dcol + part, r);
                        else tmem_ld16_wait(dcol + part, r);
                    }
                    if (part + 64 >= kCols) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&d_free[sp]);
                    }
                    // acc[m] += (d_x * dot) * Sw, two columns per instruction; a
                    // pair of columns never straddles two sub-blocks.
#pragma unroll
                    for (int k = 0; k < 64; k += 2) {
                        if (k >= w) break;
                        const int c = part + k, u = c / MT, m = c % MT;
                        const float sw = __uint_as_float(swb[u]);
                        const float2 a = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                                    make_float2(sw, sw), make_float2(acc[m], acc[m + 1]));
                        acc[m] = a.x;
                        acc[m + 1] = a.y;
                    }
                }
            } else {
                // kMH columns of each sub-block u, at u * MT + c0, in at most
                // two loads (the first with the scale columns)
                constexpr int kP0 = (kMH <= 48) ? kMH : 32;
                constexpr int kP1 = kMH - kP0;
#pragma unroll
                for (int u = 0; u < C::kU; ++u) {
                    const uint32_t col = dcol + (uint32_t)(u * MT);
                    {
                        uint32_t r[kP0];
                        if (u == 0) tmem_ld_cols_wait<kP0, C::kU>(col, scol, r, swb);
                        else tmem_ld_cols_wait<kP0, 0>(col, scol, r, swb);
                        if (kP1 == 0 && u == C::kU - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&d_free[sp]);
                        }
                        const float sw = __uint_as_float(swb[u]);
#pragma unroll
                        for (int k = 0; k < kP0; k += 2) {
                            const float2 a = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                                        make_float2(sw, sw), make_float2(acc[k], acc[k + 1]));
                            acc[k] = a.x;
                            acc[k + 1] = a.y;
                        }
                    }
                    if constexpr (kP1 > 0) {
                        uint32_t r[kP1];
                        tmem_ld_cols_wait<kP1, 0>(col + kP0, scol, r, swb);
                        if (u == C::kU - 1) {
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) mbar_arrive(&d_free[sp]);
                        }
                        const float sw = __uint_as_float(swb[u]);
#pragma unroll
                        for (int k = 0; k < kP1; k += 2) {
                            const float2 a = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])),
                                                        make_float2(sw, sw),
                                                        make_float2(acc[kP0 + k], acc[kP0 + k + 1]));
                            acc[kP0 + k] = a.x;
                            acc[kP0 + k + 1] = a.y;
                        }
                    }
                }
            }
            if (++sp == C::kNP) { sp = 0; sphase ^= 1; }
        }
        // Back to true units: times the last span's 2^e (exact).
        {
            const float4* f = reinterpret_cast<const float4*>(s_span);
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
        const int64_t mrows = M - (int64_t)z * MT;
        if (S == 1) {
            griddep_wait();
#pragma unroll
            for (int m = 0; m < kMH; ++m)
                if (c0 + m < mrows && n0 + t < N) y[((int64_t)z * MT + c0 + m) * ldy + n0 + t] = acc[m];
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
            const int idx = (warp < kDecWarps) ? threadIdx.x : threadIdx.x - 4 * 32;
            const int64_t mrows = M - (int64_t)z * MT;
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
                if (n0 + row < N) {
                    float* yp = y + ((int64_t)z * MT + m) * ldy + n0 + row;
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
template <int MT, int WT>
int choose_split(int dev, int fallback, int units, int pairs) {
    using C = TcCfg<MT, WT>;
    constexpr double kFixed = MT <= 32 ? 1.9 : (MT <= 64 ? 1.1 : 0.66);
    static int max_clusters[64][kMaxCluster + 1] = {};
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
            if (cudaOccupancyMaxActiveClusters(&n, matmul_tc_kernel<MT, WT>, &q) != cudaSuccess ||
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

template <int MT, int WT>
cudaError_t launch_mt(const CUtensorMap& tmap, const uint8_t* tc_op, int64_t M, int N, int K,
                      float* y, int64_t ldy, int* err, int S, int ntiles, int mtiles,
                      cudaStream_t stream) {
    using C = TcCfg<MT, WT>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(matmul_tc_kernel<MT, WT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    S = choose_split<MT, WT>(dev, S, ntiles * mtiles, K / kPairK);
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
    return cudaLaunchKernelEx(&cfg, matmul_tc_kernel<MT, WT>, tmap, tc_op, M, N, K, y, ldy, err);
}

template <int WT>
cudaError_t launch_wt(const CUtensorMap& tmap, const uint8_t* op, int64_t M, int N, int K,
                      float* y, int64_t ldy, int* err, int S, int ntiles, int mtiles,
                      cudaStream_t stream) {
    switch (tc_mtile(M)) {
        case 16: return launch_mt<16, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 32: return launch_mt<32, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 48: return launch_mt<48, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 64: return launch_mt<64, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 80: return launch_mt<80, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 96: return launch_mt<96, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 112: return launch_mt<112, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        case 128: return launch_mt<128, WT>(tmap, op, M, N, K, y, ldy, err, S, ntiles, mtiles, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

cudaError_t launch_matmul_tc(const void* w, int wt, int64_t N, int64_t K, const void* tc_operand,
                             int64_t M, float* y, int64_t ldy, void* encode, int* err,
                             int num_sms, cudaStream_t stream) {
    if (wt != kWtIQ4XS && wt != kWtQ4_0 && wt != kWtIQ4NL) return cudaErrorInvalidValue;
    const int64_t row_bytes = wt_row_bytes(wt, K);
    // one TMA box: 128 rows x (two super-blocks, or eight 18-byte blocks)
    const int box_bytes = (wt == kWtIQ4XS) ? kPairBytes : kB18GroupBytes;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(box_bytes / 4), (cuuint32_t)kTileN};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = reinterpret_cast<EncodeTiledFn>(encode)(
        &tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box,
        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;

    const int mtiles = (int)tc_num_mtiles(M);
    const int ntiles = (int)((N + kTileN - 1) / kTileN);
    const int pairs = (int)(K / kPairK);
    int S = num_sms / (ntiles * mtiles);
    if (S > kMaxCluster) S = kMaxCluster;
    if (S > pairs) S = pairs;
    if (S < 1) S = 1;
    const uint8_t* op = reinterpret_cast<const uint8_t*>(tc_operand);
    const int Ni = (int)N, Ki = (int)K;
    if (wt == kWtQ4_0) return launch_wt<kWtQ4_0>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
    if (wt == kWtIQ4NL) return launch_wt<kWtIQ4NL>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
    return launch_wt<kWtIQ4XS>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
}

}  // namespace iq4xs
