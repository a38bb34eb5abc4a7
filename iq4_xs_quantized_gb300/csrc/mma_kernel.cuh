// mma_kernel.cuh -- the warp-level tensor-core MMA matmul (mma.sync
// m16n8k16, fp16 operands, fp32 accumulators held in registers) for small and
// medium batches: the kernel, its launch configurations and the launch cost
// model, shared by the IQ4_XS launches (matmul_mma.cu) and the launches for
// weights in 18-byte blocks of 32, Q4_0 and IQ4_NL (matmul_mma_b18.cu), two
// translation units that compile in parallel.
//
// Method (V100TPS engine page, new-kernel table and the tile-geometry
// passage after it): per 32-weight sub-block an integer dot product of the
// decoded codebook values with the Q8_1 codes, scaled by d_w*(ls-32)*d_x into
// fp32.  As on the tcgen05 path both operands are small integers held
// exactly in fp16 (codebook values |kv| <= 127, codes |q| <= 127), so a
// sub-block's two k16 MMAs leave its exact integer dot P in the fp32
// accumulator (every product and partial sum is an integer below 2^24).
//
// Why a warp-level MMA in the memory-bound range.  For M <= 32 the weight
// bytes bound the call; what limits a kernel is how many instructions and
// shared-memory wavefronts it spends per weight.  Here the decoded weights go
// from the byte-table lookup straight into the A fragment registers and every
// sub-block's accumulator comes back in registers for its scale-in, so no
// weight tile is stored anywhere, no accumulator is read back from tensor
// memory and no hand-off between warp roles is needed per sub-block.
//
// Weights in 18-byte blocks (Q4_0, IQ4_NL; same qs byte layout per 32
// weights, one fp16 d per block and no sub-block scale): a stage is the
// same 512 weights of a row, 288 bytes in two 144-byte TMA boxes; the row
// scale is the block's d, and the byte table holds the format's 16 values.
//
// Tiles.  A CTA owns R weight rows (R a multiple of 16 up to 256, chosen per
// call so that the row tiles times the K split fill the SMs) and an
// activation tile of 8*NT rows (MMA N = 8 per fragment, NT fragments).
// Weights are the A operand (MMA M = 16 rows per fragment).  A stage is 512
// weights of every row (two super-blocks, one R x 272 B TMA box) plus the
// matching Q8_1 codes; the 8 consumer warps split it as kRG row groups x
// kSG sub-block groups: warp (rg, sg) takes fragments rg, rg + kRG, ...
// (at most kTMax) and kSPW consecutive sub-blocks of one super-block.  K is
// split over a thread-block cluster of S CTAs whose partial tiles are summed
// in rank order through distributed shared memory.
//
// K order inside a sub-block.  MMA k pair p of k16 step s (k = 2p, 2p+1)
// holds qs byte b = 4*(p % 4) + 2*s + (p / 4), i.e. sub-block elements b
// (low nibble) and 16 + b (high nibble).  Lane (g, t) of the warp (g = lane /
// 4, t = lane % 4) then needs bytes 4t..4t+3 of its two weight rows g and
// g+8 -- one 32-bit word each -- and Q8_1 codes 4t..4t+3 and 16+4t..16+4t+3
// of activation row g, two words.  One shared-memory lookup per qs byte
// returns the fp16x2 (kv[low nibble], kv[high nibble]) that is exactly one A
// register.
//
// Roles: warps 0-7 consume stages; warp 8 lane 0 is the TMA producer (W
// boxes before the wait for the preceding grid, Q8_1 code boxes after it).
// Each consumer warp first turns the stage's block headers into its row
// scales d_w*(ls-32) and the activation scales d_x into fp32, in tables of
// its own kept in the unused half of every 256-byte row of the byte table.
// Every mbarrier wait is bounded; a wait that runs out records its code in
// the device error word, raises the CTA's abort flag, and the CTA drains its
// copies and leaves y unwritten.
#pragma once
#include <cuda.h>

#include "internal.cuh"

namespace iq4xs {

// Launch choices kept once (matmul_mma.cu) for both translation units: the
// forced test configuration (0 = none), and the measured launch for a shape
// and activation-tile height, if the calibration installed one.
void mma_forced_config(int* rows, int* splits, int* ctas_per_sm);
bool mma_measured_launch(int64_t N, int64_t K, int mt, int* rows, int* splits, int* ctas_per_sm);
// Q4_0 / IQ4_NL weights (wt) on the warp-MMA path, dense and grouped
// (matmul_mma_b18.cu).
cudaError_t launch_matmul_mma_b18(int wt, const void* w, int64_t N, int64_t K, const int8_t* qs, const void* ds,
                                  int64_t M, float* y, int64_t ldy, void* encode, int* err, int num_sms,
                                  int skip_w_stage, cudaStream_t stream);
cudaError_t launch_matmul_mma_grouped_b18(int wt, const void* w, int64_t expert_stride, int64_t G, int64_t N,
                                          int64_t K, const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                          int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                          int num_sms, int skip_w_stage, cudaStream_t stream);

namespace {


constexpr int kMmaConsumers = 8;              // consumer warps
constexpr int kMmaProducerWarp = kMmaConsumers;
constexpr int kMmaThreads = 32 * (kMmaConsumers + 1);

constexpr int kMmaMaxCluster = 8;
constexpr int kMmaMaxRows = 256;              // TMA box height
constexpr int kMmaMaxStages = 4;
constexpr int kWideLutBytes = 256 * 256;      // byte table: entry j at 256 j, copy l at 4 l (bytes 0..127)
constexpr int kGapBytes = kWideLutBytes / 2;  // bytes 128..255 of every table row
constexpr int kQBoxK = 128;                   // Q8_1 codes per box row (one 128-byte swizzle row)
constexpr int kQBoxesPerStage = kPairK / kQBoxK;  // 4
constexpr int kMmaSmemLimit = 227 * 1024;
constexpr int kOffRingMma = kWideLutBytes;
constexpr int kMmaBarBytes = 128;             // full[4], empty[4], abort flag
constexpr int kMmaSmemLimit2 = 113 * 1024;   // per CTA with two CTAs per SM
__device__ volatile int g_never_abort_mma = 0;  // an abort flag that is never set

// Physical address (bytes from the table start) of byte o of the gap space.
__host__ __device__ constexpr uint32_t gap_addr(uint32_t o) { return ((o >> 7) << 8) + 128u + (o & 127u); }

// NT: 8-row activation fragments per tile; T: 16-row weight fragments per
// consumer warp.  The 8 consumer warps are 2 row groups x 4 sub-block
// groups, so a CTA owns R = 32 T weight rows and a warp takes fragments
// rg, rg + 2, ..., rg + 2 (T - 1) and 4 consecutive sub-blocks of a stage.
// kB18: weights in 18-byte blocks of 32 (Q4_0, IQ4_NL) instead of 136-byte
// super-blocks of 256; a stage is 512 weights of a row either way (272 or
// 288 bytes).
// kPersist (the grouped form): the partial tiles and the item descriptors
// get a region of their own after the ring.
template <int NT, int T, int kOcc = 1, bool kB18 = false, bool kPersist = false>
struct MmaCfg {
    static_assert(NT >= 1 && NT <= 4, "1..4 fragments of 8 activation rows");
    static_assert(T >= 1 && T * NT <= 16, "accumulators: T x NT x 4 registers per lane");
    static constexpr int kMt = 8 * NT;                    // activation rows per tile
    static constexpr int kRG = 2;                         // row groups
    static constexpr int kSG = kMmaConsumers / kRG;       // sub-block groups
    static constexpr int kSPW = kSubPerPair / kSG;        // sub-blocks per warp and stage (4)
    static constexpr int kR = 16 * kRG * T;               // weight rows per CTA
    static_assert(kR <= kMmaMaxRows, "TMA box height");
    static_assert(kSubPerBlock % kSPW == 0, "a warp's sub-blocks lie in one super-block");
    static constexpr int kQBox = kMt * kQBoxK;            // one code box (a multiple of 1024 B)
    static constexpr int kQStage = kQBoxesPerStage * kQBox;
    static constexpr int kRowB = kB18 ? 2 * kB18GroupBytes : kPairBytes;  // W bytes of a row per stage
    static constexpr int kWBytes = (kR * kRowB + 1023) / 1024 * 1024;
    static constexpr int kStage = kWBytes + kQStage;
    static constexpr int kRedStride = kMt + 4;             // fp32 per row of a partial tile
    static constexpr int kRedBytes = kPersist ? kMmaConsumers / 2 * kR * kRedStride * 4 : 0;
    static constexpr int kExtra = kPersist ? kRedBytes + kMmaMaxStages * 16 : 0;
    // kOcc CTAs per SM: the whole shared memory (227 KB) for one, or half
    // of it (113 KB) for two -- then a launch's CTAs can start beside the
    // preceding launch's last ones.
    static_assert(kOcc == 1 || kOcc == 2, "one or two CTAs per SM");
    static constexpr int kRing =
        (kOcc == 1 ? kMmaSmemLimit : kMmaSmemLimit2) - kOffRingMma - kMmaBarBytes - kExtra;
    static constexpr int kNS = kRing / kStage < kMmaMaxStages ? kRing / kStage : kMmaMaxStages;
    static_assert(kNS >= 2, "two stages in flight");
    static constexpr int kSmem = kOffRingMma + kNS * kStage + kExtra + kMmaBarBytes;
    // Per-warp tables (gap space): row scales [k][s][g][h] (rows
    // 16 f + g + 8 h of fragment f = rg + 2 k), then d_x [s][m].
    static constexpr int kSwFloats = kSPW * T * 16;
    static constexpr int kDxFloats = kSPW * kMt;
    static constexpr int kWarpTab = ((kSwFloats + kDxFloats) * 4 + 127) / 128 * 128;
    static_assert(kMmaConsumers * kWarpTab <= kGapBytes, "tables fit the byte table's gaps");
    static constexpr int kXItems = (kDxFloats + 31) / 32;  // d_x loads per lane and stage
    static constexpr int kCombos = T * 8;                  // (fragment, g) pairs of a warp
    static_assert(kPersist || kSG * kR * kRedStride * 4 <= kNS * kStage, "partials fit the ring");
    static_assert(!kPersist || kRedBytes == kSG * kR * kRedStride * 4, "a partial tile per sub-block group");
    static_assert(kSmem <= (kOcc == 1 ? kMmaSmemLimit : kMmaSmemLimit2), "shared memory per CTA");
    static_assert(kR * kRedStride * 4 <= kWideLutBytes, "CTA tile fits the byte table");
};

__device__ __forceinline__ void mma_f16_16816(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1,
                                              const float c[4]) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%10, %11, %12, %13};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
          "f"(c[3]));
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t local_addr, uint32_t rank) {
    uint32_t a;
    float4 v;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(local_addr), "r"(rank));
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a)
                 : "memory");
    return v;
}
__device__ __forceinline__ void consumers_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kMmaConsumers) : "memory");
}
// consumers_sync that also returns whether v held in any consumer thread.
__device__ __forceinline__ bool consumers_any(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.or.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "n"(32 * kMmaConsumers)
        : "memory");
    return r != 0;
}
// kGrouped: mixture-of-experts form, persistent.  The layer's work items
// are, for each expert with rows (in expert order; rows from row_offsets, a
// device array read after the wait for the preceding grid), each R-row tile
// of its W and each kMt-row tile of its activation rows (the activation
// tile varying fastest, so that CTAs working at once share a W tile in L2);
// CTA c takes items c, c + gridDim.x, ...  One pass over K per item, no K
// split.  The producer warp walks the experts once, 32 at a time, and runs
// ahead across items: each item's descriptor goes into a small ring in
// shared memory before its first stage is issued, and an empty stage after
// the last item tells the consumers to stop.  The partial tiles of the
// sub-block groups have a region of their own, so the next item's stages
// stream in while the consumers sum the current one.  Otherwise grid z is
// the activation tile of rows [z kMt, (z + 1) kMt) and grid (x, y) the
// weight-row tile and the K range.
template <int NT, int T, int kOcc, bool kGrouped, bool kB18 = false>
__global__ void __launch_bounds__(kMmaThreads, kOcc)
    matmul_mma_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_q,
                      const __half* __restrict__ ds, int64_t M, int N, int K, float* __restrict__ y, int64_t ldy,
                      int* err, const int32_t* __restrict__ row_offsets, int G, int wt, int skip_stage) {
    using C = MmaCfg<NT, T, kOcc, kB18, kGrouped>;
    constexpr int kTMax = T, kMt = C::kMt, kSPW = C::kSPW, kRG = C::kRG, R = C::kR, NS = C::kNS;
    extern __shared__ __align__(1024) uint8_t smem[];
    if (smem_u32(smem) & 1023u) {  // the 128-byte-swizzled code boxes need 1024-byte alignment
        if (threadIdx.x == 0) atomicExch(err, kDevErrLayout);
        return;
    }
    constexpr int stage_b = C::kStage, wbytes = C::kWBytes;
    const Bc bc = bc_open(err);
    if (!bc_range(bc, 0, C::kSmem, dyn_smem_bytes(), kBcMmaSmem)) return;  // every CTA alike
    uint8_t* extra = smem + kOffRingMma + NS * stage_b;  // grouped: partial tiles, then descriptors
    uint64_t* full = reinterpret_cast<uint64_t*>(extra + C::kExtra);
    uint64_t* empty = full + kMmaMaxStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + kMmaMaxStages);
    int4* desc = reinterpret_cast<int4*>(extra + C::kRedBytes);  // grouped: {expert, n0, first row, end row}
    const uint32_t sbase = smem_u32(smem);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = gridDim.y;
    const uint32_t rank = (S > 1) ? cluster_ctarank() : 0;
    const int n0 = blockIdx.x * R;  // dense form
    const int z = blockIdx.z;
    const int pairs = (K + kPairK - 1) / kPairK;
    const int p0 = (int)((int64_t)pairs * rank / S);
    const int p1 = (int)((int64_t)pairs * (rank + 1) / S);
    const int nst = p1 - p0;
    // dense form: activation rows [row_lo, row_hi)
    const int64_t row_lo = (int64_t)z * kMt, row_hi = (row_lo + kMt < M) ? row_lo + kMt : M;

    // Stage gs of the current item: K pair p0 + gs % nst (grouped: items of
    // nst stages one after the other), weight rows from n0w, activation rows
    // from rq, expert e.  Stage skip_stage (a test of the bounded waits; -1
    // in every ordinary call) is not issued: its barrier never completes.
    auto load_w = [&](int gs, int n0w, int e) {
        if (gs == skip_stage) return;
        const int slot = gs % NS;
        uint8_t* dst = smem + kOffRingMma + slot * stage_b;
        const int x = (p0 + gs % nst) * (C::kRowB / 4);
        if (!bc_tma(bc, x, 4, C::kRowB / 4, (int64_t)(K / kPairK) * (C::kRowB / 4), n0w, N, kBcMmaWAlign, kBcMmaW))
            return;
        if constexpr (kGrouped) bc_range(bc, e, 1, G, kBcMmaW);
        mbar_arrive_expect_tx(&full[slot], (uint32_t)(R * C::kRowB + C::kQStage));
        if constexpr (kGrouped && kB18) {
            tma_load_3d(dst, &tmap_w, x, n0w, e, &full[slot]);
            tma_load_3d(dst + R * kB18GroupBytes, &tmap_w, x + kB18GroupBytes / 4, n0w, e, &full[slot]);
        } else if constexpr (kGrouped) {
            tma_load_3d(dst, &tmap_w, x, n0w, e, &full[slot]);
        } else if constexpr (kB18) {
            // two boxes of R rows x 144 B (eight 18-byte blocks each), one
            // after the other: 144-byte rows put the 8 rows a warp reads at
            // once on distinct banks, where 288-byte rows would not
            tma_load_2d(dst, &tmap_w, x, n0w, &full[slot]);
            tma_load_2d(dst + R * kB18GroupBytes, &tmap_w, x + kB18GroupBytes / 4, n0w, &full[slot]);
        } else {
            tma_load_2d(dst, &tmap_w, x, n0w, &full[slot]);
        }
    };
    auto load_q = [&](int gs, int64_t rq64) {
        if (gs == skip_stage) return;
        const int slot = gs % NS;
        const int rq = (int)rq64;
#pragma unroll
        for (int b = 0; b < kQBoxesPerStage; ++b) {
            const int x = (p0 + gs % nst) * kPairK + b * kQBoxK;
            if (bc_tma(bc, x, 1, kQBoxK, K, rq, M, kBcMmaQAlign, kBcMmaQ))
                tma_load_2d(smem + kOffRingMma + slot * stage_b + wbytes + b * C::kQBox, &tmap_q, x, rq, &full[slot]);
        }
    };
    const int pre = nst < NS ? nst : NS;  // dense form: stages issued at set-up
    if (warp == kMmaProducerWarp && lane == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kMmaConsumers);
        }
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
        prefetch_tmap(&tmap_w);
        prefetch_tmap(&tmap_q);
        // Dense form: the first W stages (model state) go out at once, before
        // the byte table is built and before the preceding grid (which
        // writes the codes) has finished.
        if constexpr (!kGrouped)
            for (int ps = 0; ps < pre; ++ps) load_w(ps, n0, 0);
    }
    // Byte table: row j = 32 copies (one per bank) of the fp16x2 word
    // (kv[j & 15], kv[j >> 4]) in its first 128 bytes.
    for (int i = threadIdx.x; i < 256 * 8; i += kMmaThreads) {
        const uint32_t e = !kB18 ? f16x2_byte_entry<kWtIQ4XS>(i >> 3)
                           : (wt == kWtQ4_0 ? f16x2_byte_entry<kWtQ4_0>(i >> 3) : f16x2_byte_entry<kWtIQ4NL>(i >> 3));
        *reinterpret_cast<uint4*>(smem + (i >> 3) * 256 + (i & 7) * 16) = make_uint4(e, e, e, e);
    }
    __syncthreads();
    griddep_launch_dependents();

    bool ok = true;
    if (warp == kMmaProducerWarp) {
        int issued = 0;
        bool ended = false;  // grouped: the empty stage after the last item was posted
        if constexpr (!kGrouped) {
            if (lane == 0) {
                griddep_wait();  // the codes come from the preceding grid
                for (int ps = 0; ps < pre; ++ps) load_q(ps, row_lo);
                issued = pre;
                for (int gs = pre; gs < nst && ok; ++gs) {
                    const int slot = gs % NS;
                    if (gs >= NS) {
                        ok = mbar_wait(&empty[slot], ((gs / NS) - 1) & 1, abort_flag, err, kDevErrTimeoutMmaSlot);
                        if (!ok) break;
                    }
                    load_w(gs, n0, 0);
                    load_q(gs, row_lo);
                    ++issued;
                }
            }
            __syncwarp();
        } else {
            griddep_wait();  // the offsets and the codes come from the preceding grid
            const int64_t ntx = (N + R - 1) / R;
            // The expert cursor: experts [e0, e0 + 32) held one per lane (rows
            // [lo, hi), items cnt, inclusive prefix incl within the 32), base =
            // items of the experts before e0.
            int e0 = 0, lo = 0, hi = 0;
            int64_t base = 0, cnt = 0, incl = 0, tot = 0;
            bool have = false;
            int64_t item = blockIdx.x;
            for (int k = 0;; ++k, item += gridDim.x) {
                bool done = false;
                for (;;) {
                    if (!have) {
                        if (e0 >= G) {
                            done = true;
                            break;
                        }
                        const int e = e0 + lane;
                        const bool in = e < G && bc_global(bc, row_offsets + e, 8, row_offsets,
                                                           (int64_t)(G + 1) * 4, kBcMmaOffsets);
                        lo = in ? __ldg(row_offsets + e) : 0;
                        hi = in ? __ldg(row_offsets + e + 1) : 0;
                        // offsets outside the rows of y: the expert is skipped
                        if (hi > lo && !bc_range(bc, lo, (int64_t)hi - lo, M, kBcMmaRows)) hi = lo;
                        cnt = hi > lo ? ntx * ((hi - lo + kMt - 1) / kMt) : 0;
                        incl = cnt;
#pragma unroll
                        for (int o = 1; o < 32; o <<= 1) {
                            const int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
                            if (lane >= o) incl += v;
                        }
                        tot = __shfl_sync(0xffffffffu, incl, 31);
                        have = true;
                    }
                    if (item < base + tot) break;
                    base += tot;
                    e0 += 32;
                    have = false;
                }
                int4 d = make_int4(-1, 0, 0, 0);
                if (!done) {
                    const int f = __ffs(__ballot_sync(0xffffffffu, base + incl > item)) - 1;
                    const int lo_f = __shfl_sync(0xffffffffu, lo, f), hi_f = __shfl_sync(0xffffffffu, hi, f);
                    const int64_t j = item - base - __shfl_sync(0xffffffffu, incl - cnt, f);
                    const int64_t tiles = (hi_f - lo_f + kMt - 1) / kMt;
                    const int tr = (int)(j % tiles);
                    const int r0 = lo_f + kMt * tr;
                    d = make_int4(e0 + f, (int)(j / tiles) * R, r0, r0 + kMt < hi_f ? r0 + kMt : hi_f);
                }
                if (lane == 0) {
                    // Item k's stages are gs0 .. gs0 + nst - 1.  Its descriptor
                    // slot was last read when the consumers started item
                    // k - kMmaMaxStages, before they released stage gs0 - NS.
                    const int gs0 = k * nst;
                    for (int ps = 0; ps < nst && ok; ++ps) {
                        const int gs = gs0 + ps, slot = gs % NS;
                        if (gs >= NS) {
                            ok = mbar_wait(&empty[slot], ((gs / NS) - 1) & 1, abort_flag, err,
                                           kDevErrTimeoutMmaSlot);
                            if (!ok) break;
                        }
                        if (ps == 0) desc[k % kMmaMaxStages] = d;  // published by the stage's arrival
                        if (d.x < 0) {
                            mbar_arrive(&full[slot]);  // no more items: an empty stage
                            ended = true;
                            break;
                        }
                        load_w(gs, d.y, d.x);
                        load_q(gs, d.z);
                        ++issued;
                    }
                }
                ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
                if (done || !ok) break;
            }
        }
        if (lane == 0) {
            // Drain: the last stage issued into each slot has landed (the
            // earlier ones were consumed before their slot was reused; so
            // was stage issued - NS once the empty stage took its slot).  Not
            // stopped by an abort: no copy may land after the CTA exits.
            const int first = issued - NS + (ended ? 1 : 0);
            for (int gs = (first > 0 ? first : 0); gs < issued; ++gs)
                if (gs != skip_stage)
                    mbar_wait(&full[gs % NS], (gs / NS) & 1, &g_never_abort_mma, err, kDevErrTimeoutDrain);
        }
        __syncwarp();
    } else {
        // ---------------------------------------------------------- consumers
        const int g = lane >> 2, t = lane & 3;
        const int rg = warp / C::kSG, sg = warp % C::kSG;
        const int sub_w = sg * kSPW;             // first sub-block of the stage this warp takes
        const int super_w = sub_w / kSubPerBlock;
        const int jj0 = sub_w % kSubPerBlock;
        const uint32_t lane4 = (uint32_t)lane * 4u;
        const uint32_t tab = (uint32_t)(warp * C::kWarpTab);   // this warp's tables, gap space
        const uint32_t* ds32 = reinterpret_cast<const uint32_t*>(ds);
        const int64_t K32 = (K + kSub - 1) / kSub;
        float acc[kTMax][NT][4];
        // Activation scales of K pair `pair` for this warp's sub-blocks: item
        // e = (row m = rb + e / kSPW, sub-block e % kSPW), fp16 d in ds; rows
        // from rhi on read as 0.
        uint32_t dxv[C::kXItems];
        auto load_dx = [&](int64_t rb, int64_t rhi, int pair) {
#pragma unroll
            for (int k = 0; k < C::kXItems; ++k) {
                const int e = lane + 32 * k;
                const int64_t m = rb + e / kSPW;
                const int64_t sub = (int64_t)pair * kSubPerPair + sub_w + e % kSPW;
                dxv[k] = (e < C::kDxFloats && m < rhi && sub < K32 &&
                          bc_global(bc, ds32 + m * K32 + sub, 4, ds, M * K32 * 4, kBcMmaDs))
                             ? __ldg(ds32 + m * K32 + sub)
                             : 0u;
            }
        };
        griddep_wait();  // ds comes from the preceding grid
        // Row-scale work of this lane: (fragment slot k, g) pairs c = lane +
        // 32 i, rows 16 f + g and 16 f + g + 8, all kSPW sub-blocks.
        const int wrow_lane = 16 * rg + g;       // row of fragment slot 0 for this lane (+ 16 kRG k)
        auto zero_acc = [&]() {
#pragma unroll
            for (int i = 0; i < kTMax; ++i)
#pragma unroll
                for (int f = 0; f < NT; ++f)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[i][f][e] = 0.f;
        };
        // Stage gs (landed) of an item with activation rows [rb, rhi): this
        // warp's tables, then its MMAs; the activation scales of K pair
        // next_pair of the same item (if >= 0) are requested meanwhile.
        auto consume = [&](int gs, int64_t rb, int64_t rhi, int next_pair) {
            const int slot = gs % NS;
            // Plain loads from here on: ordered after the barrier wait (an
            // asm statement with a memory clobber) and free to be scheduled
            // among themselves.
            const uint8_t* wst = smem + kOffRingMma + slot * stage_b;
            const uint8_t* qst = wst + wbytes;
            // ---- per-stage tables: row scales and activation scales
            // Row scales of this warp's kSPW = 4 consecutive sub-blocks
            // jj0..jj0+3 of one super-block: from the header's 16 bits of
            // low nibbles and 8 bits of high pairs shifted once, each
            // ls - 32 comes out exact through the float 2^23 + ls.  In
            // 18-byte blocks: block jj0 + u's own fp16 d, in box super_w.
            static_assert(kSPW == 4, "four sub-blocks per header read");
#pragma unroll
            for (int c = lane; c < C::kCombos; c += 32) {
                const int k = c >> 3, gg = c & 7;
                const int r = 16 * (rg + kRG * k) + gg;
                float sw[2][4];
                if constexpr (kB18) {
                    const uint8_t* bx = wst + super_w * (R * kB18GroupBytes) + kB18Bytes * jj0;
#pragma unroll
                    for (int h = 0; h < 2; ++h)
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            sw[h][u] = __half2float(*reinterpret_cast<const __half*>(
                                bx + (r + 8 * h) * kB18GroupBytes + kB18Bytes * u));
                } else {
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint2 hd =
                        *reinterpret_cast<const uint2*>(wst + (r + 8 * h) * kPairBytes + super_w * kBlockBytes);
                    const float d = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
                    const uint32_t lo16 = hd.y >> (4 * jj0);          // ls low nibbles of jj0..jj0+3
                    const uint32_t hi8 = hd.x >> (16 + 2 * jj0);      // ls high bit pairs
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const uint32_t ls = ((lo16 >> (4 * u)) & 0xFu) | (((hi8 >> (2 * u)) & 3u) << 4);
                        const float l = __uint_as_float(0x4B000000u | ls) - 8388640.0f;  // ls - 32, exact
                        sw[h][u] = d * l;
                    }
                }
                }
                // block (k, s2) of 64 bytes at gap offset 64 (4 k + s2): two
                // 128-byte chunks per k, entries (rows r, r + 8) at +8 gg
                uint8_t* tk = smem + gap_addr(tab + (uint32_t)(256 * k)) + 8 * gg;
#pragma unroll
                for (int s2 = 0; s2 < 4; ++s2)
                    *reinterpret_cast<float2*>(tk + 256 * (s2 >> 1) + 64 * (s2 & 1)) = make_float2(sw[0][s2], sw[1][s2]);
            }
#pragma unroll
            for (int k = 0; k < C::kXItems; ++k) {
                const int e = lane + 32 * k;
                if (e < C::kDxFloats)
                    *reinterpret_cast<float*>(smem + gap_addr(tab + (uint32_t)((C::kSwFloats + (e % kSPW) * kMt + e / kSPW) * 4))) =
                        __half2float(__ushort_as_half((unsigned short)(dxv[k] & 0xFFFFu)));
            }
            __syncwarp();
            if (next_pair >= 0) load_dx(rb, rhi, next_pair);  // in flight during this stage
            // The four sub-blocks unrolled (loads of the next sub-block's words
            // overlap this one's lookups and MMAs: 5-6 % faster at 8 rows,
            // 6-14 % at 16) where the registers allow it: one activation
            // fragment, or two with at most four weight fragments per warp
            // (not in the grouped form, which spills there); one at a time
            // otherwise.
            constexpr int kUnrollS = (NT == 1 || (NT == 2 && T <= 4 && !kGrouped)) ? kSPW : 1;
#pragma unroll kUnrollS
            for (int s = 0; s < kSPW; ++s) {
                const int j = sub_w + s;                 // sub-block within the stage
                const int jj = j % kSubPerBlock;
                const int box = j / 4, jq = j % 4;
                // B fragments: activation row 8 f + g, Q8_1 codes 4t..4t+3 and
                // 16+4t..16+4t+3 of the sub-block (128-byte swizzle: 16-byte
                // chunk c of box row r sits at chunk c ^ (r % 8)).
                uint32_t bfr[NT][4];
                float2 dx[NT];
#pragma unroll
                for (int f = 0; f < NT; ++f) {
                    const uint8_t* rowa = qst + box * C::kQBox + (8 * f + g) * kQBoxK + 4 * t;
                    const uint32_t lo4 = *reinterpret_cast<const uint32_t*>(rowa + (((2 * jq) ^ g) << 4));
                    const uint32_t hi4 = *reinterpret_cast<const uint32_t*>(rowa + (((2 * jq + 1) ^ g) << 4));
                    const uint4 v = q8x8_to_f16(lo4, hi4);
                    bfr[f][0] = v.x; bfr[f][1] = v.y; bfr[f][2] = v.z; bfr[f][3] = v.w;
                    dx[f] = *reinterpret_cast<const float2*>(
                        smem + gap_addr(tab + (uint32_t)((C::kSwFloats + s * kMt + 8 * f + 2 * t) * 4)));
                }
                // row scales of sub-block s: block (k, s) of 64 bytes at gap
                // offset 64 (k kSPW + s), the lane's pair (rows g, g+8) at +8 g;
                // kSPW = 4 blocks are two whole 128-byte gap chunks, so block
                // (k, s) sits 512 k physical bytes after block (0, s).
                static_assert(kSPW == 4, "two gap chunks per fragment slot");
                const uint8_t* swp = smem + gap_addr(tab + (uint32_t)(64 * s)) + 8 * g;
                // This lane's qs word (bytes 4t..4t+3 of the sub-block) of row
                // wrow_lane: in 18-byte blocks, block jj of box super_w,
                // whose codes start 2 bytes in (odd blocks: on a 4-byte
                // boundary; even ones: 2 bytes past it, so the word is
                // shifted out of the two aligned words around it).
                constexpr int kRowStride = kB18 ? kB18GroupBytes : kPairBytes;
                const uint8_t* wl =
                    kB18 ? wst + super_w * (R * kB18GroupBytes) + wrow_lane * kB18GroupBytes + kB18Bytes * jj + 2 + 4 * t
                         : wst + wrow_lane * kPairBytes + super_w * kBlockBytes + 8 + 16 * jj + 4 * t;
                static_assert(kSPW % 2 == 0, "sub-block parity = parity of s");
                auto word_at = [&](const uint8_t* p) -> uint32_t {
                    if (!kB18 || (s & 1)) return *reinterpret_cast<const uint32_t*>(p);
                    const uint32_t* a = reinterpret_cast<const uint32_t*>(p - 2);
                    return __funnelshift_r(a[0], a[1], 16);
                };
#pragma unroll
                for (int k = 0; k < kTMax; ++k) {
                    {
                        const uint8_t* wk = wl + 16 * kRG * k * kRowStride;
                        const uint32_t w0 = word_at(wk);
                        const uint32_t w1 = word_at(wk + 8 * kRowStride);
                        // A fragments of k16 steps 0 and 1: bytes (0, 1) and
                        // (2, 3) of the two rows' words; table byte offset =
                        // (byte << 8) | 4 lane.
                        uint32_t a0[4], a1[4];
                        a0[0] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w0, lane4, 0x5504u));
                        a0[1] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w1, lane4, 0x5504u));
                        a0[2] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w0, lane4, 0x5514u));
                        a0[3] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w1, lane4, 0x5514u));
                        a1[0] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w0, lane4, 0x5524u));
                        a1[1] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w1, lane4, 0x5524u));
                        a1[2] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w0, lane4, 0x5534u));
                        a1[3] = *reinterpret_cast<const uint32_t*>(smem + __byte_perm(w1, lane4, 0x5534u));
                        const float2 sw = *reinterpret_cast<const float2*>(swp + 512 * k);
                        const float zero[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int f = 0; f < NT; ++f) {
                            float p[4];
                            mma_f16_16816(p, a0, bfr[f][0], bfr[f][1], zero);
                            mma_f16_16816(p, a1, bfr[f][2], bfr[f][3], p);
                            // acc += (P * d_x) * d_w*(ls-32): rows g (p0, p1) and g+8 (p2, p3)
                            const float2 q01 = __fmul2_rn(make_float2(p[0], p[1]), dx[f]);
                            const float2 q23 = __fmul2_rn(make_float2(p[2], p[3]), dx[f]);
                            const float2 r01 =
                                __ffma2_rn(q01, make_float2(sw.x, sw.x), make_float2(acc[k][f][0], acc[k][f][1]));
                            const float2 r23 =
                                __ffma2_rn(q23, make_float2(sw.y, sw.y), make_float2(acc[k][f][2], acc[k][f][3]));
                            acc[k][f][0] = r01.x; acc[k][f][1] = r01.y;
                            acc[k][f][2] = r23.x; acc[k][f][3] = r23.y;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        };
        // The partial tiles of the sub-block groups into red, then (after a
        // barrier) their sum into y rows [rb, rhi), columns n0i.. (or, with a
        // K split, into this CTA's tile for the cluster's reduction).
        auto store_partials = [&](float* red) {
            red += sg * R * C::kRedStride;
#pragma unroll
            for (int k = 0; k < kTMax; ++k) {
#pragma unroll
                for (int f = 0; f < NT; ++f) {
                    const int r = 16 * (rg + kRG * k) + g, c = 8 * f + 2 * t;
                    *reinterpret_cast<float2*>(red + r * C::kRedStride + c) = make_float2(acc[k][f][0], acc[k][f][1]);
                    *reinterpret_cast<float2*>(red + (r + 8) * C::kRedStride + c) =
                        make_float2(acc[k][f][2], acc[k][f][3]);
                }
            }
        };
        auto sum_partials = [&](const float* red, int64_t rb, int64_t rhi, int n0i) {
            float* tile = reinterpret_cast<float*>(smem);
            const int64_t mrows = rhi - rb;
            for (int e = threadIdx.x; e < R * kMt; e += 32 * kMmaConsumers) {
                const int r = e % R, m = e / R;
                float v = red[r * C::kRedStride + m];
#pragma unroll
                for (int q = 1; q < C::kSG; ++q) v += red[(q * R + r) * C::kRedStride + m];
                if (S == 1) {
                    if (m < mrows && n0i + r < N &&
                        bc_global(bc, y + (rb + m) * ldy + n0i + r, 4, y, ((M - 1) * ldy + N) * 4, kBcMmaY))
                        y[(rb + m) * ldy + n0i + r] = v;
                } else {
                    tile[r * C::kRedStride + m] = v;
                }
            }
        };
        if constexpr (!kGrouped) {
            if (nst > 0) load_dx(row_lo, row_hi, p0);
            zero_acc();
            for (int ps = 0; ps < nst && ok; ++ps) {
                ok = mbar_wait(&full[ps % NS], (ps / NS) & 1, abort_flag, err, kDevErrTimeoutMmaStage);
                if (!ok) break;
                consume(ps, row_lo, row_hi, ps + 1 < nst ? p0 + ps + 1 : -1);
            }
            if (!ok) {
                // Wake the producer if it waits on a slot this warp will never free.
                if (lane == 0) *abort_flag = 1;
            }
            // ---- end of the K range: partial tiles of the sub-block groups
            float* red = reinterpret_cast<float*>(smem + kOffRingMma);
            consumers_sync();  // every consumer is done with the ring
            if (!*abort_flag) store_partials(red);
            consumers_sync();
            if (!*abort_flag) sum_partials(red, row_lo, row_hi, n0);
        } else {
            float* red = reinterpret_cast<float*>(extra);
            bool failed = false;
            for (int k = 0;; ++k) {
                const int gs0 = k * nst;
                ok = mbar_wait(&full[gs0 % NS], (gs0 / NS) & 1, abort_flag, err, kDevErrTimeoutMmaStage);
                const int4 d = ok ? desc[k % kMmaMaxStages] : make_int4(-1, 0, 0, 0);
                // Every consumer warp leaves together: after the last item, or
                // when a wait of any of them ran out.
                failed = consumers_any(!ok);
                if (failed || d.x < 0) break;
                load_dx(d.z, d.w, p0);
                zero_acc();
                for (int ps = 0; ps < nst && ok; ++ps) {
                    const int gs = gs0 + ps;
                    if (ps > 0) {
                        ok = mbar_wait(&full[gs % NS], (gs / NS) & 1, abort_flag, err, kDevErrTimeoutMmaStage);
                        if (!ok) break;
                    }
                    consume(gs, d.z, d.w, ps + 1 < nst ? p0 + ps + 1 : -1);
                }
                failed = consumers_any(!ok);  // and every consumer is done with this item's stages
                if (failed) break;
                store_partials(red);
                consumers_sync();
                sum_partials(red, d.z, d.w, d.y);
            }
            if (failed && threadIdx.x == 0) *abort_flag = 1;  // the producer stops issuing
        }
    }

    if (S > 1) {
        // Split-K: rank r sums rows [R r / S, R (r + 1) / S) of every rank's
        // tile in rank order (deterministic).  Every thread of every CTA
        // passes both cluster barriers, aborted or not; after an abort the
        // output is undefined and the tiles are not summed.
        __syncwarp();
        cluster_arrive_release();
        cluster_wait();
        if (warp < kMmaConsumers && !*abort_flag) {
            // Four activation rows of one weight row per item: the S ranks'
            // 16-byte slices are all requested before any is summed.
            const int r0 = R * (int)rank / S, r1 = R * ((int)rank + 1) / S;
            const int64_t mrows = row_hi - row_lo;  // one tile (K splits only without experts)
            for (int e = threadIdx.x; e < (r1 - r0) * (kMt / 4); e += 32 * kMmaConsumers) {
                const int r = r0 + e % (r1 - r0), m = 4 * (e / (r1 - r0));
                const uint32_t off = sbase + (uint32_t)((r * C::kRedStride + m) * 4);
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (bc_range(bc, (r * C::kRedStride + m) * 4, 16, R * C::kRedStride * 4, kBcMmaSplit)) {
                    float4 part[kMmaMaxCluster];
#pragma unroll
                    for (int q = 0; q < kMmaMaxCluster; ++q)
                        if (q < S) part[q] = ld_cluster_f32x4(off, (uint32_t)q);
#pragma unroll
                    for (int q = 0; q < kMmaMaxCluster; ++q)
                        if (q < S) {
                            v.x += part[q].x;
                            v.y += part[q].y;
                            v.z += part[q].z;
                            v.w += part[q].w;
                        }
                }
                const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if (m + i < mrows && n0 + r < N &&
                        bc_global(bc, y + (row_lo + m + i) * ldy + n0 + r, 4, y, ((M - 1) * ldy + N) * 4, kBcMmaY))
                        y[(row_lo + m + i) * ldy + n0 + r] = vv[i];
            }
        }
        __syncwarp();
        cluster_arrive_release();
        cluster_wait();  // no rank exits while another reads its tile
    }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The kernel's dynamic shared-memory limit, raised once per device.
template <int NT, int T, int kOcc, bool kGrouped, bool kB18 = false>
cudaError_t mma_smem_attr(int dev) {
    static bool done[64] = {};
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(matmul_mma_kernel<NT, T, kOcc, kGrouped, kB18>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               MmaCfg<NT, T, kOcc, kB18, kGrouped>::kSmem);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

// Cached per device: clusters of S (1..8) the device runs at once for the
// kernel <NT, T, kOcc, kB18> (cudaOccupancyMaxActiveClusters, queried once).
template <int NT, int T, int kOcc, bool kB18 = false>
int mma_max_clusters(int dev, int s, int num_sms) {
    using C = MmaCfg<NT, T, kOcc, kB18>;
    static int cache[64][kMmaMaxCluster + 1] = {};
    int mc = (dev >= 0 && dev < 64) ? cache[dev][s] : 0;
    if (mc > 0) return mc;
    if (mma_smem_attr<NT, T, kOcc, false, kB18>(dev) != cudaSuccess) cudaGetLastError();
    cudaLaunchConfig_t q = {};
    q.gridDim = dim3(1, (unsigned)s, 1);
    q.blockDim = dim3(kMmaThreads);
    q.dynamicSmemBytes = C::kSmem;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 1;
    at[0].val.clusterDim.y = (unsigned)s;
    at[0].val.clusterDim.z = 1;
    q.attrs = at;
    q.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, matmul_mma_kernel<NT, T, kOcc, false, kB18>, &q) != cudaSuccess ||
        n < 1) {
        cudaGetLastError();
        n = kOcc * num_sms / s;
    }
    mc = n > 0 ? n : 1;
    if (dev >= 0 && dev < 64) cache[dev][s] = mc;
    return mc;
}

template <int NT, int T, int kOcc, bool kB18 = false>
cudaError_t launch_nt(const void* w, int64_t row_bytes, EncodeTiledFn enc, const CUtensorMap& tq, const __half* ds,
                      int64_t M, int N, int K, int S, float* y, int64_t ldy, int* err, int wt, int skip_stage,
                      cudaStream_t stream) {
    using C = MmaCfg<NT, T, kOcc, kB18>;
    int dev = 0;
    cudaGetDevice(&dev);
    const cudaError_t ea = mma_smem_attr<NT, T, kOcc, false, kB18>(dev);
    if (ea != cudaSuccess) return ea;
    // W: one box = R rows x one super-block pair (272 B), or R rows x eight
    // 18-byte blocks (144 B, two boxes a stage); K % 512 == 0, so rows are
    // 16-byte strided.  Rows past N read as zeros (d = 0).
    CUtensorMap tw;
    {
        const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
        const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
        const cuuint32_t box[2] = {(cuuint32_t)((kB18 ? kB18GroupBytes : kPairBytes) / 4), (cuuint32_t)C::kR};
        const cuuint32_t estride[2] = {1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    const int ntiles = (N + C::kR - 1) / C::kR;
    const int mtiles = (int)((M + C::kMt - 1) / C::kMt);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles, (unsigned)S, (unsigned)mtiles);
    cfg.blockDim = dim3(kMmaThreads);
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
    return cudaLaunchKernelEx(&cfg, matmul_mma_kernel<NT, T, kOcc, false, kB18>, tw, tq, ds, M, N, K, y, ldy, err,
                              static_cast<const int32_t*>(nullptr), 0, wt, skip_stage);
}

// One launch configuration: R weight rows per CTA and CTAs per SM, with its
// cluster-occupancy query and its launcher.
struct MmaConfig {
    int R, occ;
    int (*max_clusters)(int dev, int s, int num_sms);
    cudaError_t (*launch)(const void*, int64_t, EncodeTiledFn, const CUtensorMap&, const __half*, int64_t, int,
                          int, int, float*, int64_t, int*, int, int, cudaStream_t);
};
template <int NT, int T, int kOcc, bool kB18 = false>
constexpr MmaConfig cfg_of() {
    return {MmaCfg<NT, T, kOcc, kB18>::kR, kOcc, &mma_max_clusters<NT, T, kOcc, kB18>,
            &launch_nt<NT, T, kOcc, kB18>};
}
// Launch cost model, per activation-tile width: a wave of CTAs costs F, plus
// a per 128-row stage of one CTA (times the CTAs sharing an SM) and d per
// stage whatever its rows; every CTA beyond the first in a cluster adds c
// (the split-K reduction and the cluster's scheduling).  In microseconds,
// fitted by least squares to about 1,700 timed launches of every
// configuration on ten weight shapes (4096 x 4096 and the nine projections
// of a ~27B decoder layer) at 8, 16, 24 and 32 activation rows.
struct LaunchCost {
    double F, a, d, c;
};
constexpr LaunchCost kLaunchCost[4] = {
    {3.66, 1.21, 0.29, 0.71}, {4.20, 1.89, 0.11, 1.35}, {4.64, 3.14, 0.10, 1.06}, {4.64, 3.14, 0.10, 1.06}};

// The configuration (R, CTAs per SM) and K split S (= cluster size) for a
// call: the forced one (tests), else the measured one for this shape and
// tile height if the calibration installed it (measured on IQ4_XS weights,
// taken for every format), else the least
// modelled time waves x (F + a x occ x R / 128 x st x b + d x st) +
// c x (S - 1), st = ceil(pairs / S) stages per CTA and b = the stage row's
// bytes / 272, over the list's configurations and S = 1..8 (at most the K
// pairs), with waves from the clusters of S the device runs at once for
// that configuration.  Ties keep the earlier configuration (larger R, one
// CTA per SM) and the smaller S.
template <int NT, bool kB18>
void choose_config(const MmaConfig* list, int count, int64_t M, int N, int K, int num_sms, int* best_c,
                   int* best_s) {
    constexpr LaunchCost kC = kLaunchCost[NT - 1];
    constexpr double kRowScale = (double)MmaCfg<NT, 1, 1, kB18>::kRowB / kPairBytes;
    int dev = 0;
    cudaGetDevice(&dev);
    const int mtiles = (int)((M + 8 * NT - 1) / (8 * NT));
    const int pairs = (K + kPairK - 1) / kPairK;
    *best_c = 0;
    *best_s = 1;
    double best = 1e30;
    for (int ci = 0; ci < count; ++ci) {
        const MmaConfig& c = list[ci];
        const int units = (N + c.R - 1) / c.R * mtiles;
        for (int s = 1; s <= kMmaMaxCluster && s <= pairs; ++s) {
            const int mc = c.max_clusters(dev, s, num_sms);
            const int waves = (units + mc - 1) / mc;
            const double st = (double)((pairs + s - 1) / s);
            const double tm =
                waves * (kC.F + kC.a * c.occ * (double)c.R / 128.0 * st * kRowScale + kC.d * st) + kC.c * (s - 1);
            if (tm < best * 0.999) {
                best = tm;
                *best_c = ci;
                *best_s = s;
            }
        }
    }
    int fr = 0, fs = 0, fo = 0;
    mma_forced_config(&fr, &fs, &fo);
    int mr = 0, ms = 0, mo = 0;
    if (fr <= 0 && fs <= 0 && fo <= 0 && mma_measured_launch(N, K, 8 * NT, &mr, &ms, &mo)) {
        for (int ci = 0; ci < count; ++ci)
            if (list[ci].R == mr && list[ci].occ == mo && ms >= 1 && ms <= kMmaMaxCluster && ms <= pairs) {
                *best_c = ci;
                *best_s = ms;
                return;
            }
    }
    if (fr > 0 || fo > 0) {
        // the forced configuration, or the nearest one the list holds: the
        // largest R up to the one wanted with the wanted CTAs per SM, else
        // with any
        const int want_r = fr > 0 ? fr : list[*best_c].R, want_o = fo > 0 ? fo : list[*best_c].occ;
        int pick = -1;
        for (int pass = 0; pass < 2 && pick < 0; ++pass)
            for (int ci = 0; ci < count; ++ci) {
                const MmaConfig& c = list[ci];
                if (c.R > want_r || (pass < 1 && c.occ != want_o)) continue;
                if (pick < 0 || c.R > list[pick].R) pick = ci;
            }
        *best_c = pick < 0 ? count - 1 : pick;
    }
    if (fs > 0) *best_s = fs < pairs ? fs : pairs;
}

template <int NT, bool kB18, int kCount>
cudaError_t launch_best(const MmaConfig (&list)[kCount], const void* w, int64_t row_bytes, EncodeTiledFn enc,
                        const CUtensorMap& tq, const __half* ds, int64_t M, int N, int K, float* y, int64_t ldy,
                        int* err, int wt, int skip_stage, int num_sms, cudaStream_t stream) {
    int ci = 0, s = 1;
    choose_config<NT, kB18>(list, kCount, M, N, K, num_sms, &ci, &s);
    return list[ci].launch(w, row_bytes, enc, tq, ds, M, N, K, s, y, ldy, err, wt, skip_stage, stream);
}

// Q8_1 codes: one box = mt rows x 128 codes, 128-byte swizzle; rows past
// M read as zeros.
inline cudaError_t encode_q_map(EncodeTiledFn enc, const int8_t* qs, int64_t K, int64_t M, int mt,
                                CUtensorMap* tq) {
    const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t gstride[1] = {(cuuint64_t)K};
    const cuuint32_t box[2] = {(cuuint32_t)kQBoxK, (cuuint32_t)mt};
    const cuuint32_t estride[2] = {1, 1};
    return enc(tq, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<int8_t*>(qs), gdim, gstride, box, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
               ? cudaSuccess
               : cudaErrorInvalidValue;
}


// Grouped (mixture-of-experts) launch of the persistent <NT, T> kernel for
// weights of layout kB18 (format wt): W of expert g through a 3D tensor map
// (row words x rows x experts, expert_stride bytes apart); one CTA per SM,
// or fewer when the layer has fewer work items (at most row tiles x
// (activation tiles of all rows + experts with rows)).
template <int NT, int T, bool kB18>
cudaError_t launch_grouped_nt(const void* w, int64_t expert_stride, int G, int64_t row_bytes, EncodeTiledFn enc,
                              const CUtensorMap& tq, const __half* ds, const int32_t* row_offsets, int64_t rows,
                              int slots, int N, int K, float* y, int64_t ldy, int* err, int wt, int num_sms,
                              int skip_w_stage, cudaStream_t stream) {
    using C = MmaCfg<NT, T, 1, kB18, true>;
    int dev = 0;
    cudaGetDevice(&dev);
    const cudaError_t ea = mma_smem_attr<NT, T, 1, true, kB18>(dev);
    if (ea != cudaSuccess) return ea;
    CUtensorMap tw;
    {
        const cuuint64_t gdim[3] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N, (cuuint64_t)G};
        const cuuint64_t gstride[2] = {(cuuint64_t)row_bytes, (cuuint64_t)expert_stride};
        const cuuint32_t box[3] = {(cuuint32_t)((kB18 ? kB18GroupBytes : kPairBytes) / 4), (cuuint32_t)C::kR, 1};
        const cuuint32_t estride[3] = {1, 1, 1};
        if (enc(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(w), gdim, gstride, box, estride,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return cudaErrorInvalidValue;
    }
    cudaLaunchConfig_t cfg = {};
    const int64_t items = (N + C::kR - 1) / C::kR * ((rows + C::kMt - 1) / C::kMt + slots);
    cfg.gridDim = dim3((unsigned)(items < num_sms ? items : num_sms), 1, 1);
    cfg.blockDim = dim3(kMmaThreads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, matmul_mma_kernel<NT, T, 1, true, kB18>, tw, tq, ds, rows, N, K, y, ldy, err,
                              row_offsets, G, wt, skip_w_stage);
}

// The grouped form's launch: activation tiles of mma_tile_rows(mean rows per
// expert with rows) rows (larger experts take several tiles); 128-row
// weight tiles, or 64 / 32 when the experts' row tiles alone do not give
// every SM a work item; at 32 activation rows 64 at most (the partial tiles
// of 128 rows would leave one stage).
template <bool kB18>
cudaError_t launch_grouped(int wt, const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                           const int8_t* qs, const void* ds, const int32_t* row_offsets, int64_t total_rows, float* y,
                           int64_t ldy, void* encode, int* err, int num_sms, int skip_w_stage, cudaStream_t stream) {
    const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(encode);
    const int64_t row_bytes = wt_row_bytes(wt, K);
    const int slots = (int)(G < total_rows ? G : total_rows);  // experts that can have rows
    const int64_t mean = (total_rows + slots - 1) / slots;
    const int mt = mma_tile_rows(mean);
    CUtensorMap tq;
    const cudaError_t eq = encode_q_map(enc, qs, K, total_rows, mt, &tq);
    if (eq != cudaSuccess) return eq;
    const __half* dsh = reinterpret_cast<const __half*>(ds);
    const int Ni = (int)N, Ki = (int)K, Gi = (int)G;
    const int64_t ctas128 = (N + 127) / 128 * slots;
    int rows_cta = ctas128 >= num_sms ? 128 : ((N + 63) / 64 * slots >= num_sms ? 64 : 32);
    if (mt == 32 && rows_cta > 64) rows_cta = 64;
#define IQ4XS_MMA_G(nt, t)                                                                                      \
    launch_grouped_nt<nt, t, kB18>(w, expert_stride, Gi, row_bytes, enc, tq, dsh, row_offsets, total_rows, slots, \
                                   Ni, Ki, y, ldy, err, wt, num_sms, skip_w_stage, stream)
    switch (mt * 1000 + rows_cta) {
        case 8128: return IQ4XS_MMA_G(1, 4);
        case 8064: return IQ4XS_MMA_G(1, 2);
        case 8032: return IQ4XS_MMA_G(1, 1);
        case 16128: return IQ4XS_MMA_G(2, 4);
        case 16064: return IQ4XS_MMA_G(2, 2);
        case 16032: return IQ4XS_MMA_G(2, 1);
        case 24128: return IQ4XS_MMA_G(3, 4);
        case 24064: return IQ4XS_MMA_G(3, 2);
        case 24032: return IQ4XS_MMA_G(3, 1);
        case 32064: return IQ4XS_MMA_G(4, 2);
        case 32032: return IQ4XS_MMA_G(4, 1);
        default: return cudaErrorInvalidValue;
    }
#undef IQ4XS_MMA_G
}

}  // namespace
}  // namespace iq4xs
