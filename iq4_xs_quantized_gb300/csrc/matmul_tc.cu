// matmul_tc.cu -- IQ4_XS x Q8_1 matmul on the 5th-generation tensor cores.
//
// Method (V100TPS engine page, new-kernel table and the tile-geometry passage
// after it): per 32-weight sub-block, an exact integer dot product of decoded
// codebook values with Q8_1 codes, scaled by d_w*(ls-32)*d_x into fp32.
//
// GB300 design.  sm_103a has no integer tcgen05 kind, so the exact small
// integers travel as fp16 (kv in [-127, 113], q in [-127, 127]: every product
// and every 32-term sum is an integer below 2^24, exact in the fp32 TMEM
// accumulator).  One CTA owns 128 weight rows (= 128 TMEM lanes = UMMA M)
// and an activation tile of MT rows (= UMMA N); K is split over a cluster
// whose CTAs reduce their partial tiles through distributed shared memory.
//
// Warp-specialized roles, each a loop over the CTA's sub-blocks, decoupled by
// mbarrier rings so that no round trip sits on the critical path:
//   warpgroups 0, 1 (decoders)  sub-blocks of parity g: thread t decodes row
//                               t's sub-block from the staged W bytes to exact
//                               fp16 in the canonical K-major layout (A ring);
//                               after a barrier over the warpgroup, its first
//                               thread issues two tcgen05.mma 128 x MT x 16 for
//                               that sub-block into a fresh TMEM accumulator
//                               (kND slots).  Issuing from the decoders keeps
//                               the MMA issue off a separate warp whose
//                               integer work would queue behind the decoders'
//                               on the shared ALU pipes.
//   warp 12 (producer)          TMA: W stages of 2 super-blocks (128 x 272 B,
//                               2D tensor map); activation stages of 4
//                               sub-blocks (bulk copies of the pre-tiled fp16
//                               codes and their fp32 block scales)
//   warp 13                     allocates and frees TMEM
//   warpgroup 2 (epilogue)      thread t loads row t's int-valued fp32 results
//                               (all columns, then one wait) and scales them by
//                               d_w*(ls-32)*d_x into fp32 register accumulators
// Every mbarrier wait is bounded (2 s); a timeout sets the device error word
// and an abort flag that releases every other wait, the CTA drains its copies
// and frees its TMEM, and the call's output is undefined.
#include <cuda.h>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kTcThreads = 32 * 16;   // 4 warpgroups
constexpr int kDecGroups = 2;         // decoder warpgroups 0, 1 (sub-block parity)
constexpr int kEpiWarp0 = 8;          // epilogue: warps 8-11
constexpr int kProducerWarp = 12;
constexpr int kTmemWarp = 13;         // TMEM owner; warps 14, 15 idle
constexpr int kTmemCols = 512;        // whole TMEM; one CTA per SM (see kMinSmem)
constexpr int kMaxCluster = 8;
constexpr int kMinSmem = 120 * 1024;  // > half of the SM's shared memory: one CTA per SM
constexpr int kDecUnit = 2;           // sub-blocks a decoder warpgroup takes per step
constexpr int kALbo = kTileN * 16;    // A: byte distance between K-adjacent core matrices
constexpr int kCoreSbo = 128;         // 8 rows x 16 B core matrices, contiguous along M/N
// Per-warpgroup register budgets (setmaxnreg).  The block launches with
// 65536 / 512 = 128 registers per thread; the budgets sum to
// 128 * (2 * 96 + 248 + 56) = 63488, within the 65536 it holds.
constexpr int kRegsDecode = 96;
constexpr int kRegsEpilogue = 248;
constexpr int kRegsControl = 56;
static_assert(128 * (kDecGroups * kRegsDecode + kRegsEpilogue + kRegsControl) <= kTcThreads * 128,
              "register split fits the launch allocation");

template <int R>
__device__ __forceinline__ void reg_alloc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(R));
}
template <int R>
__device__ __forceinline__ void reg_dealloc() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(R));
}

template <int MT>
struct TcCfg {
    static_assert(MT % 16 == 0 && MT >= 16 && MT <= kMaxMTile, "UMMA N for M=128");
    // A (decoded fp16) slots = TMEM accumulators.  The slots in flight set
    // the throughput of the decode -> MMA -> epilogue ring (each slot's round
    // trip is a few thousand cycles), so use as many as TMEM and shared
    // memory allow.  Decoder g's steps use slots whose index / kDecUnit has
    // parity g.
    static constexpr int kNA = (MT <= 64) ? 8 : 4;
    static constexpr int kND = kNA;
    static_assert(kNA % (kDecGroups * kDecUnit) == 0, "slots split evenly between decoders");
    static_assert(kND * MT <= kTmemCols, "accumulators fit TMEM");
    static constexpr int kNW = (MT <= 48) ? 3 : 2;             // W stages
    static constexpr int kNB = (MT <= 96) ? 4 : 3;             // activation stages
    static constexpr int kBQhBytes = kBStageChunks * MT * 16;  // fp16 codes of 4 sub-blocks
    static constexpr int kBDxBytes = kBStageSubs * MT * 4;     // their fp32 block scales
    // slot stride, padded to 1 KB; the copies into a slot fill kBQhBytes + kBDxBytes
    static constexpr int kBStageBytes = (kBQhBytes + kBDxBytes + 1023) / 1024 * 1024;
    static constexpr int kPartCols = (MT > 64) ? 64 : MT;      // TMEM columns read per wait
    static constexpr int kOffW = 0;
    static constexpr int kOffB = kOffW + kNW * kWStageBytes;
    static constexpr int kOffA = kOffB + kNB * kBStageBytes;
    static constexpr int kOffBar = kOffA + kNA * kASubBytes;
    static_assert(kOffBar <= 226 * 1024, "stages and slots fit shared memory");
    // W full/empty, B full/empty, MMA done / accumulator free per slot, drain
    static constexpr int kNumBars = 2 * kNW + 2 * kNB + 2 * kND + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;   // tmem base, abort flag
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmem = (kUsed + 1024 > kMinSmem) ? kUsed + 1024 : kMinSmem;
    static constexpr int kRedStride = MT + 1;                  // fp32 words per row
    static_assert(kTileN * kRedStride * 4 <= kNW * kWStageBytes, "reduction tile fits the W ring");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kOffB % 1024 == 0 && kOffA % 1024 == 0 && kBStageBytes % 16 == 0, "alignment");
    static_assert(kPartCols % 16 == 0, "TMEM read granularity");
};

constexpr int kEpilogueBarrier = 1;  // named barrier id for the 4 epilogue warps
constexpr int kDecodeBarrier0 = 2;   // named barrier ids 2, 3: decoder warpgroups 0, 1

__device__ __forceinline__ void named_barrier_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ float ld_dsmem_f32(uint32_t local_saddr, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local_saddr), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

template <int MT>
__global__ void __launch_bounds__(kTcThreads, 1)
    matmul_tc_kernel(const __grid_constant__ CUtensorMap tmap_w,
                     const uint8_t* __restrict__ tc_op, int64_t M, int N, int K,
                     float* __restrict__ y, int64_t ldy, int* err) {
    using C = TcCfg<MT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
    uint64_t* w_full = bars;
    uint64_t* w_empty = w_full + C::kNW;
    uint64_t* b_full = w_empty + C::kNW;
    uint64_t* b_empty = b_full + C::kNB;
    // mma_done[s]: the MMAs of the sub-block in slot s are complete (its A
    // slot may be rewritten, its accumulator read); d_free[s]: the epilogue
    // has read accumulator s.  Since an MMA into slot s waits for d_free[s],
    // mma_done[s] never runs two phases ahead of either waiter.
    uint64_t* mma_done = b_empty + C::kNB;
    uint64_t* d_free = mma_done + C::kND;
    uint64_t* drain = d_free + C::kND;
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
    const int nbst = nsub / kBStageSubs;
    const int64_t K8 = K / kChunkElems, K32 = K / kSub;
    const uint8_t* qh_tile = tc_op + (int64_t)z * K8 * MT * 16;
    const uint8_t* dx_tile = tc_op + tc_qh_bytes(M, K) + (int64_t)z * K32 * MT * 4;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNW; ++i) {
            mbar_init(&w_full[i], 1);
            mbar_init(&w_empty[i], (kDecGroups + 1) * kTileN);  // both decoders + epilogue
        }
        for (int i = 0; i < C::kNB; ++i) {
            mbar_init(&b_full[i], 1);
            // one MMA commit per decoder warpgroup + the epilogue (block scales)
            mbar_init(&b_empty[i], kDecGroups + kTileN);
        }
        for (int i = 0; i < C::kND; ++i) { mbar_init(&mma_done[i], 1); mbar_init(&d_free[i], kTileN); }
        mbar_init(drain, kDecGroups);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kProducerWarp && lane == 0) prefetch_tmap(&tmap_w);
    if (warp == kTmemWarp) tmem_alloc(tmem_base_ptr, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_ptr;
    // Let the next kernel in the stream begin its launch; it waits for this
    // grid's completion before touching anything this grid reads or writes.
    griddep_launch_dependents();

    if (warp >= kProducerWarp) {
        reg_dealloc<kRegsControl>();
        if (warp == kProducerWarp && lane == 0) {
            // ------------------------------------------------------- producer
            int issued_w = 0, issued_b = 0;
            bool ok = true;
            // W is read-only model state: its first stages stream before the
            // preceding kernel (which produces the activations) has finished.
            const int pre = (C::kNW < (p1 - p0)) ? C::kNW : (p1 - p0);
            for (int ps = 0; ps < pre; ++ps) {
                mbar_arrive_expect_tx(&w_full[ps], kWStageBytes);
                tma_load_2d(smem + C::kOffW + ps * kWStageBytes, &tmap_w,
                            (p0 + ps) * (kPairBytes / 4), n0, &w_full[ps]);
                ++issued_w;
            }
            griddep_wait();
            for (int bs = 0; bs < nbst && ok; ++bs) {
                if (bs % (kSubPerPair / kBStageSubs) == 0) {
                    const int ps = bs / (kSubPerPair / kBStageSubs);
                    if (ps >= pre) {
                        const int slot = ps % C::kNW;
                        ok = mbar_wait(&w_empty[slot], ((ps / C::kNW) - 1) & 1, abort_flag, err,
                                       kDevErrTimeoutW);
                        if (!ok) break;
                        mbar_arrive_expect_tx(&w_full[slot], kWStageBytes);
                        tma_load_2d(smem + C::kOffW + slot * kWStageBytes, &tmap_w,
                                    (p0 + ps) * (kPairBytes / 4), n0, &w_full[slot]);
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
                mbar_arrive_expect_tx(&b_full[slot], C::kBQhBytes + C::kBDxBytes);
                bulk_load(dst, qh_tile + sub0 * kChunksPerSub * MT * 16, C::kBQhBytes, &b_full[slot]);
                bulk_load(dst + C::kBQhBytes, dx_tile + sub0 * MT * 4, C::kBDxBytes, &b_full[slot]);
                ++issued_b;
            }
            // Drain: the last copies issued into each ring slot have landed.
            for (int ps = (issued_w > C::kNW ? issued_w - C::kNW : 0); ps < issued_w; ++ps)
                mbar_wait(&w_full[ps % C::kNW], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutDrain);
            for (int bs = (issued_b > C::kNB ? issued_b - C::kNB : 0); bs < issued_b; ++bs)
                mbar_wait(&b_full[bs % C::kNB], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutDrain);
        } else if (warp == kTmemWarp) {
            // Every MMA issued by both decoder warpgroups has completed before
            // TMEM is released (one commit from each).
            mbar_wait(drain, 0, abort_flag, err, kDevErrTimeoutDrain);
        }
    } else if (warp < kEpiWarp0) {
        // ------------------------------------------------------------ decoders
        reg_dealloc<kRegsDecode>();
        const int g = warp >> 2;                   // sub-block parity of this warpgroup
        const int t = threadIdx.x & (kTileN - 1);  // row within the tile
        uint8_t* a_row = smem + C::kOffA + t * 16;
        constexpr uint32_t idesc = idesc_f16_m128(MT);
        const uint32_t a_base = smem_u32(smem + C::kOffA);
        const uint32_t b_base = smem_u32(smem + C::kOffB);
        bool ok = true;
        // Step: sub-blocks l0, l0+1 (l0 = 4k + 2g), always in slots 2g, 2g+1,
        // always in one super-block and one activation stage.
        for (int l0 = kDecUnit * g; l0 < nsub; l0 += kDecUnit * kDecGroups) {
            const int ps = l0 / kSubPerPair, jj = l0 % kSubPerPair, wslot = ps % C::kNW;
            if (ok && jj < kDecUnit * kDecGroups)
                ok = mbar_wait(&w_full[wslot], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutW);
            const uint8_t* rowp = smem + C::kOffW + wslot * kWStageBytes + t * kPairBytes +
                                  (jj / kSubPerBlock) * kBlockBytes;
            const int j = jj % kSubPerBlock;
            uint2 q[2 * kDecUnit];
#pragma unroll
            for (int u = 0; u < kDecUnit; ++u) {
                q[2 * u] = *reinterpret_cast<const uint2*>(rowp + 8 + 16 * (j + u));
                q[2 * u + 1] = *reinterpret_cast<const uint2*>(rowp + 16 + 16 * (j + u));
            }
            if (jj >= kSubPerPair - kDecUnit * kDecGroups) mbar_arrive(&w_empty[wslot]);
            uint32_t h[16 * kDecUnit];
#pragma unroll
            for (int u = 0; u < 2 * kDecUnit; ++u) {
                decode_f16x2(q[u].x, h + 8 * u);
                decode_f16x2(q[u].y, h + 8 * u + 4);
            }
            const int s0 = l0 % C::kNA;
            if (ok && l0 >= C::kNA) {
#pragma unroll
                for (int u = 0; u < kDecUnit; ++u)
                    if (ok) ok = mbar_wait(&mma_done[s0 + u], ((l0 / C::kNA) - 1) & 1, abort_flag, err,
                                           kDevErrTimeoutA);
            }
#pragma unroll
            for (int u = 0; u < kDecUnit; ++u) {
                uint8_t* ap = a_row + (s0 + u) * kASubBytes;
#pragma unroll
                for (int c = 0; c < kChunksPerSub; ++c)
                    *reinterpret_cast<uint4*>(ap + c * kALbo) =
                        make_uint4(h[16 * u + 4 * c], h[16 * u + 4 * c + 1], h[16 * u + 4 * c + 2],
                                   h[16 * u + 4 * c + 3]);
            }
            fence_proxy_async_smem();
            // All 128 rows of both slots are written (and fenced for the async
            // proxy); the warpgroup's first thread issues their MMAs.
            named_barrier_sync(kDecodeBarrier0 + g, kTileN);
            if (t == 0) {
                const int bs = l0 / kBStageSubs, bslot = bs % C::kNB;
                if (ok && l0 >= C::kNA) {
#pragma unroll
                    for (int u = 0; u < kDecUnit; ++u)
                        if (ok) ok = mbar_wait(&d_free[s0 + u], ((l0 / C::kNA) - 1) & 1, abort_flag, err,
                                               kDevErrTimeoutFree);
                }
                if (ok)
                    ok = mbar_wait(&b_full[bslot], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutB);
                tc_fence_after();
#pragma unroll
                for (int u = 0; u < kDecUnit; ++u) {
                    const int li = l0 + u, sa = s0 + u;
                    if (ok) {
                        const uint32_t d_tmem = tmem + (uint32_t)(sa * MT);
                        const uint32_t a_addr = a_base + sa * kASubBytes;
                        const uint32_t b_addr = b_base + bslot * C::kBStageBytes +
                                                (li % kBStageSubs) * kChunksPerSub * MT * 16;
#pragma unroll
                        for (int i = 0; i < kMmaPerSub; ++i) {
                            const uint64_t adesc = smem_desc(a_addr + i * 2 * kALbo, kALbo, kCoreSbo);
                            const uint64_t bdesc =
                                smem_desc(b_addr + i * 2 * MT * 16, MT * 16, kCoreSbo);
                            tc_mma_f16(d_tmem, adesc, bdesc, idesc, i);
                        }
                    }
                    // Commits are made even after an abort so that every
                    // waiter's barrier still completes.
                    tc_commit(&mma_done[sa]);
                }
                // this warpgroup's sub-blocks of the activation stage are issued
                tc_commit(&b_empty[bslot]);
            }
        }
        if (t == 0) tc_commit(drain);
    } else {
        // ------------------------------------------------------------ epilogue
        reg_alloc<kRegsEpilogue>();
        const int t = threadIdx.x - kEpiWarp0 * 32;  // row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        bool ok = true;
        for (int li = 0; li < nsub; ++li) {
            const int ps = li / kSubPerPair, jj = li % kSubPerPair, wslot = ps % C::kNW;
            const int bs = li / kBStageSubs, bslot = bs % C::kNB;
            if (ok && jj == 0)
                ok = mbar_wait(&w_full[wslot], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutW);
            const uint8_t* rowp = smem + C::kOffW + wslot * kWStageBytes + t * kPairBytes +
                                  (jj / kSubPerBlock) * kBlockBytes;
            const uint2 hdr = *reinterpret_cast<const uint2*>(rowp);
            if (jj == kSubPerPair - 1) mbar_arrive(&w_empty[wslot]);
            const float Sw = iq4xs_scale(hdr.x, hdr.y, jj % kSubPerBlock);
            const float2 Sw2 = make_float2(Sw, Sw);
            if (ok && li % kBStageSubs == 0)
                ok = mbar_wait(&b_full[bslot], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutB);
            const float4* dx4 = reinterpret_cast<const float4*>(
                smem + C::kOffB + bslot * C::kBStageBytes + C::kBQhBytes + (li % kBStageSubs) * MT * 4);
            const int sd = li % C::kND;
            if (ok) ok = mbar_wait(&mma_done[sd], (li / C::kND) & 1, abort_flag, err, kDevErrTimeoutMma);
            tc_fence_after();
#pragma unroll
            for (int part = 0; part < MT; part += C::kPartCols) {
                constexpr int kW = C::kPartCols;  // columns of this part (the last may be narrower)
                const int cols = (MT - part < kW) ? MT - part : kW;
                uint32_t r[kW];
                const uint32_t taddr = tmem + lane_base + (uint32_t)(sd * MT + part);
                if (cols == 64) tmem_ld64_wait(taddr, r);
                else if (cols == 48) tmem_ld48_wait(taddr, r);
                else if (cols == 32) tmem_ld32_wait(taddr, r);
                else tmem_ld16_wait(taddr, r);
                if (part + C::kPartCols >= MT) {
                    tc_fence_before();
                    mbar_arrive(&d_free[sd]);
                }
#pragma unroll
                for (int k = 0; k < kW; k += 4) {
                    if (k >= cols) break;
                    const int m = part + k;
                    const float4 d = dx4[m / 4];
                    const float2 s01 = __fmul2_rn(Sw2, make_float2(d.x, d.y));
                    const float2 s23 = __fmul2_rn(Sw2, make_float2(d.z, d.w));
                    const float2 a01 =
                        __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), s01,
                                   make_float2(acc[m], acc[m + 1]));
                    const float2 a23 =
                        __ffma2_rn(make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])),
                                   s23, make_float2(acc[m + 2], acc[m + 3]));
                    acc[m] = a01.x;
                    acc[m + 1] = a01.y;
                    acc[m + 2] = a23.x;
                    acc[m + 3] = a23.y;
                }
            }
            if (li % kBStageSubs == kBStageSubs - 1) mbar_arrive(&b_empty[bslot]);
        }
        // Partial tile -> y (one CTA) or -> shared memory for the cluster
        // reduction, which reuses the W ring.  Before any epilogue thread
        // writes there, all four epilogue warps must have read their last
        // block headers from it (named barrier); the decoders' last reads of
        // it preceded the last accumulator these threads waited for, and
        // every W copy issued has been consumed.
        const int64_t mrows = M - (int64_t)z * MT;
        if (S == 1) {
            griddep_wait();
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < mrows && n0 + t < N) y[((int64_t)z * MT + m) * ldy + n0 + t] = acc[m];
        } else {
            named_barrier_sync(kEpilogueBarrier, kTileN);
            float* red = reinterpret_cast<float*>(smem + C::kOffW);
#pragma unroll
            for (int m = 0; m < MT; ++m) red[t * C::kRedStride + m] = acc[m];
        }
    }

    if (S > 1) {
        // Split-K reduction over the cluster through distributed shared memory:
        // CTA `rank` sums rows [rank*128/S, (rank+1)*128/S) over all CTAs in
        // rank order (deterministic) and writes them.
        __syncwarp();
        cluster_sync_all();
        if (warp < kProducerWarp) {
            griddep_wait();
            const int64_t mrows = M - (int64_t)z * MT;
            const uint32_t red_s = smem_u32(smem + C::kOffW);
            const int r0 = (int)(kTileN * rank / S), r1 = (int)(kTileN * (rank + 1) / S);
            const int rows = r1 - r0;
            for (int e = threadIdx.x; e < rows * MT; e += kProducerWarp * 32) {
                const int row = r0 + e % rows, m = e / rows;
                float v = 0.f;
                for (int q = 0; q < S; ++q)
                    v += ld_dsmem_f32(red_s + (uint32_t)((row * C::kRedStride + m) * 4), (uint32_t)q);
                if (m < mrows && n0 + row < N) y[((int64_t)z * MT + m) * ldy + n0 + row] = v;
            }
        }
        __syncwarp();
        cluster_sync_all();
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

template <int MT>
cudaError_t launch_mt(const CUtensorMap& tmap, const uint8_t* tc_op, int64_t M, int N, int K,
                      float* y, int64_t ldy, int* err, int S, int ntiles, int mtiles,
                      cudaStream_t stream) {
    using C = TcCfg<MT>;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(matmul_tc_kernel<MT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles, (unsigned)S, (unsigned)mtiles);
    cfg.blockDim = dim3(kTcThreads);
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
    return cudaLaunchKernelEx(&cfg, matmul_tc_kernel<MT>, tmap, tc_op, M, N, K, y, ldy, err);
}

}  // namespace

cudaError_t launch_matmul_tc(const void* w, int64_t N, int64_t K, const void* tc_operand,
                             int64_t M, float* y, int64_t ldy, void* encode, int* err,
                             int num_sms, cudaStream_t stream) {
    const int64_t row_bytes = (K / kQK) * kBlockBytes;
    CUtensorMap tmap;
    const cuuint64_t gdim[2] = {(cuuint64_t)(row_bytes / 4), (cuuint64_t)N};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_bytes};
    const cuuint32_t box[2] = {(cuuint32_t)(kPairBytes / 4), (cuuint32_t)kTileN};
    const cuuint32_t estride[2] = {1, 1};
    CUresult cr = reinterpret_cast<EncodeTiledFn>(encode)(
        &tmap, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(w), gdim, gstride, box,
        estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS) return cudaErrorInvalidValue;

    const int MT = tc_mtile(M);
    const int mtiles = (int)tc_num_mtiles(M);
    const int ntiles = (int)((N + kTileN - 1) / kTileN);
    const int pairs = (int)(K / kPairK);
    int S = num_sms / (ntiles * mtiles);
    if (S > kMaxCluster) S = kMaxCluster;
    if (S > pairs) S = pairs;
    if (S < 1) S = 1;
    const uint8_t* op = reinterpret_cast<const uint8_t*>(tc_operand);
    const int Ni = (int)N, Ki = (int)K;
    switch (MT) {
        case 16: return launch_mt<16>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 32: return launch_mt<32>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 48: return launch_mt<48>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 64: return launch_mt<64>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 80: return launch_mt<80>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 96: return launch_mt<96>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 112: return launch_mt<112>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        case 128: return launch_mt<128>(tmap, op, M, Ni, Ki, y, ldy, err, S, ntiles, mtiles, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace iq4xs
