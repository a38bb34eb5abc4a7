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
//   warp 8 (producer)  TMA: W stages of 2 super-blocks (128 x 272 B, 2D tensor
//                      map) and activation stages of 4 sub-blocks (bulk copy
//                      of the pre-tiled fp16 operand).
//   warp 9 (issuer)    allocates TMEM; one thread issues tcgen05.mma
//                      128 x MT x 16 twice per sub-block into a fresh TMEM
//                      accumulator, commits to mbarriers.
//   warps 0-7          two groups of 4 warps; group g takes the sub-blocks of
//                      parity g.  Thread t decodes row t's sub-block from the
//                      staged bytes to exact fp16 in the canonical K-major
//                      layout, then scales the previous sub-block's TMEM result
//                      into its fp32 register accumulators.
//
// Every mbarrier wait is bounded (2 s); a timeout sets the device error word
// and an abort flag that releases every other wait, the CTA drains its copies
// and frees its TMEM, and the call's output is undefined.
#include <cuda.h>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kTcWorkerWarps = 8;
constexpr int kTcProducerWarp = 8;
constexpr int kTcIssuerWarp = 9;
constexpr int kTcThreads = 32 * 10;
constexpr int kGroups = 2;        // worker groups (sub-block parity)
constexpr int kSlots = 2;         // A buffers / TMEM accumulators per group
constexpr int kTmemCols = 512;    // whole TMEM; one CTA per SM (see kMinSmem)
constexpr int kMaxCluster = 8;
constexpr int kMinSmem = 120 * 1024;  // > half of the SM's shared memory: one CTA per SM
constexpr int kALbo = kTileN * 16;    // A: byte distance between K-adjacent core matrices
constexpr int kCoreSbo = 128;         // 8 rows x 16 B core matrices, contiguous along M/N

template <int MT>
struct TcCfg {
    static_assert(MT % 16 == 0 && MT >= 16 && MT <= kMaxMTile, "UMMA N for M=128");
    static_assert(kGroups * kSlots * MT <= kTmemCols, "TMEM accumulators fit");
    static constexpr int kNW = (MT <= 64) ? 3 : 2;            // W stages
    static constexpr int kNB = 3;                             // activation stages
    static constexpr int kBStageBytes = kBStageChunks * MT * 16;
    static constexpr int kOffW = 0;
    static constexpr int kOffB = kOffW + kNW * kWStageBytes;
    static constexpr int kOffA = kOffB + kNB * kBStageBytes;
    static constexpr int kOffBar = kOffA + kGroups * kSlots * kASubBytes;
    // barriers: W full/empty, B full/empty, per (group, slot): a_full, mma_done, d_free; drain
    static constexpr int kNumBars = 2 * kNW + 2 * kNB + 3 * kGroups * kSlots + 1;
    static constexpr int kOffMisc = kOffBar + 8 * kNumBars;   // tmem base, abort flag
    static constexpr int kUsed = kOffMisc + 16;
    static constexpr int kSmem = (kUsed + 1024 > kMinSmem) ? kUsed + 1024 : kMinSmem;
    static constexpr int kRedStride = MT + 1;                  // fp32 words per row
    static_assert(kTileN * kRedStride * 4 <= kNW * kWStageBytes, "reduction tile fits the W ring");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
    static_assert(kOffB % 1024 == 0 && kOffA % 1024 == 0, "stage alignment");
};

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
    uint64_t* a_full = b_empty + C::kNB;          // [g][s]
    uint64_t* mma_done = a_full + kGroups * kSlots;
    uint64_t* d_free = mma_done + kGroups * kSlots;
    uint64_t* drain = d_free + kGroups * kSlots;
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
    const int npairs = p1 - p0;
    const int nsub = npairs * kSubPerPair;
    const int nbst = nsub / kBStageSubs;
    const int64_t K8 = K / kChunkElems, K32 = K / kSub;
    const uint8_t* qh_tile = tc_op + (int64_t)z * K8 * MT * 16;
    const float* dx_tile =
        reinterpret_cast<const float*>(tc_op + tc_qh_bytes(M, K)) + (int64_t)z * K32 * MT;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kNW; ++i) { mbar_init(&w_full[i], 1); mbar_init(&w_empty[i], kTcWorkerWarps * 32); }
        for (int i = 0; i < C::kNB; ++i) { mbar_init(&b_full[i], 1); mbar_init(&b_empty[i], 1); }
        for (int i = 0; i < kGroups * kSlots; ++i) {
            mbar_init(&a_full[i], 4 * 32);
            mbar_init(&mma_done[i], 1);
            mbar_init(&d_free[i], 4 * 32);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == kTcProducerWarp && lane == 0) prefetch_tmap(&tmap_w);
    if (warp == kTcIssuerWarp) tmem_alloc(tmem_base_ptr, kTmemCols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_ptr;

    if (warp == kTcProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int issued_w = 0, issued_b = 0;
            bool ok = true;
            for (int bs = 0; bs < nbst && ok; ++bs) {
                if (bs % (kSubPerPair / kBStageSubs) == 0) {
                    const int ps = bs / (kSubPerPair / kBStageSubs);
                    const int slot = ps % C::kNW;
                    if (ps >= C::kNW)
                        ok = mbar_wait(&w_empty[slot], ((ps / C::kNW) - 1) & 1, abort_flag, err, kDevErrTimeoutW);
                    if (!ok) break;
                    mbar_arrive_expect_tx(&w_full[slot], kWStageBytes);
                    tma_load_2d(smem + C::kOffW + slot * kWStageBytes, &tmap_w,
                                (p0 + ps) * (kPairBytes / 4), n0, &w_full[slot]);
                    ++issued_w;
                }
                const int slot = bs % C::kNB;
                if (bs >= C::kNB)
                    ok = mbar_wait(&b_empty[slot], ((bs / C::kNB) - 1) & 1, abort_flag, err, kDevErrTimeoutB);
                if (!ok) break;
                mbar_arrive_expect_tx(&b_full[slot], C::kBStageBytes);
                const int64_t chunk0 = ((int64_t)p0 * kSubPerPair + (int64_t)bs * kBStageSubs) * kChunksPerSub;
                bulk_load(smem + C::kOffB + slot * C::kBStageBytes, qh_tile + chunk0 * MT * 16,
                          C::kBStageBytes, &b_full[slot]);
                ++issued_b;
            }
            // Drain: the last copies issued into each ring slot have landed.
            for (int ps = (issued_w > C::kNW ? issued_w - C::kNW : 0); ps < issued_w; ++ps)
                mbar_wait(&w_full[ps % C::kNW], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutDrain);
            for (int bs = (issued_b > C::kNB ? issued_b - C::kNB : 0); bs < issued_b; ++bs)
                mbar_wait(&b_full[bs % C::kNB], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutDrain);
        }
    } else if (warp == kTcIssuerWarp) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_m128(MT);
            const uint32_t a_base = smem_u32(smem + C::kOffA);
            const uint32_t b_base = smem_u32(smem + C::kOffB);
            bool ok = true;
            for (int li = 0; li < nsub && ok; ++li) {
                const int g = li & 1, u = li >> 1, s = u & 1, gs = g * kSlots + s;
                ok = mbar_wait(&a_full[gs], (u >> 1) & 1, abort_flag, err, kDevErrTimeoutA);
                if (ok && u >= 2) ok = mbar_wait(&d_free[gs], ((u - 2) >> 1) & 1, abort_flag, err, kDevErrTimeoutFree);
                const int bs = li / kBStageSubs, bslot = bs % C::kNB;
                if (ok && li % kBStageSubs == 0)
                    ok = mbar_wait(&b_full[bslot], (bs / C::kNB) & 1, abort_flag, err, kDevErrTimeoutB);
                if (!ok) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem + (uint32_t)(gs * MT);
                const uint32_t a_addr = a_base + gs * kASubBytes;
                const uint32_t b_addr =
                    b_base + bslot * C::kBStageBytes + (li % kBStageSubs) * kChunksPerSub * MT * 16;
#pragma unroll
                for (int i = 0; i < kMmaPerSub; ++i) {
                    const uint64_t adesc = smem_desc(a_addr + i * 2 * kALbo, kALbo, kCoreSbo);
                    const uint64_t bdesc = smem_desc(b_addr + i * 2 * MT * 16, MT * 16, kCoreSbo);
                    tc_mma_f16(d_tmem, adesc, bdesc, idesc, i);
                }
                tc_commit(&mma_done[gs]);
                if (li % kBStageSubs == kBStageSubs - 1) tc_commit(&b_empty[bslot]);
            }
            // Every MMA issued so far has completed before TMEM is released.
            tc_commit(drain);
            mbar_wait(drain, 0, abort_flag, err, kDevErrTimeoutDrain);
        }
    } else {
        // ------------------------------------------------------------ workers
        const int g = warp / 4;
        const int t = threadIdx.x & (kTileN - 1);  // row within the tile == TMEM lane
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        uint8_t* a_base = smem + C::kOffA;
        float acc[MT];
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        bool ok = true;
        float S_prev = 0.f;
        int nu = 0;  // uses issued by this group

        auto epilogue = [&](int v, float Sv) {
            const int s = v & 1, gs = g * kSlots + s;
            const int li = g + 2 * v;
            if (ok) ok = mbar_wait(&mma_done[gs], (v >> 1) & 1, abort_flag, err, kDevErrTimeoutMma);
            tc_fence_after();
            const float* dxp = dx_tile + ((int64_t)p0 * kSubPerPair + li) * MT;
#pragma unroll
            for (int c = 0; c < MT / 16; ++c) {
                uint32_t r[16];
                tmem_ld16(tmem + lane_base + (uint32_t)(gs * MT + 16 * c), r);
                tc_wait_ld();
                if (c == MT / 16 - 1) {
                    tc_fence_before();
                    mbar_arrive(&d_free[gs]);
                }
#pragma unroll
                for (int k = 0; k < 16; k += 4) {
                    const float4 d4 = __ldg(reinterpret_cast<const float4*>(dxp + 16 * c + k));
                    const float2 s01 = __fmul2_rn(make_float2(Sv, Sv), make_float2(d4.x, d4.y));
                    const float2 s23 = __fmul2_rn(make_float2(Sv, Sv), make_float2(d4.z, d4.w));
                    float2 a01 = make_float2(acc[16 * c + k], acc[16 * c + k + 1]);
                    float2 a23 = make_float2(acc[16 * c + k + 2], acc[16 * c + k + 3]);
                    a01 = __ffma2_rn(make_float2(__uint_as_float(r[k]), __uint_as_float(r[k + 1])), s01, a01);
                    a23 = __ffma2_rn(make_float2(__uint_as_float(r[k + 2]), __uint_as_float(r[k + 3])), s23, a23);
                    acc[16 * c + k] = a01.x;
                    acc[16 * c + k + 1] = a01.y;
                    acc[16 * c + k + 2] = a23.x;
                    acc[16 * c + k + 3] = a23.y;
                }
            }
        };

        for (int li = g; li < nsub; li += kGroups) {
            const int u = li >> 1, s = u & 1, gs = g * kSlots + s;
            const int ps = li / kSubPerPair, jj = li % kSubPerPair, wslot = ps % C::kNW;
            if (ok && jj < kGroups)
                ok = mbar_wait(&w_full[wslot], (ps / C::kNW) & 1, abort_flag, err, kDevErrTimeoutW);
            // Row t's bytes of super-block jj/8 in the staged pair.
            const uint8_t* rowp = smem + C::kOffW + wslot * kWStageBytes + t * kPairBytes +
                                  (jj / kSubPerBlock) * kBlockBytes;
            const int j = jj % kSubPerBlock;
            const uint2 hdr = *reinterpret_cast<const uint2*>(rowp);
            const uint2 q01 = *reinterpret_cast<const uint2*>(rowp + 8 + 16 * j);
            const uint2 q23 = *reinterpret_cast<const uint2*>(rowp + 16 + 16 * j);
            if (jj >= kSubPerPair - kGroups) mbar_arrive(&w_empty[wslot]);
            const float S = iq4xs_scale(hdr.x, hdr.y, j);
            uint32_t h[16];
            decode_f16x2(q01.x, h + 0);
            decode_f16x2(q01.y, h + 4);
            decode_f16x2(q23.x, h + 8);
            decode_f16x2(q23.y, h + 12);
            // A[g][s] was last read by the MMA of use u-2, whose completion the
            // epilogue of use u-2 (run in the previous iteration) waited for.
            uint8_t* ap = a_base + gs * kASubBytes + t * 16;
#pragma unroll
            for (int c = 0; c < kChunksPerSub; ++c)
                *reinterpret_cast<uint4*>(ap + c * kALbo) =
                    make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
            fence_proxy_async_smem();
            mbar_arrive(&a_full[gs]);
            if (u >= 1) epilogue(u - 1, S_prev);
            S_prev = S;
            nu = u + 1;
        }
        if (nu >= 1) epilogue(nu - 1, S_prev);

        // Combine the two groups' partial sums in shared memory (the W ring
        // is idle once every worker has passed the first barrier).
        float* red = reinterpret_cast<float*>(smem + C::kOffW);
        named_barrier_sync(1, kTcWorkerWarps * 32);
        if (g == 1) {
#pragma unroll
            for (int m = 0; m < MT; ++m) red[t * C::kRedStride + m] = acc[m];
        }
        named_barrier_sync(1, kTcWorkerWarps * 32);
        if (g == 0) {
            const int64_t mrows = M - (int64_t)z * MT;
#pragma unroll
            for (int m = 0; m < MT; ++m) {
                const float v = acc[m] + red[t * C::kRedStride + m];
                if (S == 1) {
                    if (m < mrows && n0 + t < N) y[((int64_t)z * MT + m) * ldy + n0 + t] = v;
                } else {
                    red[t * C::kRedStride + m] = v;
                }
            }
        }
    }

    if (S > 1) {
        // Split-K reduction over the cluster through distributed shared memory:
        // CTA `rank` sums rows [rank*128/S, (rank+1)*128/S) over all CTAs in
        // rank order (deterministic) and writes them.
        cluster_sync_all();
        if (warp < kTcWorkerWarps) {
            const uint32_t red_s = smem_u32(smem + C::kOffW);
            const int r0 = (int)(kTileN * rank / S), r1 = (int)(kTileN * (rank + 1) / S);
            const int64_t mrows = M - (int64_t)z * MT;
            const int rows = r1 - r0;
            for (int e = threadIdx.x; e < rows * MT; e += kTcWorkerWarps * 32) {
                const int row = r0 + e % rows, m = e / rows;
                float v = 0.f;
                for (int q = 0; q < S; ++q)
                    v += ld_dsmem_f32(red_s + (uint32_t)((row * C::kRedStride + m) * 4), (uint32_t)q);
                if (m < mrows && n0 + row < N) y[((int64_t)z * MT + m) * ldy + n0 + row] = v;
            }
        }
        cluster_sync_all();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == kTcIssuerWarp) {
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
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = (unsigned)S;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
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
