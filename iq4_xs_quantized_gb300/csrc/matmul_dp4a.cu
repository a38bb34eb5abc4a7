// matmul_dp4a.cu -- small-M IQ4_XS x Q8_1 matmul on the CUDA cores.
//
// V100TPS engine page: the mmvq table (per-row mul_mat_vec_q, cost linear in
// M) and the tile-geometry passage (vec_dot_iq4_xs_q8_1: int8 dot products of
// decoded nibbles with Q8_1 codes, scaled by d_w*(ls-32)*d_x).  Here one warp
// streams kRows weight rows; lane l takes sub-blocks l, l+32, ..., so a warp
// reads 4 consecutive super-blocks (544 contiguous bytes) per row per step.
// All weight loads of kIters steps are issued before any arithmetic, so each
// SM keeps tens of KB in flight (a 4096 x 4096 matrix is ~58 KB per SM).
// Nibbles decode to int8 through the codebook held in registers (prmt),
// 8 dp4a give the exact int32 sub-block dot, and one fp32 FMA per
// (row, m, sub-block) scales it in.  Lanes are reduced with shuffles.
#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kDp4aThreads = 256;
constexpr int kRows = 2;   // weight rows per warp
constexpr int kWarpsPerCta = kDp4aThreads / 32;
// Launch shapes, chosen from the grid size G (CTAs) against the SM count:
// resident CTAs per SM x sub-block steps whose loads each warp keeps in
// flight (registers bound their product).
//   shape 0, G <= 2 SMs (one wave, e.g. 4096 rows): 2 CTAs, 4 steps at M=1.
//   shape 1, G <= 3 SMs (5120-6144 rows): 3 CTAs x 2 steps at M=1, so that
//            every CTA is resident at once, spread over the SMs.
//   shape 2, more (several waves): 4 CTAs x 1 step at M=1, so that CTAs of
//            the next wave are already streaming while the current ones
//            decode and reduce.
// M=2 takes 3 CTAs x 1 step from shape 1 on; M >= 3 (ALU-bound) keeps
// shape 0.  Measured on GB300 (us, shape 0 -> chosen shape): M=1 5120x5120
// 8.8 -> 6.8 (shape 1), 5120x17408 26.6 -> 20.5 (1), 34816x5120 35.4 ->
// 29.1 (2); M=2 34816x5120 40.0 -> 36.2.
template <int MC>
constexpr int max_shape() { return MC == 1 ? 2 : (MC == 2 ? 1 : 0); }
template <int MC, int S>
constexpr int ctas_per_sm() { return S == 0 ? 2 : (MC == 1 ? (S == 1 ? 3 : 4) : 3); }
template <int MC, int S>
constexpr int iters_for() {
    return S == 0 ? (MC == 1 ? 4 : (MC <= 4 ? 2 : 1)) : (MC == 1 ? (S == 1 ? 2 : 1) : 1);
}

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}

// Rows [0, M) of x against the warp's kRows weight rows n0.. of W (format
// WT), MC activation rows per pass.  `waited`: the wait for the preceding
// grid (which wrote the activations) has been done already.  The buffers'
// extents (checked in the bounds-checked build) follow from N, K, M, ldy.
template <int MC, int WT, int kIters>
__device__ __forceinline__ void dp4a_rows(const uint8_t* __restrict__ w, int64_t N, int64_t K,
                                          const int8_t* __restrict__ qs,
                                          const __half2* __restrict__ ds, int64_t M,
                                          float* __restrict__ y, int64_t ldy, int64_t n0, int lane,
                                          bool waited, const Bc& bc) {
    const int64_t nsub = K / kSub;
    const int64_t row_bytes = wt_row_bytes(WT, K);
    const int64_t w_ext = N * row_bytes, qs_ext = M * K, ds_ext = M * nsub * 4;
    const int64_t y_ext = ((M - 1) * ldy + N) * 4;
    for (int64_t m0 = 0; m0 < M; m0 += MC) {
        float acc[kRows][MC];
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) acc[r][mi] = 0.f;

        for (int64_t sb = 0; sb < nsub; sb += 32 * kIters) {
            // Weight bytes (read-only model state) for kIters steps, all in flight.
            uint32_t raw[kIters][kRows][6];
#pragma unroll
            for (int it = 0; it < kIters; ++it) {
                const int64_t s = sb + lane + 32 * it;
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    if (s < nsub && n0 + r < N &&
                        wt_sub_in_bounds<WT>(bc, w + (n0 + r) * row_bytes, s, w, w_ext, kBcDp4aW)) {
                        wt_load_sub<WT>(w + (n0 + r) * row_bytes, s, raw[it][r]);
                    } else {
#pragma unroll
                        for (int k = 0; k < 6; ++k) raw[it][r][k] = 0;
                    }
                }
            }
            // The activations come from the preceding grid.
            if (!waited) {
                griddep_wait();
                waited = true;
            }
            // Small MC: every step's activation codes are loaded up front so
            // their latency overlaps the weight loads still in flight.
            constexpr int kPre = (MC <= 2) ? kIters : 1;
            uint4 qpre[kPre][MC][2];
            float dpre[kPre][MC];
            auto load_act = [&](int it, uint4 (&qa)[MC][2], float (&dx)[MC]) {
                const int64_t s = sb + lane + 32 * it;
#pragma unroll
                for (int mi = 0; mi < MC; ++mi) {
                    if (s < nsub && m0 + mi < M &&
                        bc_global(bc, qs + (m0 + mi) * K + s * kSub, kSub, qs, qs_ext, kBcDp4aQs) &&
                        bc_global(bc, ds + (m0 + mi) * nsub + s, 4, ds, ds_ext, kBcDp4aDs)) {
                        const uint4* qp = reinterpret_cast<const uint4*>(qs + (m0 + mi) * K + s * kSub);
                        qa[mi][0] = __ldg(qp);
                        qa[mi][1] = __ldg(qp + 1);
                        dx[mi] = __low2float(__ldg(ds + (m0 + mi) * nsub + s));
                    } else {
                        qa[mi][0] = qa[mi][1] = make_uint4(0, 0, 0, 0);
                        dx[mi] = 0.f;
                    }
                }
            };
            if (kPre == kIters) {
#pragma unroll
                for (int it = 0; it < kPre; ++it) load_act(it, qpre[it], dpre[it]);
            }
#pragma unroll
            for (int it = 0; it < kIters; ++it) {
                const int64_t s = sb + lane + 32 * it;
                if (s >= nsub) break;
                const int pi = (kPre == kIters) ? it : 0;
                if (kPre != kIters) load_act(it, qpre[0], dpre[0]);
                const uint4 (&qa)[MC][2] = qpre[pi];
                const float (&dx)[MC] = dpre[pi];
#pragma unroll
                for (int r = 0; r < kRows; ++r) {
                    uint32_t q[4];
                    const float S = wt_unpack_sub<WT>(raw[it][r], s, q);
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int c = 0; c < 4; ++c) decode_s8<WT>(q[c], lo[c], hi[c]);
#pragma unroll
                    for (int mi = 0; mi < MC; ++mi) {
                        // elements 4c..4c+3 <-> code word c; elements 16+4c.. <-> word 4+c
                        int P = dp4a(lo[0], qa[mi][0].x, 0);
                        P = dp4a(lo[1], qa[mi][0].y, P);
                        P = dp4a(lo[2], qa[mi][0].z, P);
                        P = dp4a(lo[3], qa[mi][0].w, P);
                        P = dp4a(hi[0], qa[mi][1].x, P);
                        P = dp4a(hi[1], qa[mi][1].y, P);
                        P = dp4a(hi[2], qa[mi][1].z, P);
                        P = dp4a(hi[3], qa[mi][1].w, P);
                        acc[r][mi] = fmaf((float)P, S * dx[mi], acc[r][mi]);
                    }
                }
            }
        }
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) {
                float v = acc[r][mi];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][mi] = v;
            }
        // Lane r*MC + mi writes one output (kRows * MC <= 32).
#pragma unroll
        for (int r = 0; r < kRows; ++r)
#pragma unroll
            for (int mi = 0; mi < MC; ++mi)
                if (lane == r * MC + mi && n0 + r < N && m0 + mi < M &&
                    bc_global(bc, y + (m0 + mi) * ldy + n0 + r, 4, y, y_ext, kBcDp4aY))
                    y[(m0 + mi) * ldy + n0 + r] = acc[r][mi];
    }
}

template <int MC, int WT, int S>  // activation rows per pass, weight format, launch shape
__global__ void __launch_bounds__(kDp4aThreads, ctas_per_sm<MC, S>())
    matmul_dp4a_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K,
                       const int8_t* __restrict__ qs, const __half2* __restrict__ ds, int64_t M,
                       float* __restrict__ y, int64_t ldy, int* err) {
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t n0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * kRows;
    if (n0 >= N) return;  // whole warp
    const Bc bc = bc_open(err);
    dp4a_rows<MC, WT, iters_for<MC, S>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, false, bc);
}

// Grouped (mixture-of-experts) form: G experts, expert g with its own W at
// w + g * expert_stride and the activation / output rows
// [row_offsets[g], row_offsets[g+1]) (a device array, read after the wait for
// the preceding grid, which may have produced it).  blockIdx.y = k takes the
// k-th expert that has rows; the host sizes the grid from the total row
// count, so slots past the last non-empty expert exit at once.  The batch
// width follows each expert's own row count, so an expert with one row costs
// what a one-row matmul costs.  kNarrow (decode batches: at most two rows per
// routed expert on average): batch widths of one and two rows only (larger
// experts take several passes), which fit three CTAs per SM -- the launch
// shape that keeps the next wave streaming on these many-wave grids.  A row's
// result does not depend on the batch width (each lane sums its sub-blocks
// in the same order), so both forms give the same bits.
template <bool kNarrow, int WT>
__global__ void __launch_bounds__(kDp4aThreads, kNarrow ? 3 : 2)
    matmul_dp4a_grouped_kernel(const uint8_t* __restrict__ w, int64_t expert_stride, int64_t G,
                               int64_t N, int64_t K, const int8_t* __restrict__ qs,
                               const __half2* __restrict__ ds, const int32_t* __restrict__ row_offsets,
                               int64_t total_rows, float* __restrict__ y, int64_t ldy, int* err) {
    griddep_launch_dependents();
    const int lane = threadIdx.x & 31;
    const int64_t n0 = ((int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5)) * kRows;
    if (n0 >= N) return;  // whole warp
    const Bc bc = bc_open(err);
    griddep_wait();
    // The k-th non-empty expert: the offsets of 128 experts are loaded at
    // once (independent loads), then a ballot per 32 of them.
    int64_t g = -1;
    uint32_t k = blockIdx.y;
    for (int64_t base = 0; base < G && g < 0; base += 4 * 32) {
        int32_t lo[4], hi[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int64_t e = base + 32 * j + lane;
            const bool in = e < G && bc_global(bc, row_offsets + e, 8, row_offsets, (G + 1) * 4, kBcDp4aOffsets);
            lo[j] = in ? __ldg(row_offsets + e) : 0;
            hi[j] = in ? __ldg(row_offsets + e + 1) : 0;
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t mask = __ballot_sync(0xffffffffu, hi[j] > lo[j]);
            const uint32_t cnt = __popc(mask);
            if (g < 0) {
                if (k < cnt) g = base + 32 * j + (int64_t)__fns(mask, 0, (int)k + 1);
                else k -= cnt;
            }
        }
    }
    if (g < 0) return;  // fewer non-empty experts than slots (whole warp)
    const int64_t r0 = row_offsets[g], M = row_offsets[g + 1] - r0;
    if (!bc_range(bc, r0, M, total_rows, kBcDp4aRows)) return;  // offsets outside the rows of y
    w += g * expert_stride;
    qs += r0 * K;
    ds += r0 * (K / kSub);
    y += r0 * ldy;
    constexpr int X = WT;
    if constexpr (kNarrow) {
        if (M == 1) dp4a_rows<1, X, iters_for<1, 1>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
        else dp4a_rows<2, X, iters_for<2, 1>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
    } else {
        if (M == 1) dp4a_rows<1, X, iters_for<1, 0>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
        else if (M == 2) dp4a_rows<2, X, iters_for<2, 0>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
        else if (M <= 4) dp4a_rows<4, X, iters_for<4, 0>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
        else dp4a_rows<8, X, iters_for<8, 0>()>(w, N, K, qs, ds, M, y, ldy, n0, lane, true, bc);
    }
}

cudaLaunchConfig_t dp4a_config(int64_t N, unsigned slots, cudaStream_t stream,
                               cudaLaunchAttribute* attr) {
    const int64_t warps = (N + kRows - 1) / kRows;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + kWarpsPerCta - 1) / kWarpsPerCta), slots);
    cfg.blockDim = dim3(kDp4aThreads);
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

template <int MC, int WT>
cudaError_t launch_mc(const uint8_t* w, int64_t N, int64_t K, const int8_t* qs, const __half2* ds,
                      int64_t M, float* y, int64_t ldy, int* err, int num_sms, cudaStream_t stream) {
    static_assert(kRows * MC <= 32, "one output per lane");
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = dp4a_config(N, 1, stream, attr);
    const int64_t G = cfg.gridDim.x, sms = num_sms > 0 ? num_sms : 1;
    const int shape = G <= 2 * sms ? 0 : (G <= 3 * sms ? 1 : 2);
    if constexpr (max_shape<MC>() >= 2)
        if (shape >= 2)
            return cudaLaunchKernelEx(&cfg, matmul_dp4a_kernel<MC, WT, 2>, w, N, K, qs, ds, M, y, ldy, err);
    if constexpr (max_shape<MC>() >= 1)
        if (shape >= 1)
            return cudaLaunchKernelEx(&cfg, matmul_dp4a_kernel<MC, WT, 1>, w, N, K, qs, ds, M, y, ldy, err);
    return cudaLaunchKernelEx(&cfg, matmul_dp4a_kernel<MC, WT, 0>, w, N, K, qs, ds, M, y, ldy, err);
}

template <int WT>
cudaError_t launch_wt(const uint8_t* w, int64_t N, int64_t K, const int8_t* qs, const __half2* ds,
                      int64_t M, float* y, int64_t ldy, int* err, int num_sms, cudaStream_t stream) {
    if (M == 1) return launch_mc<1, WT>(w, N, K, qs, ds, M, y, ldy, err, num_sms, stream);
    if (M == 2) return launch_mc<2, WT>(w, N, K, qs, ds, M, y, ldy, err, num_sms, stream);
    if (M <= 4) return launch_mc<4, WT>(w, N, K, qs, ds, M, y, ldy, err, num_sms, stream);
    return launch_mc<8, WT>(w, N, K, qs, ds, M, y, ldy, err, num_sms, stream);
}

}  // namespace

cudaError_t launch_matmul_dp4a(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs,
                               const void* ds, int64_t M, float* y, int64_t ldy, int* err,
                               int num_sms, cudaStream_t stream) {
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(w);
    const __half2* d2 = reinterpret_cast<const __half2*>(ds);
    switch (wt) {
        case kWtIQ4XS: return launch_wt<kWtIQ4XS>(wb, N, K, qs, d2, M, y, ldy, err, num_sms, stream);
        case kWtQ4_0: return launch_wt<kWtQ4_0>(wb, N, K, qs, d2, M, y, ldy, err, num_sms, stream);
        case kWtIQ4NL: return launch_wt<kWtIQ4NL>(wb, N, K, qs, d2, M, y, ldy, err, num_sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

namespace {

template <int WT>
cudaError_t launch_grouped_wt(const uint8_t* wb, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                              const int8_t* qs, const __half2* d2, const int32_t* row_offsets, int64_t total_rows,
                              float* y, int64_t ldy, int* err, cudaStream_t stream) {
    // at most min(G, total rows) experts have rows
    const unsigned slots = (unsigned)(G < total_rows ? G : total_rows);
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = dp4a_config(N, slots, stream, attr);
    if (total_rows <= 2 * (int64_t)slots)  // at most two rows per routed expert on average
        return cudaLaunchKernelEx(&cfg, matmul_dp4a_grouped_kernel<true, WT>, wb, expert_stride, G, N, K, qs, d2,
                                  row_offsets, total_rows, y, ldy, err);
    return cudaLaunchKernelEx(&cfg, matmul_dp4a_grouped_kernel<false, WT>, wb, expert_stride, G, N, K, qs, d2,
                              row_offsets, total_rows, y, ldy, err);
}

}  // namespace

cudaError_t launch_matmul_dp4a_grouped(const void* w, int wt, int64_t expert_stride, int64_t G, int64_t N,
                                       int64_t K, const int8_t* qs, const void* ds,
                                       const int32_t* row_offsets, int64_t total_rows, float* y,
                                       int64_t ldy, int* err, cudaStream_t stream) {
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(w);
    const __half2* d2 = reinterpret_cast<const __half2*>(ds);
    switch (wt) {
        case kWtIQ4XS:
            return launch_grouped_wt<kWtIQ4XS>(wb, expert_stride, G, N, K, qs, d2, row_offsets, total_rows, y, ldy,
                                               err, stream);
        case kWtQ4_0:
            return launch_grouped_wt<kWtQ4_0>(wb, expert_stride, G, N, K, qs, d2, row_offsets, total_rows, y, ldy,
                                              err, stream);
        case kWtIQ4NL:
            return launch_grouped_wt<kWtIQ4NL>(wb, expert_stride, G, N, K, qs, d2, row_offsets, total_rows, y, ldy,
                                               err, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace iq4xs
