// matmul_dp4a.cu -- small-M IQ4_XS x Q8_1 matmul on the CUDA cores.
//
// V100TPS engine page: the mmvq table (per-row mul_mat_vec_q, cost linear in
// M) and the tile-geometry passage (vec_dot_iq4_xs_q8_1: int8 dot products of
// decoded nibbles with Q8_1 codes, scaled by d_w*(ls-32)*d_x).  Here one warp
// streams R weight rows; lane l takes sub-blocks l, l+32, ... of every row, so
// a warp reads 4 consecutive super-blocks (544 contiguous bytes) per row per
// step.  Nibbles decode to int8 through the codebook held in registers
// (prmt), 8 dp4a give the exact int32 sub-block dot, and one fp32 FMA per
// (row, m, sub-block) scales it in.  Lanes are reduced with shuffles.
#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kDp4aThreads = 256;
constexpr int kDp4aRows = 2;  // weight rows per warp
constexpr int kWarpsPerCta = kDp4aThreads / 32;

__device__ __forceinline__ int dp4a(uint32_t a, uint32_t b, int c) {
    return __dp4a((int)a, (int)b, c);
}

template <int MC>  // activation rows per pass
__global__ void __launch_bounds__(kDp4aThreads)
    matmul_dp4a_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K,
                       const int8_t* __restrict__ qs, const __half2* __restrict__ ds, int64_t M,
                       float* __restrict__ y, int64_t ldy) {
    const int lane = threadIdx.x & 31;
    const int64_t warp = (int64_t)blockIdx.x * kWarpsPerCta + (threadIdx.x >> 5);
    const int64_t n0 = warp * kDp4aRows;
    if (n0 >= N) return;  // whole warp
    const int64_t nsub = K / kSub;
    const int64_t row_bytes = (K / kQK) * kBlockBytes;

    for (int64_t m0 = 0; m0 < M; m0 += MC) {
        float acc[kDp4aRows][MC];
#pragma unroll
        for (int r = 0; r < kDp4aRows; ++r)
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) acc[r][mi] = 0.f;

        for (int64_t s = lane; s < nsub; s += 32) {
            // Q8_1 codes and scales of this sub-block for MC activation rows.
            uint4 qa[MC][2];
            float dx[MC];
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) {
                if (m0 + mi < M) {
                    const uint4* qp = reinterpret_cast<const uint4*>(qs + (m0 + mi) * K + s * kSub);
                    qa[mi][0] = __ldg(qp);
                    qa[mi][1] = __ldg(qp + 1);
                    dx[mi] = __low2float(__ldg(ds + (m0 + mi) * nsub + s));
                } else {
                    qa[mi][0] = qa[mi][1] = make_uint4(0, 0, 0, 0);
                    dx[mi] = 0.f;
                }
            }
            const int j = (int)(s % kSubPerBlock);
            const int64_t blk_off = (s / kSubPerBlock) * kBlockBytes;
#pragma unroll
            for (int r = 0; r < kDp4aRows; ++r) {
                const int64_t n = n0 + r;
                if (n >= N) break;
                const uint8_t* blk = w + n * row_bytes + blk_off;
                const uint2 hdr = __ldg(reinterpret_cast<const uint2*>(blk));
                const uint2 q01 = __ldg(reinterpret_cast<const uint2*>(blk + 8 + 16 * j));
                const uint2 q23 = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 16 * j));
                const float S = iq4xs_scale(hdr.x, hdr.y, j);
                uint32_t lo[4], hi[4];
                decode_s8(q01.x, lo[0], hi[0]);
                decode_s8(q01.y, lo[1], hi[1]);
                decode_s8(q23.x, lo[2], hi[2]);
                decode_s8(q23.y, lo[3], hi[3]);
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
#pragma unroll
        for (int r = 0; r < kDp4aRows; ++r)
#pragma unroll
            for (int mi = 0; mi < MC; ++mi) {
                float v = acc[r][mi];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                acc[r][mi] = v;
            }
        if (lane == 0) {
#pragma unroll
            for (int r = 0; r < kDp4aRows; ++r)
#pragma unroll
                for (int mi = 0; mi < MC; ++mi)
                    if (n0 + r < N && m0 + mi < M) y[(m0 + mi) * ldy + n0 + r] = acc[r][mi];
        }
    }
}

}  // namespace

cudaError_t launch_matmul_dp4a(const void* w, int64_t N, int64_t K, const int8_t* qs,
                               const void* ds, int64_t M, float* y, int64_t ldy,
                               cudaStream_t stream) {
    const int64_t warps = (N + kDp4aRows - 1) / kDp4aRows;
    const unsigned grid = (unsigned)((warps + kWarpsPerCta - 1) / kWarpsPerCta);
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(w);
    const __half2* d2 = reinterpret_cast<const __half2*>(ds);
    if (M == 1)
        matmul_dp4a_kernel<1><<<grid, kDp4aThreads, 0, stream>>>(wb, N, K, qs, d2, M, y, ldy);
    else if (M == 2)
        matmul_dp4a_kernel<2><<<grid, kDp4aThreads, 0, stream>>>(wb, N, K, qs, d2, M, y, ldy);
    else if (M <= 4)
        matmul_dp4a_kernel<4><<<grid, kDp4aThreads, 0, stream>>>(wb, N, K, qs, d2, M, y, ldy);
    else
        matmul_dp4a_kernel<8><<<grid, kDp4aThreads, 0, stream>>>(wb, N, K, qs, d2, M, y, ldy);
    return cudaGetLastError();
}

}  // namespace iq4xs
