// dequantize.cu -- IQ4_XS / Q4_0 / IQ4_NL -> dense fp32 / bfloat16
// (V100TPS engine page, kernel table at M=64: dequantize_block_iq4_xs
// writing the whole weight before a dense GEMM -- the baseline path the
// batched kernel replaces).  weight = sub-block scale * nibble value, exact
// in fp32: IQ4_XS fp32(d) * (ls - 32) * kvalues_iq4nl[q]; Q4_0 fp32(d) * (q - 8);
// IQ4_NL fp32(d) * kvalues_iq4nl[q].
#include <cuda_bf16.h>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kDqThreads = 256;

// One thread per (row n, sub-block s): 32 outputs, written contiguously.
template <bool kBf16, int WT>
__global__ void __launch_bounds__(kDqThreads)
    dequantize_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K, void* __restrict__ out, int* err) {
    const int64_t nsub = K / kSub;
    const int64_t idx = (int64_t)blockIdx.x * kDqThreads + threadIdx.x;
    if (idx >= N * nsub) return;
    const int64_t n = idx / nsub;
    const int64_t s = idx % nsub;
    const Bc bc = bc_open(err);
    uint32_t raw[6] = {0, 0, 0, 0, 0, 0}, words[4];
    const uint8_t* row = w + n * wt_row_bytes(WT, K);
    if (wt_sub_in_bounds<WT>(bc, row, s, w, N * wt_row_bytes(WT, K), kBcDqW)) wt_load_sub<WT>(row, s, raw);
    const float S = wt_unpack_sub<WT>(raw, s, words);
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t lo4, hi4;
        decode_s8<WT>(words[c], lo4, hi4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[4 * c + k] = S * (float)(int8_t)(lo4 >> (8 * k));
            v[16 + 4 * c + k] = S * (float)(int8_t)(hi4 >> (8 * k));
        }
    }
    if (!bc_global(bc, reinterpret_cast<const char*>(out) + (n * K + s * kSub) * (kBf16 ? 2 : 4),
                   kSub * (kBf16 ? 2 : 4), out, N * K * (kBf16 ? 2 : 4), kBcDqOut))
        return;
    if (kBf16) {
        __nv_bfloat16* o = reinterpret_cast<__nv_bfloat16*>(out) + n * K + s * kSub;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            __nv_bfloat16 b[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) b[k] = __float2bfloat16_rn(v[8 * c + k]);
            reinterpret_cast<uint4*>(o)[c] = *reinterpret_cast<const uint4*>(b);
        }
    } else {
        float4* o = reinterpret_cast<float4*>(reinterpret_cast<float*>(out) + n * K + s * kSub);
#pragma unroll
        for (int c = 0; c < 8; ++c)
            o[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
}

template <int WT>
void launch_dq(const uint8_t* w, int64_t N, int64_t K, void* out, int out_dtype, unsigned grid,
               int* err, cudaStream_t stream) {
    if (out_dtype == 1)
        dequantize_kernel<true, WT><<<grid, kDqThreads, 0, stream>>>(w, N, K, out, err);
    else
        dequantize_kernel<false, WT><<<grid, kDqThreads, 0, stream>>>(w, N, K, out, err);
}

}  // namespace

cudaError_t launch_dequantize(const void* w, int wt, int64_t N, int64_t K, void* out,
                              int out_dtype, int* err, cudaStream_t stream) {
    const int64_t total = N * (K / kSub);
    const unsigned grid = (unsigned)((total + kDqThreads - 1) / kDqThreads);
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(w);
    switch (wt) {
        case kWtIQ4XS: launch_dq<kWtIQ4XS>(wb, N, K, out, out_dtype, grid, err, stream); break;
        case kWtQ4_0: launch_dq<kWtQ4_0>(wb, N, K, out, out_dtype, grid, err, stream); break;
        case kWtIQ4NL: launch_dq<kWtIQ4NL>(wb, N, K, out, out_dtype, grid, err, stream); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace iq4xs
