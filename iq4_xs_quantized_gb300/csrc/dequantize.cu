// dequantize.cu -- IQ4_XS -> dense fp32 / bfloat16 (V100TPS engine page,
// kernel table at M=64: dequantize_block_iq4_xs writing the whole weight
// before a dense GEMM -- the baseline path the batched kernel replaces).
// weight = fp32(d) * (ls - 32) * kvalues_iq4nl[nibble], exact in fp32.
#include <cuda_bf16.h>

#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kDqThreads = 256;

// One thread per (row n, sub-block s): 32 outputs, written contiguously.
template <bool kBf16>
__global__ void __launch_bounds__(kDqThreads)
    dequantize_kernel(const uint8_t* __restrict__ w, int64_t N, int64_t K, void* __restrict__ out) {
    const int64_t nsub = K / kSub;
    const int64_t idx = (int64_t)blockIdx.x * kDqThreads + threadIdx.x;
    if (idx >= N * nsub) return;
    const int64_t n = idx / nsub;
    const int64_t s = idx % nsub;
    const int j = (int)(s % kSubPerBlock);
    const uint8_t* blk = w + (n * (K / kQK) + s / kSubPerBlock) * kBlockBytes;
    const uint2 hdr = __ldg(reinterpret_cast<const uint2*>(blk));  // 8-byte aligned
    const uint2 q01 = __ldg(reinterpret_cast<const uint2*>(blk + 8 + 16 * j));
    const uint2 q23 = __ldg(reinterpret_cast<const uint2*>(blk + 16 + 16 * j));
    const float S = iq4xs_scale(hdr.x, hdr.y, j);
    const uint32_t words[4] = {q01.x, q01.y, q23.x, q23.y};
    float v[32];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        uint32_t lo4, hi4;
        decode_s8(words[c], lo4, hi4);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[4 * c + k] = S * (float)(int8_t)(lo4 >> (8 * k));
            v[16 + 4 * c + k] = S * (float)(int8_t)(hi4 >> (8 * k));
        }
    }
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

}  // namespace

cudaError_t launch_dequantize(const void* w, int64_t N, int64_t K, void* out, int out_dtype,
                              cudaStream_t stream) {
    const int64_t total = N * (K / kSub);
    const unsigned grid = (unsigned)((total + kDqThreads - 1) / kDqThreads);
    if (out_dtype == 1)
        dequantize_kernel<true><<<grid, kDqThreads, 0, stream>>>(
            reinterpret_cast<const uint8_t*>(w), N, K, out);
    else
        dequantize_kernel<false><<<grid, kDqThreads, 0, stream>>>(
            reinterpret_cast<const uint8_t*>(w), N, K, out);
    return cudaGetLastError();
}

}  // namespace iq4xs
