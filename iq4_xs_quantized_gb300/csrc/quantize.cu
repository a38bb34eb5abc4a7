// quantize.cu -- Q8_1 activation quantization (V100TPS engine page, kernel
// table at M=64: the activations enter the batched matmul through
// quantize_q8_1).  Per block of 32 values: amax = max|x|, d = amax/127,
// q = round(x/d) (ties away from zero), s = d*sum(q); d and s stored as fp16.
//
// One thread owns 4 consecutive values (one float4 load), 8 threads own a
// Q8_1 block, a CTA owns 1024 values of one row.  Both matmul paths read the
// two arrays it writes as they are.
#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kElemsPerThread = 4;
constexpr int kElemsPerCta = kQuantThreads * kElemsPerThread;  // 1024
constexpr int kThreadsPerBlock = kSub / kElemsPerThread;        // 8
static_assert(kThreadsPerBlock == 8, "8 lanes per Q8_1 block: xor-shuffles 1, 2, 4");

// grid: x = ceil(K / 1024), y = rows.  K % 256 == 0, so a warp's 128 values
// are either all inside K or all outside it.
__global__ void __launch_bounds__(kQuantThreads)
    quantize_q8_1_kernel(const float* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                         int8_t* __restrict__ qs, __half2* __restrict__ ds) {
    // x may come from the preceding grid, and qs/ds may still be read by it:
    // wait for it, then let the next grid start launching.
    griddep_wait();
    griddep_launch_dependents();
    const int64_t m = blockIdx.y;
    const int64_t e0 = (int64_t)blockIdx.x * kElemsPerCta + threadIdx.x * kElemsPerThread;
    const bool live = e0 < K;  // whole warps (see above)
    const int lane = threadIdx.x & 31;
    const int l8 = lane & 7;  // position of this thread inside its Q8_1 block

    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live) v = __ldg(reinterpret_cast<const float4*>(x + m * ldx + e0));

    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const float d = __fdiv_rn(amax, 127.0f);
    int q[4] = {0, 0, 0, 0};
    if (d != 0.0f) {
        q[0] = (int)roundf(__fdiv_rn(v.x, d));
        q[1] = (int)roundf(__fdiv_rn(v.y, d));
        q[2] = (int)roundf(__fdiv_rn(v.z, d));
        q[3] = (int)roundf(__fdiv_rn(v.w, d));
    }
    int sum = q[0] + q[1] + q[2] + q[3];
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    sum += __shfl_xor_sync(0xffffffffu, sum, 4);
    const __half d_h = __float2half_rn(d);
    const int64_t blk = e0 / kSub;  // global Q8_1 block (= sub-block) index

    if (live) {
        const uint32_t packed = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
                                ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
        *reinterpret_cast<uint32_t*>(qs + m * K + e0) = packed;
        if (l8 == 0) ds[m * (K / kSub) + blk] = __halves2half2(d_h, __float2half_rn(d * (float)sum));
    }
}

}  // namespace

cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs,
                                 void* ds, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kQuantThreads);
    cfg.gridDim = dim3((unsigned)((K + kElemsPerCta - 1) / kElemsPerCta), (unsigned)M);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel, x, M, K, ldx, qs, reinterpret_cast<__half2*>(ds));
}

}  // namespace iq4xs
