// quantize.cu -- Q8_1 activation quantization (V100TPS engine page, kernel
// table at M=64: the activations enter the batched matmul through
// quantize_q8_1).  Per block of 32 values: amax = max|x|, d = amax/127,
// q = round(x/d) (ties away from zero), s = d*sum(q); d and s stored as fp16.
//
// One thread owns 4 consecutive values (one float4 load), 8 threads own a
// Q8_1 block, a CTA owns one span of 1024 values of one row.  The kernel
// optionally also writes the prepared tensor-core operand: each dequantized
// value q*d_h times the span's power of two 2^-e as an exact pair of fp16
// values (hi + lo), in the K-permuted, tiled order the faster form of the
// tcgen05 matmul consumes, and the span's 2^e.
#include "internal.cuh"

namespace iq4xs {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kElemsPerThread = 4;
constexpr int kElemsPerCta = kQuantThreads * kElemsPerThread;  // 1024
constexpr int kThreadsPerBlock = kSub / kElemsPerThread;        // 8
static_assert(kThreadsPerBlock == 8, "8 lanes per Q8_1 block: xor-shuffles 1, 2, 4");
static_assert(kElemsPerCta == kScaleSpan, "one CTA per activation scale span");

// grid: x = ceil(K / 1024), y = rows (M, or the padded tile rows when the
// tensor-core operand is requested).  K % 256 == 0, so a warp's 128 values
// are either all inside K or all outside it.
template <bool kTc>
__global__ void __launch_bounds__(kQuantThreads)
    quantize_q8_1_kernel(const float* __restrict__ x, int64_t M, int64_t K, int64_t ldx,
                         int8_t* __restrict__ qs, __half2* __restrict__ ds,
                         uint4* __restrict__ qh, float* __restrict__ spanscale, int MT, int* err) {
    // The next grid (the matmul) may launch at once: it reads qs/ds only
    // after its own wait for this grid, and this grid completes only after
    // the preceding one (whose CTAs are all resident by now: this grid
    // launched when each had started).  The matmul's CTAs take SMs as the
    // preceding grid's leave and stream their weights meanwhile.  x may come
    // from the preceding grid, and qs/ds/the operand may still be read by it:
    // wait for it before reading or writing anything.  Its lines are only
    // requested into L2 before the wait: a prefetch is a hint that reads no
    // value, and L2 is where the preceding grid's writes land.
    griddep_launch_dependents();
    const int64_t m = blockIdx.y;
    const int64_t e0 = (int64_t)blockIdx.x * kElemsPerCta + threadIdx.x * kElemsPerThread;
    const bool live = e0 < K;  // whole warps (see above)
    if (live && m < M) asm volatile("prefetch.global.L2 [%0];" ::"l"(x + m * ldx + e0));
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int l8 = lane & 7;  // position of this thread inside its Q8_1 block
    const Bc bc = bc_open(err);
    const int64_t nsub = K / kSub;

    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (live && m < M && bc_global(bc, x + m * ldx + e0, 16, x, ((M - 1) * ldx + K) * 4, kBcQuantX))
        v = __ldg(reinterpret_cast<const float4*>(x + m * ldx + e0));

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

    if (live && m < M) {
        const uint32_t packed = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
                                ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
        if (bc_global(bc, qs + m * K + e0, 4, qs, M * K, kBcQuantQs))
            *reinterpret_cast<uint32_t*>(qs + m * K + e0) = packed;
        if (l8 == 0 && bc_global(bc, ds + m * nsub + blk, 4, ds, M * nsub * 4, kBcQuantDs))
            ds[m * nsub + blk] = __halves2half2(d_h, __float2half_rn(d * (float)sum));
    }

    if constexpr (kTc) {
        // The span's largest stored scale -> its power of two: the smallest
        // e >= 0 with 127 * max(d_h) * 2^-e < 65504, so no hi overflows.
        __shared__ float s_warp[kQuantThreads / 32];
        float dmax = __half2float(d_h);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o));
        if (lane == 0) s_warp[threadIdx.x >> 5] = dmax;
        __syncthreads();
        dmax = s_warp[0];
#pragma unroll
        for (int w = 1; w < kQuantThreads / 32; ++w) dmax = fmaxf(dmax, s_warp[w]);
        int e = 0;
        float lim = 65504.0f / 127.0f;
        while (dmax >= lim && e < 64) {
            lim *= 2.0f;
            ++e;
        }
        const int64_t mt = m / MT;
        const int64_t r = m % MT;
        const int64_t span_i = (mt * tc_num_spans(K) + blockIdx.x) * MT + r;
        if (threadIdx.x == 0 && bc_global(bc, spanscale + span_i, 4, spanscale,
                                          tc_operand_total_bytes(M, K) - tc_qh_bytes(M, K), kBcQuantSpan))
            spanscale[span_i] = ldexpf(1.0f, e);
        // Element e of the block goes to K position 2*(e % 16) + e / 16.  The
        // thread holding e = 4*l8 .. 4*l8+3 (l8 < 4) pairs with lane ^ 4,
        // which holds e + 16, and writes one 16-byte chunk (8 positions) of
        // each plane.  q*dh is exact in fp32 (at most 19 significant bits),
        // as are the rounding to hi and the remainder lo.
        int p[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = __shfl_xor_sync(0xffffffffu, q[k], 4);
        if (live && l8 < 4) {
            const float dh = __half2float(d_h) * ldexpf(1.0f, -e);  // exact (power of two)
            __half hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float val = (float)((k & 1) ? p[k / 2] : q[k / 2]) * dh;
                hi[k] = __float2half_rn(val);
                lo[k] = __float2half_rn(val - __half2float(hi[k]));
            }
            uint4* sub = qh + (mt * nsub + blk) * (kPlanes * kChunksPerSub * MT);
            const int64_t op_bytes = tc_qh_bytes(M, K);
            if (bc_global(bc, sub + l8 * MT + r, 16, qh, op_bytes, kBcQuantOp))
                sub[l8 * MT + r] = *reinterpret_cast<const uint4*>(hi);
            if (bc_global(bc, sub + (kChunksPerSub + l8) * MT + r, 16, qh, op_bytes, kBcQuantOp))
                sub[(kChunksPerSub + l8) * MT + r] = *reinterpret_cast<const uint4*>(lo);
        }
    }
}

}  // namespace

cudaError_t launch_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs,
                                 void* ds, void* tc_operand, int* err, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(kQuantThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    __half2* d2 = reinterpret_cast<__half2*>(ds);
    const unsigned spans = (unsigned)tc_num_spans(K);
    if (tc_operand == nullptr) {
        cfg.gridDim = dim3(spans, (unsigned)M);
        return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<false>, x, M, K, ldx, qs, d2,
                                  (uint4*)nullptr, (float*)nullptr, 0, err);
    }
    const int MT = tc_mtile(M);
    cfg.gridDim = dim3(spans, (unsigned)(tc_num_mtiles(M) * MT));  // padding rows written as zeros
    uint8_t* op = reinterpret_cast<uint8_t*>(tc_operand);
    return cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<true>, x, M, K, ldx, qs, d2,
                              reinterpret_cast<uint4*>(op),
                              reinterpret_cast<float*>(op + tc_qh_bytes(M, K)), MT, err);
}

}  // namespace iq4xs
