// matmul_mma_b18.cu -- Q4_0 and IQ4_NL weights (18-byte blocks of 32: fp16 d,
// then 16 bytes of nibbles) on the warp-level MMA matmul of mma_kernel.cuh,
// dense and grouped (mixture of experts).
//
// The formats' definitions are the same as on the CUDA-core and tcgen05
// paths: a block's weight i is d * value[nibble i], value = nibble - 8 for
// Q4_0 and the 16-entry non-linear table for IQ4_NL, every value an integer
// with |value| <= 127, so a sub-block's two k16 MMAs leave the exact integer
// dot in the fp32 accumulator and only the scale-in d_w * d_x rounds.
//
// The kernel is the IQ4_XS one with the 18-byte layout (its stage row is 288
// bytes in two 144-byte boxes, the row scale is the block's d) and the
// format's values in the byte table.  The launch list is the IQ4_XS one, and
// the launch is chosen the same way: the measured IQ4_XS launch for the
// shape and tile height if the calibration installed one (the kernels differ
// only in the decode and 6 % more weight bytes), else the cost model with
// the larger stage rows weighed in.
#include "mma_kernel.cuh"

namespace iq4xs {
namespace {

template <int NT>
struct MmaConfigsB18;
template <>
struct MmaConfigsB18<1> {
    static constexpr MmaConfig list[] = {cfg_of<1, 8, 1, true>(), cfg_of<1, 7, 1, true>(), cfg_of<1, 6, 1, true>(),
                                         cfg_of<1, 5, 1, true>(), cfg_of<1, 4, 1, true>(), cfg_of<1, 3, 1, true>(),
                                         cfg_of<1, 2, 1, true>(), cfg_of<1, 1, 1, true>(), cfg_of<1, 2, 2, true>(),
                                         cfg_of<1, 1, 2, true>()};
};
template <>
struct MmaConfigsB18<2> {
    static constexpr MmaConfig list[] = {cfg_of<2, 8, 1, true>(), cfg_of<2, 7, 1, true>(), cfg_of<2, 6, 1, true>(),
                                         cfg_of<2, 5, 1, true>(), cfg_of<2, 4, 1, true>(), cfg_of<2, 3, 1, true>(),
                                         cfg_of<2, 2, 1, true>(), cfg_of<2, 1, 1, true>(), cfg_of<2, 1, 2, true>()};
};
template <>
struct MmaConfigsB18<3> {
    static constexpr MmaConfig list[] = {cfg_of<3, 4, 1, true>(), cfg_of<3, 3, 1, true>(), cfg_of<3, 2, 1, true>(),
                                         cfg_of<3, 1, 1, true>(), cfg_of<3, 1, 2, true>()};
};
template <>
struct MmaConfigsB18<4> {
    static constexpr MmaConfig list[] = {cfg_of<4, 4, 1, true>(), cfg_of<4, 3, 1, true>(), cfg_of<4, 2, 1, true>(),
                                         cfg_of<4, 1, 1, true>()};
};

}  // namespace

cudaError_t launch_matmul_mma_b18(int wt, const void* w, int64_t N, int64_t K, const int8_t* qs, const void* ds,
                                  int64_t M, float* y, int64_t ldy, void* encode, int* err, int num_sms,
                                  int skip_w_stage, cudaStream_t stream) {
    if (wt != kWtQ4_0 && wt != kWtIQ4NL) return cudaErrorInvalidValue;
    const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(encode);
    const int64_t row_bytes = wt_row_bytes(wt, K);
    const int mt = mma_tile_rows(M);
    CUtensorMap tq;
    const cudaError_t eq = encode_q_map(enc, qs, K, M, mt, &tq);
    if (eq != cudaSuccess) return eq;
    const __half* dsh = reinterpret_cast<const __half*>(ds);
    const int Ni = (int)N, Ki = (int)K;
#define IQ4XS_MMA_BEST(nt) \
    launch_best<nt, true>(MmaConfigsB18<nt>::list, w, row_bytes, enc, tq, dsh, M, Ni, Ki, y, ldy, err, wt, \
                          skip_w_stage, num_sms, stream)
    switch (mt) {
        case 8: return IQ4XS_MMA_BEST(1);
        case 16: return IQ4XS_MMA_BEST(2);
        case 24: return IQ4XS_MMA_BEST(3);
        default: return IQ4XS_MMA_BEST(4);
    }
#undef IQ4XS_MMA_BEST
}

cudaError_t launch_matmul_mma_grouped_b18(int wt, const void* w, int64_t expert_stride, int64_t G, int64_t N,
                                          int64_t K, const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                          int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                          int num_sms, int skip_w_stage, cudaStream_t stream) {
    if (wt != kWtQ4_0 && wt != kWtIQ4NL) return cudaErrorInvalidValue;
    return launch_grouped<true>(wt, w, expert_stride, G, N, K, qs, ds, row_offsets, total_rows, y, ldy, encode,
                                err, num_sms, skip_w_stage, stream);
}

}  // namespace iq4xs
