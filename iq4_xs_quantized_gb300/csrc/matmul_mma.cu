// matmul_mma.cu -- IQ4_XS launches of the warp-level MMA matmul (the kernel
// and its launch model are in mma_kernel.cuh): the launch configurations
// per activation-tile width, the measured launch table and the forced test
// configuration, and the path's entry points, dense and grouped (other
// weight formats go on to matmul_mma_b18.cu).
#include <atomic>
#include <mutex>

#include "mma_kernel.cuh"

namespace iq4xs {
namespace {

// Test override of the launch configuration (0 = the model's choice).
std::atomic<int> g_force_rows{0}, g_force_s{0}, g_force_occ{0};

// Measured launches (installed from the calibration): for a weight shape
// and activation-tile height, the rows per CTA, K split and CTAs per SM
// that timed fastest.
struct LaunchEntry {
    int64_t N, K;
    int mt, R, S, occ;
};
constexpr int kMaxLaunchEntries = 256;
std::mutex g_launch_mu;
LaunchEntry g_launch[kMaxLaunchEntries];
int g_launch_n = 0;

bool measured_launch(int64_t N, int64_t K, int mt, LaunchEntry* out) {
    std::lock_guard<std::mutex> lock(g_launch_mu);
    for (int i = 0; i < g_launch_n; ++i)
        if (g_launch[i].N == N && g_launch[i].K == K && g_launch[i].mt == mt) {
            *out = g_launch[i];
            return true;
        }
    return false;
}

// Per activation-tile width: T = 1..8 (4 from 24 activation rows on, the
// accumulators' registers) at one CTA per SM, and the tiles that leave room
// for two CTAs per SM (113 KB each, two stages: up to 64 rows at 8
// activation rows, 32 at 16 and 24).
template <int NT>
struct MmaConfigs;
template <>
struct MmaConfigs<1> {
    static constexpr MmaConfig list[] = {cfg_of<1, 8, 1>(), cfg_of<1, 7, 1>(), cfg_of<1, 6, 1>(), cfg_of<1, 5, 1>(),
                                         cfg_of<1, 4, 1>(), cfg_of<1, 3, 1>(), cfg_of<1, 2, 1>(), cfg_of<1, 1, 1>(),
                                         cfg_of<1, 2, 2>(), cfg_of<1, 1, 2>()};
};
template <>
struct MmaConfigs<2> {
    static constexpr MmaConfig list[] = {cfg_of<2, 8, 1>(), cfg_of<2, 7, 1>(), cfg_of<2, 6, 1>(), cfg_of<2, 5, 1>(),
                                         cfg_of<2, 4, 1>(), cfg_of<2, 3, 1>(), cfg_of<2, 2, 1>(), cfg_of<2, 1, 1>(),
                                         cfg_of<2, 1, 2>()};
};
template <>
struct MmaConfigs<3> {
    static constexpr MmaConfig list[] = {cfg_of<3, 4, 1>(), cfg_of<3, 3, 1>(), cfg_of<3, 2, 1>(), cfg_of<3, 1, 1>(),
                                         cfg_of<3, 1, 2>()};
};
template <>
struct MmaConfigs<4> {
    static constexpr MmaConfig list[] = {cfg_of<4, 4, 1>(), cfg_of<4, 3, 1>(), cfg_of<4, 2, 1>(),
                                         cfg_of<4, 1, 1>()};
};

template <int NT>
void report_config(int64_t M, int N, int K, int num_sms, int* rows, int* splits, int* ctas_per_sm) {
    const auto& list = MmaConfigs<NT>::list;
    int ci = 0, s = 1;
    choose_config<NT, false>(list, (int)(sizeof(list) / sizeof(list[0])), M, N, K, num_sms, &ci, &s);
    *rows = list[ci].R;
    *splits = s;
    *ctas_per_sm = list[ci].occ;
}

}  // namespace

void mma_forced_config(int* rows, int* splits, int* ctas_per_sm) {
    *rows = g_force_rows.load();
    *splits = g_force_s.load();
    *ctas_per_sm = g_force_occ.load();
}

bool mma_measured_launch(int64_t N, int64_t K, int mt, int* rows, int* splits, int* ctas_per_sm) {
    LaunchEntry e;
    if (!measured_launch(N, K, mt, &e)) return false;
    *rows = e.R;
    *splits = e.S;
    *ctas_per_sm = e.occ;
    return true;
}

void mma_launch_config(int64_t M, int64_t N, int64_t K, int num_sms, int* rows, int* splits, int* ctas_per_sm) {
    const int Ni = (int)N, Ki = (int)K;
    switch (mma_tile_rows(M)) {
        case 8: return report_config<1>(M, Ni, Ki, num_sms, rows, splits, ctas_per_sm);
        case 16: return report_config<2>(M, Ni, Ki, num_sms, rows, splits, ctas_per_sm);
        case 24: return report_config<3>(M, Ni, Ki, num_sms, rows, splits, ctas_per_sm);
        default: return report_config<4>(M, Ni, Ki, num_sms, rows, splits, ctas_per_sm);
    }
}

int mma_set_launch_table(const int64_t* entries, int count) {
    if (count < 0 || count > kMaxLaunchEntries || (count > 0 && !entries)) return -1;
    for (int i = 0; i < count; ++i) {
        const int64_t* v = entries + 6 * i;
        if (v[0] < 1 || v[1] < kPairK || v[1] % kPairK || (v[2] != 8 && v[2] != 16 && v[2] != 24 && v[2] != 32) ||
            v[3] < 32 || v[3] > kMmaMaxRows || v[3] % 32 || v[4] < 1 || v[4] > kMmaMaxCluster || v[5] < 1 ||
            v[5] > 2)
            return -1;
    }
    std::lock_guard<std::mutex> lock(g_launch_mu);
    for (int i = 0; i < count; ++i) {
        const int64_t* v = entries + 6 * i;
        g_launch[i] = {v[0], v[1], (int)v[2], (int)v[3], (int)v[4], (int)v[5]};
    }
    g_launch_n = count;
    return 0;
}

void mma_force_config(int rows_per_cta, int k_splits, int ctas_per_sm) {
    g_force_rows.store(rows_per_cta);
    g_force_s.store(k_splits);
    g_force_occ.store(ctas_per_sm);
}

cudaError_t launch_matmul_mma_grouped(const void* w, int wt, int64_t expert_stride, int64_t G, int64_t N,
                                      int64_t K, const int8_t* qs, const void* ds, const int32_t* row_offsets,
                                      int64_t total_rows, float* y, int64_t ldy, void* encode, int* err,
                                      int num_sms, int skip_w_stage, cudaStream_t stream) {
    if (wt != kWtIQ4XS)
        return launch_matmul_mma_grouped_b18(wt, w, expert_stride, G, N, K, qs, ds, row_offsets, total_rows, y, ldy,
                                             encode, err, num_sms, skip_w_stage, stream);
    return launch_grouped<false>(wt, w, expert_stride, G, N, K, qs, ds, row_offsets, total_rows, y, ldy, encode,
                                 err, num_sms, skip_w_stage, stream);
}

int mma_tile_rows(int64_t M) {
    const int64_t nt = (M + 7) / 8;
    return 8 * (int)(nt < 4 ? nt : 4);
}

cudaError_t launch_matmul_mma(const void* w, int wt, int64_t N, int64_t K, const int8_t* qs, const void* ds,
                              int64_t M, float* y, int64_t ldy, void* encode, int* err, int num_sms,
                              int skip_w_stage, cudaStream_t stream) {
    if (wt != kWtIQ4XS)
        return launch_matmul_mma_b18(wt, w, N, K, qs, ds, M, y, ldy, encode, err, num_sms, skip_w_stage, stream);
    const EncodeTiledFn enc = reinterpret_cast<EncodeTiledFn>(encode);
    const int64_t row_bytes = wt_row_bytes(kWtIQ4XS, K);
    const int mt = mma_tile_rows(M);
    CUtensorMap tq;
    const cudaError_t eq = encode_q_map(enc, qs, K, M, mt, &tq);
    if (eq != cudaSuccess) return eq;
    const __half* dsh = reinterpret_cast<const __half*>(ds);
    const int Ni = (int)N, Ki = (int)K;
#define IQ4XS_MMA_BEST(nt) \
    launch_best<nt, false>(MmaConfigs<nt>::list, w, row_bytes, enc, tq, dsh, M, Ni, Ki, y, ldy, err, kWtIQ4XS, \
                           skip_w_stage, num_sms, stream)
    switch (mt) {
        case 8: return IQ4XS_MMA_BEST(1);
        case 16: return IQ4XS_MMA_BEST(2);
        case 24: return IQ4XS_MMA_BEST(3);
        default: return IQ4XS_MMA_BEST(4);
    }
#undef IQ4XS_MMA_BEST
}

}  // namespace iq4xs
