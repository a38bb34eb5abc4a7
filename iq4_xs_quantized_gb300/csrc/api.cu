// api.cu -- the extern "C" boundary of libiq4xs.so (declared in
// include/iq4xs.h): argument validation, per-device set-up, path dispatch.
// All validation happens on the host before any launch.
#include <cuda.h>

#include <atomic>
#include <mutex>

#include "../../include/iq4xs.h"
#include "internal.cuh"

namespace iq4xs {

// Device error word: kernels whose bounded waits run out (and, in the
// bounds-checked build, checked accesses that miss their buffer) record a
// code in word 0; words 2-3 hold the bounds-checked build's test margin.
__device__ __align__(16) int g_device_error[kErrWords] = {0, 0, 0, 0};

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kGroupedTcMinRows = 32;   // grouped: tcgen05 from this mean rows per expert slot on
constexpr int64_t kGroupedMmaMinRows = 24;  // grouped: warp MMA from this many rows on (at most G)
constexpr int64_t kMaxM = 32768;

struct DevState {
    bool ready = false;
    int status = IQ4XS_OK;
    int num_sms = 0;
    int* err = nullptr;       // device address of g_device_error (kErrWords ints)
    void* encode = nullptr;   // cuTensorMapEncodeTiled
};

std::mutex g_mu;
DevState g_dev[kMaxDevices];
std::atomic<int64_t> g_crossover{4};
std::atomic<int64_t> g_baseline_min{0};  // 0 = never advise the dequantize + GEMM route
std::atomic<int> g_pdl{1};
std::atomic<int> g_skip_w_stage{-1};  // armed by iq4xs_test_skip_w_stage, one launch

std::atomic<int64_t> g_mma_max{8};      // the warp-MMA path up to this M (above the DP4A range)

// Measured crossovers per weight-size class: entry i applies to matrices of
// at least min[i] weights (N*K), the largest such entry winning; matrices
// below every entry use the global value.  One table for the DP4A range and
// one for the warp-MMA range.
constexpr int kMaxClasses = 16;
struct ClassTable {
    std::mutex mu;
    int n = 0;
    int64_t min[kMaxClasses];
    int64_t m[kMaxClasses];
    int64_t lookup(int64_t nk, int64_t dflt) {
        std::lock_guard<std::mutex> lock(mu);
        int64_t r = dflt, best = -1;
        for (int i = 0; i < n; ++i)
            if (min[i] <= nk && min[i] > best) {
                best = min[i];
                r = m[i];
            }
        return r;
    }
};
ClassTable g_dp4a_classes, g_mma_classes;

int64_t crossover_for(int64_t N, int64_t K) { return g_dp4a_classes.lookup(N * K, g_crossover.load()); }
int64_t mma_max_for(int64_t N, int64_t K) { return g_mma_classes.lookup(N * K, g_mma_max.load()); }

int set_classes(ClassTable& tab, const int64_t* min_weights, const int64_t* m_max, int count) {
    if (count < 0 || count > kMaxClasses) return IQ4XS_ERR_ARG;
    if (count > 0 && (!min_weights || !m_max)) return IQ4XS_ERR_ARG;
    for (int i = 0; i < count; ++i)
        if (min_weights[i] < 1 || m_max[i] < 0 || m_max[i] > kMaxM) return IQ4XS_ERR_ARG;
    std::lock_guard<std::mutex> lock(tab.mu);
    for (int i = 0; i < count; ++i) {
        tab.min[i] = min_weights[i];
        tab.m[i] = m_max[i];
    }
    tab.n = count;
    return IQ4XS_OK;
}

// One-time per-device set-up, done with that device current.
int device_state(DevState** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return IQ4XS_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DevState& st = g_dev[dev];
    if (!st.ready) {
        st.ready = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&st.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            st.status = IQ4XS_ERR_DEVICE;
        } else if (major != 10 || minor != 3) {
            st.status = IQ4XS_ERR_DEVICE;  // built for sm_103a only
        } else if (cudaGetSymbolAddress(reinterpret_cast<void**>(&st.err), g_device_error) !=
                   cudaSuccess) {
            cudaGetLastError();
            st.status = IQ4XS_ERR_CUDA;
        } else {
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &st.encode, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || st.encode == nullptr) {
                cudaGetLastError();
                st.status = IQ4XS_ERR_CUDA;
            }
        }
    }
    *out = &st;
    return st.status;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int from_cuda(cudaError_t e) { return e == cudaSuccess ? IQ4XS_OK : IQ4XS_ERR_CUDA; }

// The path this library's own kernels take: DP4A up to the matrix class's
// DP4A crossover, the warp-MMA path up to its MMA crossover, TC above (the
// crossovers measured on IQ4_XS serve the 18-byte-block formats too: their
// kernels are the same but for the weight layout).  Both tensor-core paths
// stage W rows with a tensor map, whose row stride must be a multiple of 16
// bytes: K % 512 == 0 (136-byte super-blocks in pairs); other K run DP4A.
int kernel_path_impl(int64_t M, int64_t N, int64_t K) {
    if (K % kPairK != 0 || M <= crossover_for(N, K)) return IQ4XS_PATH_DP4A;
    if (M <= mma_max_for(N, K)) return IQ4XS_PATH_MMA;
    return IQ4XS_PATH_TC;
}
// The grouped form: the warp-MMA form from 24 rows on (as many as the
// experts, if fewer), or once the mean rows of an expert slot leave one
// expert matrix's DP4A range (measured on a 128 x 1536 x 2048 layer: the
// CUDA-core form is 6 % faster at 16 rows, 19 % slower at 24 and 30 % at
// 64); the tcgen05 form from 32 mean rows per expert slot on (the same
// layer: 15 % slower at 24, 2 % faster at 32, 8 % at 64, 24 % at 256), for
// IQ4_XS weights (the other formats stay on the warp-MMA form); DP4A
// otherwise, and whenever K % 512 != 0.
int grouped_path_impl(int64_t G, int64_t N, int64_t K, int64_t total_rows, int wtype) {
    const int64_t slots = G < total_rows ? G : total_rows;
    const int64_t mean = (total_rows + slots - 1) / slots;
    const int64_t mma_min = G < kGroupedMmaMinRows ? G : kGroupedMmaMinRows;
    if (K % kPairK != 0 || (total_rows < mma_min && mean <= crossover_for(N, K))) return IQ4XS_PATH_DP4A;
    return (mean >= kGroupedTcMinRows && wtype == IQ4XS_WTYPE_IQ4_XS) ? IQ4XS_PATH_TC : IQ4XS_PATH_MMA;
}
// The advised path: the kernel path, or BASELINE above the measured threshold.
int select_path_impl(int64_t M, int64_t N, int64_t K) {
    const int p = kernel_path_impl(M, N, K);
    const int64_t b = g_baseline_min.load();
    return (p == IQ4XS_PATH_TC && b > 0 && M >= b) ? IQ4XS_PATH_BASELINE : p;
}

}  // namespace

bool pdl_enabled() { return g_pdl.load() != 0; }

}  // namespace iq4xs

using namespace iq4xs;

extern "C" {

int iq4xs_quantize_q8_1(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, void* ds,
                        int64_t stream) {
    if (!x || !qs || !ds) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || K <= 0 || K % kQK) return IQ4XS_ERR_SHAPE;
    if (ldx < K || (ldx * 4) % 16) return IQ4XS_ERR_ARG;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(ds, 4)) return IQ4XS_ERR_ALIGN;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    return from_cuda(
        launch_quantize_q8_1(x, M, K, ldx, qs, ds, nullptr, st->err, reinterpret_cast<cudaStream_t>(stream)));
}

int64_t iq4xs_tc_operand_bytes(int64_t M, int64_t K) {
    if (M < 1 || M > kMaxM || K <= 0 || K % kQK || K > (1 << 30)) return 0;
    return tc_operand_total_bytes(M, K);
}

int iq4xs_quantize_q8_1_tc(const float* x, int64_t M, int64_t K, int64_t ldx, int8_t* qs, void* ds,
                           void* tc_operand, int64_t stream) {
    if (!x || !qs || !ds || !tc_operand) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || K <= 0 || K % kQK) return IQ4XS_ERR_SHAPE;
    if (ldx < K || (ldx * 4) % 16) return IQ4XS_ERR_ARG;
    if (!aligned(x, 16) || !aligned(qs, 16) || !aligned(ds, 4) || !aligned(tc_operand, 16))
        return IQ4XS_ERR_ALIGN;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    return from_cuda(launch_quantize_q8_1(x, M, K, ldx, qs, ds, tc_operand, st->err,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int64_t iq4xs_weight_bytes(int wtype, int64_t N, int64_t K) {
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return 0;
    if (N < 1 || N > (1 << 30) || K <= 0 || K % kQK || K > (1 << 30)) return 0;
    return N * wt_row_bytes(wtype, K);
}

int iq4xs_matmul(const void* w, int64_t N, int64_t K, const int8_t* qs, const void* ds, int64_t M,
                 float* y, int64_t ldy, int path, int64_t stream) {
    return iq4xs_matmul_wt(w, IQ4XS_WTYPE_IQ4_XS, N, K, qs, ds, M, y, ldy, path, stream);
}

int iq4xs_matmul_wt(const void* w, int wtype, int64_t N, int64_t K, const int8_t* qs,
                    const void* ds, int64_t M, float* y, int64_t ldy, int path, int64_t stream) {
    if (!w || !qs || !ds || !y) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    if (path < IQ4XS_PATH_AUTO || path > IQ4XS_PATH_MMA || path == IQ4XS_PATH_BASELINE) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || N < 1 || N > (1 << 30) || K <= 0 || K % kQK || K > (1 << 30))
        return IQ4XS_ERR_SHAPE;
    if (ldy < N) return IQ4XS_ERR_ARG;
    if (!aligned(w, 16) || !aligned(qs, 16) || !aligned(ds, 4) || !aligned(y, 4)) return IQ4XS_ERR_ALIGN;
    if (path == IQ4XS_PATH_AUTO) path = kernel_path_impl(M, N, K);
    if ((path == IQ4XS_PATH_TC || path == IQ4XS_PATH_MMA) && K % kPairK) return IQ4XS_ERR_SHAPE;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (path == IQ4XS_PATH_MMA)
        return from_cuda(
            launch_matmul_mma(w, wtype, N, K, qs, ds, M, y, ldy, st->encode, st->err, st->num_sms,
                              g_skip_w_stage.exchange(-1), s));
    if (path == IQ4XS_PATH_TC)
        return from_cuda(launch_matmul_tc(w, wtype, N, K, qs, ds, nullptr, M, y, ldy, st->encode,
                                          st->err, st->num_sms, g_skip_w_stage.exchange(-1), s));
    return from_cuda(launch_matmul_dp4a(w, wtype, N, K, qs, ds, M, y, ldy, st->err, st->num_sms, s));
}

int iq4xs_matmul_tc_operand(const void* w, int wtype, int64_t N, int64_t K, const void* tc_operand,
                            int64_t M, float* y, int64_t ldy, int64_t stream) {
    if (!w || !tc_operand || !y) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || N < 1 || N > (1 << 30) || K <= 0 || K % kPairK || K > (1 << 30))
        return IQ4XS_ERR_SHAPE;
    if (ldy < N) return IQ4XS_ERR_ARG;
    if (!aligned(w, 16) || !aligned(tc_operand, 16) || !aligned(y, 4)) return IQ4XS_ERR_ALIGN;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    return from_cuda(launch_matmul_tc(w, wtype, N, K, nullptr, nullptr, tc_operand, M, y, ldy,
                                      st->encode, st->err, st->num_sms, g_skip_w_stage.exchange(-1),
                                      reinterpret_cast<cudaStream_t>(stream)));
}

namespace {
inline int64_t align16(int64_t v) { return (v + 15) / 16 * 16; }
// Workspace of iq4xs_linear: the Q8_1 codes, then (16-byte aligned) the
// {d, s} pairs -- `q8` bytes, 1.125 per activation -- and on the
// tensor-core path the prepared operand after them (`total`).
struct LinearLayout {
    int64_t qs, ds, op, q8, total;
    int path;
};
bool linear_layout(int64_t M, int64_t N, int64_t K, LinearLayout* L) {
    if (M < 1 || M > kMaxM || N < 1 || N > (1 << 30) || K <= 0 || K % kQK || K > (1 << 30))
        return false;
    L->path = kernel_path_impl(M, N, K);
    L->qs = 0;
    L->ds = align16(M * K);
    L->q8 = L->ds + align16(M * (K / kSub) * 4);
    L->op = L->q8;
    L->total = L->q8 + (L->path == IQ4XS_PATH_TC ? tc_operand_total_bytes(M, K) : 0);
    return true;
}
}  // namespace

int64_t iq4xs_linear_workspace_bytes(int64_t M, int64_t N, int64_t K) {
    LinearLayout L;
    return linear_layout(M, N, K, &L) ? L.total : 0;
}

int64_t iq4xs_linear_workspace_min_bytes(int64_t M, int64_t N, int64_t K) {
    LinearLayout L;
    return linear_layout(M, N, K, &L) ? L.q8 : 0;
}

int iq4xs_linear(const void* w, int64_t N, int64_t K, const float* x, int64_t M, int64_t ldx,
                 float* y, int64_t ldy, void* workspace, int64_t workspace_bytes,
                 int64_t stream) {
    return iq4xs_linear_wt(w, IQ4XS_WTYPE_IQ4_XS, N, K, x, M, ldx, y, ldy, workspace, workspace_bytes, stream);
}

int iq4xs_linear_wt(const void* w, int wtype, int64_t N, int64_t K, const float* x, int64_t M, int64_t ldx,
                    float* y, int64_t ldy, void* workspace, int64_t workspace_bytes, int64_t stream) {
    if (!w || !x || !y || !workspace) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    LinearLayout L;
    if (!linear_layout(M, N, K, &L)) return IQ4XS_ERR_SHAPE;
    if (workspace_bytes < L.q8) return IQ4XS_ERR_ARG;
    if (!aligned(workspace, 16)) return IQ4XS_ERR_ALIGN;
    uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
    int8_t* qs = reinterpret_cast<int8_t*>(ws + L.qs);
    void* ds = ws + L.ds;
    if (L.path == IQ4XS_PATH_TC && workspace_bytes >= L.total) {  // room for the prepared operand
        int rc = iq4xs_quantize_q8_1_tc(x, M, K, ldx, qs, ds, ws + L.op, stream);
        if (rc) return rc;
        return iq4xs_matmul_tc_operand(w, wtype, N, K, ws + L.op, M, y, ldy, stream);
    }
    int rc = iq4xs_quantize_q8_1(x, M, K, ldx, qs, ds, stream);
    if (rc) return rc;
    return iq4xs_matmul_wt(w, wtype, N, K, qs, ds, M, y, ldy, L.path, stream);
}

int iq4xs_matmul_grouped(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                         const int8_t* qs, const void* ds, const int32_t* row_offsets,
                         int64_t total_rows, float* y, int64_t ldy, int64_t stream) {
    return iq4xs_matmul_grouped_path(w, expert_stride, G, N, K, qs, ds, row_offsets, total_rows, y, ldy,
                                     IQ4XS_PATH_AUTO, stream);
}

int iq4xs_matmul_grouped_path(const void* w, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                              const int8_t* qs, const void* ds, const int32_t* row_offsets,
                              int64_t total_rows, float* y, int64_t ldy, int path, int64_t stream) {
    return iq4xs_matmul_grouped_wt(w, IQ4XS_WTYPE_IQ4_XS, expert_stride, G, N, K, qs, ds, row_offsets, total_rows,
                                   y, ldy, path, stream);
}

int iq4xs_matmul_grouped_wt(const void* w, int wtype, int64_t expert_stride, int64_t G, int64_t N, int64_t K,
                            const int8_t* qs, const void* ds, const int32_t* row_offsets, int64_t total_rows,
                            float* y, int64_t ldy, int path, int64_t stream) {
    if (!w || !qs || !ds || !row_offsets || !y) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    if (path != IQ4XS_PATH_AUTO && path != IQ4XS_PATH_DP4A && path != IQ4XS_PATH_MMA && path != IQ4XS_PATH_TC)
        return IQ4XS_ERR_ARG;
    if (G < 1 || G > 65535 || N < 1 || N > (1 << 30) || K <= 0 || K % kQK || K > (1 << 30))
        return IQ4XS_ERR_SHAPE;
    if (ldy < N || total_rows < 1) return IQ4XS_ERR_ARG;
    if (total_rows > kMaxM) return IQ4XS_ERR_SHAPE;  // the rows one quantize call takes
    if (expert_stride < N * wt_row_bytes(wtype, K) || expert_stride % 16) return IQ4XS_ERR_ARG;
    if (!aligned(w, 16) || !aligned(qs, 16) || !aligned(ds, 4) || !aligned(row_offsets, 4) ||
        !aligned(y, 4))
        return IQ4XS_ERR_ALIGN;
    if (path == IQ4XS_PATH_AUTO) path = grouped_path_impl(G, N, K, total_rows, wtype);
    if ((path == IQ4XS_PATH_MMA || path == IQ4XS_PATH_TC) && K % kPairK) return IQ4XS_ERR_SHAPE;
    if (path == IQ4XS_PATH_TC && wtype != IQ4XS_WTYPE_IQ4_XS) return IQ4XS_ERR_SHAPE;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (path == IQ4XS_PATH_TC)
        return from_cuda(launch_matmul_tc_grouped(w, expert_stride, G, N, K, qs, ds, row_offsets, total_rows, y,
                                                  ldy, st->encode, st->err, s));
    if (path == IQ4XS_PATH_MMA)
        return from_cuda(launch_matmul_mma_grouped(w, wtype, expert_stride, G, N, K, qs, ds, row_offsets,
                                                   total_rows, y, ldy, st->encode, st->err, st->num_sms,
                                                   g_skip_w_stage.exchange(-1), s));
    return from_cuda(launch_matmul_dp4a_grouped(w, wtype, expert_stride, G, N, K, qs, ds, row_offsets,
                                                total_rows, y, ldy, st->err, s));
}

int iq4xs_dequantize(const void* w, int64_t N, int64_t K, void* out, int out_dtype,
                     int64_t stream) {
    return iq4xs_dequantize_wt(w, IQ4XS_WTYPE_IQ4_XS, N, K, out, out_dtype, stream);
}

int iq4xs_dequantize_wt(const void* w, int wtype, int64_t N, int64_t K, void* out,
                        int out_dtype, int64_t stream) {
    if (!w || !out) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    if (out_dtype != 0 && out_dtype != 1) return IQ4XS_ERR_ARG;
    if (N < 1 || K <= 0 || K % kQK) return IQ4XS_ERR_SHAPE;
    if (!aligned(w, 16) || !aligned(out, 16)) return IQ4XS_ERR_ALIGN;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    return from_cuda(launch_dequantize(w, wtype, N, K, out, out_dtype, st->err,
                                       reinterpret_cast<cudaStream_t>(stream)));
}

int iq4xs_select_path(int64_t M, int64_t N, int64_t K, int* path_out) {
    if (!path_out) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || N < 1 || K <= 0 || K % kQK) return IQ4XS_ERR_SHAPE;
    *path_out = select_path_impl(M, N, K);
    return IQ4XS_OK;
}

int iq4xs_select_grouped_path(int64_t G, int64_t N, int64_t K, int64_t total_rows, int wtype, int* path_out) {
    if (!path_out) return IQ4XS_ERR_ARG;
    if (wtype < IQ4XS_WTYPE_IQ4_XS || wtype > IQ4XS_WTYPE_IQ4_NL) return IQ4XS_ERR_ARG;
    if (G < 1 || G > 65535 || N < 1 || N > (1 << 30) || K <= 0 || K % kQK || K > (1 << 30) || total_rows < 1 ||
        total_rows > kMaxM)
        return IQ4XS_ERR_SHAPE;
    *path_out = grouped_path_impl(G, N, K, total_rows, wtype);
    return IQ4XS_OK;
}

int iq4xs_set_crossover(int64_t m_max_dp4a) {
    if (m_max_dp4a < 0 || m_max_dp4a > kMaxM) return IQ4XS_ERR_ARG;
    g_crossover.store(m_max_dp4a);
    return IQ4XS_OK;
}

int iq4xs_set_crossover_classes(const int64_t* min_weights, const int64_t* m_max_dp4a, int count) {
    return set_classes(g_dp4a_classes, min_weights, m_max_dp4a, count);
}

int iq4xs_set_mma_crossover(int64_t m_max_mma) {
    if (m_max_mma < 0 || m_max_mma > kMaxM) return IQ4XS_ERR_ARG;
    g_mma_max.store(m_max_mma);
    return IQ4XS_OK;
}

int iq4xs_set_mma_crossover_classes(const int64_t* min_weights, const int64_t* m_max_mma, int count) {
    return set_classes(g_mma_classes, min_weights, m_max_mma, count);
}

int iq4xs_set_baseline_threshold(int64_t m_min_baseline) {
    if (m_min_baseline < 0 || m_min_baseline > kMaxM + 1) return IQ4XS_ERR_ARG;
    g_baseline_min.store(m_min_baseline);
    return IQ4XS_OK;
}

int iq4xs_set_pdl(int enable) {
    g_pdl.store(enable ? 1 : 0);
    return IQ4XS_OK;
}

int iq4xs_last_device_error(int* code_out) {
    if (!code_out) return IQ4XS_ERR_ARG;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) return IQ4XS_ERR_CUDA;
    int zero = 0;
    if (cudaMemcpyFromSymbol(code_out, g_device_error, sizeof(int)) != cudaSuccess ||
        cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
        return IQ4XS_ERR_CUDA;
    const int c = *code_out;
    if (c >= kDevErrBounds && c < kDevErrBounds + 0x100) return IQ4XS_ERR_BOUNDS;
    return ((c >= kDevErrTimeoutW && c <= kDevErrTimeoutX) || c == kDevErrTimeoutMmaStage ||
            c == kDevErrTimeoutMmaSlot)
               ? IQ4XS_ERR_TIMEOUT
               : IQ4XS_OK;
}

int iq4xs_bounds_checked(int* out) {
    if (!out) return IQ4XS_ERR_ARG;
    *out = kBoundsCheck ? 1 : 0;
    return IQ4XS_OK;
}

int iq4xs_test_bounds_margin(int64_t bytes) {
    if (!kBoundsCheck || bytes < 0 || bytes > (int64_t(1) << 40)) return IQ4XS_ERR_ARG;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) return IQ4XS_ERR_CUDA;
    const long long v = bytes;
    return from_cuda(cudaMemcpyToSymbol(g_device_error, &v, sizeof(v), 2 * sizeof(int)));
}

int iq4xs_test_skip_w_stage(int64_t stage) {
    if (stage < -1 || stage > (1 << 20)) return IQ4XS_ERR_ARG;
    g_skip_w_stage.store((int)stage);
    return IQ4XS_OK;
}

int iq4xs_test_mma_config(int64_t rows_per_cta, int64_t k_splits, int64_t ctas_per_sm) {
    if (rows_per_cta < 0 || rows_per_cta > 256 || rows_per_cta % 32 || k_splits < 0 || k_splits > 8 ||
        ctas_per_sm < 0 || ctas_per_sm > 2)
        return IQ4XS_ERR_ARG;
    mma_force_config((int)rows_per_cta, (int)k_splits, (int)ctas_per_sm);
    return IQ4XS_OK;
}

int iq4xs_set_mma_launch_table(const int64_t* entries, int count) {
    return mma_set_launch_table(entries, count) == 0 ? IQ4XS_OK : IQ4XS_ERR_ARG;
}

int iq4xs_mma_launch_config(int64_t M, int64_t N, int64_t K, int* rows_per_cta, int* k_splits, int* ctas_per_sm) {
    if (!rows_per_cta || !k_splits || !ctas_per_sm) return IQ4XS_ERR_ARG;
    if (M < 1 || M > kMaxM || N < 1 || N > (1 << 30) || K <= 0 || K % kPairK || K > (1 << 30))
        return IQ4XS_ERR_SHAPE;
    DevState* st;
    int rc = device_state(&st);
    if (rc) return rc;
    int r = 0, s = 0, o = 0;
    mma_launch_config(M, N, K, st->num_sms, &r, &s, &o);
    *rows_per_cta = r;
    *k_splits = s;
    *ctas_per_sm = o;
    return IQ4XS_OK;
}

const char* iq4xs_status_string(int status) {
    switch (status) {
        case IQ4XS_OK: return "ok";
        case IQ4XS_ERR_ARG: return "invalid argument";
        case IQ4XS_ERR_ALIGN: return "misaligned pointer";
        case IQ4XS_ERR_SHAPE: return "unsupported shape";
        case IQ4XS_ERR_DEVICE: return "no sm_103 device";
        case IQ4XS_ERR_CUDA: return "CUDA error";
        case IQ4XS_ERR_TIMEOUT: return "device wait timed out";
        case IQ4XS_ERR_BOUNDS: return "checked device access out of bounds";
        default: return "unknown status";
    }
}

}  // extern "C"
