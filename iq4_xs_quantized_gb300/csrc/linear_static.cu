// linear_static.cu -- iq4xs_linear_static: the one-call projection
// (iq4xs_linear) with its workspace in a fixed device array owned by this
// library, so the caller passes only the weights, the activations and the
// output, and nothing is allocated.
//
// Who needs it: code that cannot allocate device memory itself -- a plugin
// running inside a host framework that owns every device allocation, or a
// serving loop that must not allocate once it is running (cudaMalloc may
// synchronize the device, can fail under memory pressure, and is not
// allowed while a stream is being captured into a CUDA graph).
#include <mutex>

#include "../../include/iq4xs.h"
#include "internal.cuh"

namespace iq4xs {
namespace {

// The fixed scratch: 8 MiB, shared by every call made on a device.  Every GPU
// that loads this library holds it until the process exits.
constexpr int64_t kStaticScratchBytes = 8ll << 20;
static __device__ __align__(256) uint8_t g_linear_scratch[kStaticScratchBytes];

// In host code the array's name is only a host-side stand-in, not a device
// address, so the address is looked up once per device (with that device
// current) and passed on to the kernels.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void* g_scratch_ptr[kMaxDevices] = {};

int scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return IQ4XS_ERR_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_linear_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return IQ4XS_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return IQ4XS_OK;
}

}  // namespace
}  // namespace iq4xs

extern "C" {

int64_t iq4xs_linear_static_max_bytes(void) { return iq4xs::kStaticScratchBytes; }

int iq4xs_linear_static(const void* w, int64_t N, int64_t K, const float* x, int64_t M,
                        int64_t ldx, float* y, int64_t ldy, int64_t stream) {
    if (!w || !x || !y) return IQ4XS_ERR_ARG;
    // The Q8_1 codes and scales must fit (the faster prepared tensor-core
    // operand is used when it fits too); more than the fixed array holds is
    // refused and nothing is launched.
    const int64_t need = iq4xs_linear_workspace_min_bytes(M, N, K);
    if (need == 0) return IQ4XS_ERR_SHAPE;
    if (need > iq4xs::kStaticScratchBytes) return IQ4XS_ERR_SHAPE;
    void* scratch = nullptr;
    const int rc = iq4xs::scratch_address(&scratch);
    if (rc) return rc;
    // Every byte of the scratch that the matmul reads (the Q8_1 codes and
    // scales of rows 0..M-1, or the prepared operand including its padding
    // rows) is written by the quantizer first, so nothing needs clearing.
    return iq4xs_linear(w, N, K, x, M, ldx, y, ldy, scratch, iq4xs::kStaticScratchBytes, stream);
}

}  // extern "C"
