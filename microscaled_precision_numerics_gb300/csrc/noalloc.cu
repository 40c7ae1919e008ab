// noalloc.cu -- allocation-free entry point for the NVFP4 16x16 2D weight quantizer.
//
// mx_nvfp4_quantize_weight_2d needs a small caller-provided workspace (one 32-bit amax accumulator
// per matrix).  Some callers cannot hand one over: a plugin inside a host framework that owns all
// device memory and forbids side allocations, or a loop that must not call cudaMalloc because it
// synchronizes the device.  This entry point instead keeps that scratch in a fixed array compiled
// into the library, so it allocates nothing at call time.
//
// The array below is a host-side stand-in in host code: its name is not a device address there.
// The device address is looked up with cudaGetSymbolAddress once per device (on the first call made
// with that device current) and that pointer is what the kernels receive.
#include "../../include/mxnum.h"
#include "mx_internal.h"

#include <mutex>

namespace {

// One amax word per matrix; MX_NOALLOC_MAX_MATRICES words = 16 KiB.  Part of the library's device
// image: every GPU that loads the library holds it until the process exits.
static __device__ __align__(256) uint32_t g_w2d_noalloc_scratch[MX_NOALLOC_MAX_MATRICES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
uint32_t* g_scratch_dev_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up on first use per device.
cudaError_t scratch_for_current_device(uint32_t** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_dev_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_w2d_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_dev_ptr[dev] = static_cast<uint32_t*>(p);
    }
    *out = g_scratch_dev_ptr[dev];
    return cudaSuccess;
}

inline bool aligned16_na(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" mx_status mx_nvfp4_quantize_weight_2d_noalloc(const void* w, int64_t G, int64_t O, int64_t H,
                                                         uint8_t* q_row, uint8_t* s_row, uint8_t* q_col,
                                                         uint8_t* s_col, float* s_w, cudaStream_t stream) {
    if (!w || !q_row || !s_row || !q_col || !s_col || !s_w) return MX_ERR_INVALID_ARG;
    if (G <= 0 || O <= 0 || H <= 0) return MX_ERR_INVALID_ARG;
    if (G > MX_NOALLOC_MAX_MATRICES) return MX_ERR_UNSUPPORTED;      // more matrices than the fixed scratch holds
    if (!aligned16_na(w) || !aligned16_na(q_row) || !aligned16_na(s_row) || !aligned16_na(q_col) ||
        !aligned16_na(s_col) || !aligned16_na(s_w))
        return MX_ERR_ALIGNMENT;
    if ((O % 16) != 0 || (H % 16) != 0 || !mxk::weight_2d_grid_ok(G, O)) return MX_ERR_UNSUPPORTED;
    uint32_t* scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MX_ERR_CUDA;
    // the launcher zeroes scratch[0, G) on `stream` before accumulating into it
    const cudaError_t e = mxk::launch_nvfp4_weight_2d(static_cast<const uint16_t*>(w), G, O, H, q_row, s_row, q_col,
                                                      s_col, s_w, scratch, mxk::device_sm_count(), stream);
    return e == cudaSuccess ? MX_OK : MX_ERR_CUDA;
}
