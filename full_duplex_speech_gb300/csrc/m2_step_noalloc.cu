// mamba2_step_noalloc: the cached single-frame step for callers that cannot
// allocate device memory.
//
// mamba2_step needs a caller-provided workspace (the frame's post-conv
// activations and step sizes). Some callers have no way to provide one: a
// real-time frame loop that must not call cudaMalloc (it can synchronise the
// device and blow the 80 ms frame budget), a host program that hands this
// library only the tensors it already owns, or a foreign-language binding
// with no device allocator at all. For them this entry point uses a fixed
// scratch array that lives in the library's own device image instead.
//
// The scratch is a file-scope __device__ array of kScratchBytes (1 MiB); every
// GPU that loads the library holds it until the process exits. Its device
// address is looked up once per device (cudaGetSymbolAddress, with that device
// current) on the first call made there, and kept for the life of the process:
// calls after a cudaDeviceReset of that device are not supported. All calls
// share it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/mamba2.h"
#include "m2_launch.h"

namespace {

constexpr size_t kScratchBytes = size_t(1) << 20;
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_step_scratch[kScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" {

size_t mamba2_step_noalloc_max_bytes(void) { return kScratchBytes; }

m2_status mamba2_step_noalloc(const m2_dims* d, int n_sessions, const void* x, const void* B,
                              const void* C, const void* dt_raw, const float* A_log, const float* D,
                              const float* dt_bias, const float* conv_w, const float* conv_b,
                              float* ssm_state, void* conv_state, void* y, void* stream) {
    // The checks of mamba2_step come first and in its order (arguments, then
    // the size in place of its workspace check, then the device), so a NULL
    // pointer or a GPU other than sm_103 gives the status it gives there. A
    // request that does not fit is refused before touching the GPU.
    m2_status st = m2::check_step_args(d, n_sessions, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b,
                                       ssm_state, conv_state, y);
    if (st != M2_OK) return st;
    const size_t need = mamba2_step_workspace_bytes(d, n_sessions);
    if (need > kScratchBytes) return M2_EWORKSPACE;
    st = m2::check_device();
    if (st != M2_OK) return st;

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        m2::record_cuda_error(e);
        return M2_ECUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return M2_EUNSUPPORTED;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        if (!g_scratch_ptr[dev]) {
            // host code may not use g_step_scratch directly: it names a host-side
            // shadow, not device memory. Ask the runtime for this device's copy.
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_step_scratch);
            if (e != cudaSuccess) {
                m2::record_cuda_error(e);
                return M2_ECUDA;
            }
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    // The scratch needs no clearing: the step writes every byte it later reads
    // within the same call.
    return mamba2_step(d, n_sessions, x, B, C, dt_raw, A_log, D, dt_bias, conv_w, conv_b, ssm_state,
                       conv_state, y, scratch, kScratchBytes, stream);
}

}  // extern "C"
