// hf_noalloc.cu -- hf_hybrid_forward for callers that cannot allocate device
// memory.
//
// The ordinary forward takes a caller-allocated workspace (pooled query and
// key blocks, the selected indices, the state in tensor-core operand layout,
// and the device status word).  Some callers have no way to provide one:
// a custom-operator interface that hands over only its inputs, outputs and a
// stream; code that runs while a stream is being captured into a CUDA graph,
// where cudaMalloc is not allowed; or an engine that owns every byte of the
// device through its own pool and gives plug-ins none of it.  For them this
// file keeps the workspace in a fixed, statically sized device array that
// the CUDA runtime creates when the library is loaded, and runs the same
// kernels on it.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "hf.h"
#include "hf_internal.h"

namespace {

// The workspace of hf_hybrid_forward_noalloc.  Every device that loads the
// library holds one copy until the process exits.  Zero-initialised at load.
static __device__ __align__(256) unsigned char g_noalloc_scratch[HF_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on `dev` (the current device).  The
// first call on a device looks it up with cudaGetSymbolAddress, which may
// load the module on that device; later calls read the cached address.
cudaError_t scratch_address(int dev, void** out)
{
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" {

hf_status hf_hybrid_forward_noalloc(const hf_config* cfg, const uint16_t* Q, const uint16_t* Kc,
                                    const uint16_t* Vc, int32_t slot_stride, const int32_t* slot_map,
                                    int32_t n_win, const float* S, const float* z, uint16_t* O,
                                    int32_t* idx_out, void** status_word, void* stream)
{
    size_t need = 0;
    hf_status s = hf_workspace_size(cfg, &need);   // validates cfg
    if (s != HF_OK) return s;
    need = hf::compact_workspace_bytes(cfg);       // without the buffer for splitting tile pairs
    if (need > (size_t)HF_NOALLOC_SCRATCH_BYTES) {
        return hf::set_last_error(HF_ERR_UNSUPPORTED,
                                  "hf_hybrid_forward_noalloc: this configuration needs %zu bytes of workspace, "
                                  "more than the %u-byte static scratch; use hf_hybrid_forward with a "
                                  "caller-allocated workspace",
                                  need, (unsigned)HF_NOALLOC_SCRATCH_BYTES);
    }
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= kMaxDevices)) e = cudaErrorInvalidDevice;
    void* ws = nullptr;
    if (e == cudaSuccess) e = scratch_address(dev, &ws);
    if (e != cudaSuccess) {
        return hf::set_last_error(HF_ERR_CUDA, "hf_hybrid_forward_noalloc: static scratch lookup on device %d: %s",
                                  dev, cudaGetErrorString(e));
    }
    if (status_word) *status_word = ws;
    return hf::forward_impl(cfg, Q, Kc, Vc, slot_stride, slot_map, n_win, S, z, O, idx_out, ws, stream, 0u, nullptr, nullptr,
                            false);
}

}  // extern "C"
