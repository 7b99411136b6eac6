// csa_noalloc.cu -- csa_indexer_bwd for callers that cannot allocate device memory.
//
// Some callers have no way to hand the library a workspace: code that runs inside a framework's
// allocator-free region, a plugin whose host application owns every device allocation, or a process
// that must not call cudaMalloc after start-up (it would synchronise the device or break a memory
// budget fixed up front).  For them this file keeps the backward's scratch -- THD segment offsets, the
// teacher and dL/dI rows, per-row losses and the fp32 dK accumulator -- in one file-scope device array
// of fixed size, reserved when the library's device code is loaded on a GPU and held until the process
// exits.  Nothing here allocates or frees memory.
#include "csa_internal.cuh"

#include <mutex>

// The scratch.  Its host-side name is only a stand-in for the symbol: host code must never pass it to a
// kernel; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[CSA_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per device.
csa_status scratch_on_current_device(void **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return CSA_ERR_CUDA;
        g_scratch[dev] = ptr;
    }
    *out = g_scratch[dev];
    return CSA_OK;
}

}  // namespace

extern "C" csa_status csa_indexer_bwd_noalloc(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                                              const void *q, const void *kv, const void *kv_c, const float *sink,
                                              const int32_t *ids, const float *selscore,
                                              const float *teacher_or_null, float *loss_out, float *row_loss_out,
                                              void *dq_idx, float *dw, void *dk_idx, void *stream)
{
    const size_t need = csa_workspace_size(p);
    if (need == 0) return CSA_ERR_INVALID_ARG;
    if (need > (size_t)CSA_NOALLOC_SCRATCH_BYTES) return CSA_ERR_WORKSPACE;  // problem too large for the scratch
    void *scratch = nullptr;
    const csa_status s = scratch_on_current_device(&scratch);
    if (s != CSA_OK) return s;
    // csa_indexer_bwd overwrites or zeroes (the dK accumulator) every part of the scratch it reads
    return csa_indexer_bwd(p, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore, teacher_or_null, loss_out,
                           row_loss_out, dq_idx, dw, dk_idx, scratch, (size_t)CSA_NOALLOC_SCRATCH_BYTES, stream);
}
