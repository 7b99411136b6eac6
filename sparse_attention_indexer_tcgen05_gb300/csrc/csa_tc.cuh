// csa_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels of the CSA indexer step on sm_103a.
#pragma once

#include "csa_internal.cuh"

namespace csa {

// True when the tcgen05 score + top-k kernel takes this shape (bf16 values, H_I = 64, D_I = 128,
// every row's visible keys fit its shared-memory score buffer).
bool tc_score_supported(const Geo &g, bool bf16);

// Workspace the tensor-core kernels need (0 when none).
size_t tc_workspace_bytes(const Geo &g);

cudaError_t launch_score_topk_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w,
                                 const __nv_bfloat16 *k_idx, int32_t *ids, float *selscore, void *ws,
                                 cudaStream_t st);

// Same scores as launch_score_topk_tc, written densely for rows [row0, row0 + nrows) (test aid).
cudaError_t launch_score_dump_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w,
                                 const __nv_bfloat16 *k_idx, float *dump, long long row0, long long nrows,
                                 void *ws, cudaStream_t st);

// Reads and clears the tensor-core kernels' device error word (set when a kernel gives up a bounded
// wait on an mbarrier).  Synchronous: call after the stream has drained.
cudaError_t tc_read_clear_error(int *flag);

}  // namespace csa
