// k_score_tc.cu -- tcgen05 indexer-score + top-k kernel (placeholder until the tensor-core path lands).
#include "csa_tc.cuh"

namespace csa {

static __device__ int g_tc_error = 0;

cudaError_t tc_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_tc_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
}

bool tc_score_supported(const Geo &, bool) { return false; }
size_t tc_workspace_bytes(const Geo &) { return 0; }

cudaError_t launch_score_topk_tc(const Geo &, const __nv_bfloat16 *, const float *, const __nv_bfloat16 *,
                                 int32_t *, float *, void *, cudaStream_t)
{
    return cudaErrorNotSupported;
}

cudaError_t launch_score_dump_tc(const Geo &, const __nv_bfloat16 *, const float *, const __nv_bfloat16 *, float *,
                                 long long, long long, void *, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace csa
