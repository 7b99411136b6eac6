// csa_tc.cuh -- tensor-core (tcgen05 / TMEM / TMA) kernels of the CSA indexer step on sm_103a.
#pragma once

#include "csa_internal.cuh"

#include <cuda.h>

namespace csa {

// True when the tcgen05 score + top-k kernels take this shape (bf16 values, H_I = 64, D_I = 128): key axes up to
// 1024 with whole score rows in shared memory, longer ones with streamed score tiles and per-row candidate buffers.
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

// TMA tensor maps (bf16, 128-byte swizzle; rank <= 5): q_idx as [rows][H_I][D_I] with a 64 x H_I x 1 box, and k_idx with a
// 64 x 128-key box (2D over key rows, or 3D [n_c][B][D_I] for SBHD).
bool tc_encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box);
bool tc_encode_q_map(CUtensorMap *m, const void *q_idx, const Geo &g);
// fp32, no swizzle (rank <= 5; strides in bytes, multiples of 16)
bool tc_encode_f32(CUtensorMap *m, const float *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box);
bool tc_encode_k_map(CUtensorMap *m, const void *k_idx, const Geo &g);

// Tensor-core backward (dQ_idx, dW, dK) for bf16, H_I = 64, D_I = 128: any key axis with the sparse loss, key
// axes up to 1024 with the dense loss.
bool tc_bwd_supported(const Geo &g, bool bf16);
// Long key axis (more than 1024 keys): g stays in the KL step's slot layout and the kernels build g tiles.
bool tc_bwd_long(const Geo &g);
int tc_bwd_tiles(const Geo &g);
// Row stride (floats) of the by-key gradient rows gd[rows][ncp] the KL step writes for the backward (short axis).
int tc_bwd_ncp(const Geo &g);
size_t tc_bwd_workspace_bytes(const Geo &g);
// Where gd (short axis) or the per-row tile offsets (long axis) live inside that workspace.
float *tc_bwd_gd(const Geo &g, void *ws);
// ws: tc_bwd_workspace_bytes(g) bytes; short axis: its gd rows hold dloss/dI[row][key] for every visible key;
// long axis: gslot [rows][K] holds dloss/dI by slot of the ascending ids.
cudaError_t launch_bwd_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                          __nv_bfloat16 *dq, float *dw, float *dk_acc, void *ws, const int32_t *ids,
                          const float *gslot, cudaStream_t st);
cudaError_t bwd_tc_read_clear_error(int *flag);
// Long key axes: the row-owner backward (dQ_idx, dW) over each row's selected keys only (k_bwd_gather_tc.cu);
// gslot [rows][K] holds dloss/dI by slot of the ascending ids; sgn [rows][K] receives the signs of x per slot.
cudaError_t launch_dq_dw_gather_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                                   const int32_t *ids, const float *gslot, __nv_bfloat16 *dq, float *dw,
                                   unsigned long long *sgn, cudaStream_t st);
cudaError_t bwd_gather_read_clear_error(int *flag);

// Tensor-core teacher for bf16, H = 64, D in {64, 128, 192}, key axis <= 1024.
bool tc_teacher_supported(const Geo &g, bool bf16);
size_t tc_teacher_workspace_bytes(const Geo &g);
cudaError_t launch_teacher_tc(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *kv,
                              const __nv_bfloat16 *kv_c, const float *sink, const int32_t *ids, float *teacher,
                              void *ws, cudaStream_t st);
cudaError_t teacher_tc_read_clear_error(int *flag);

// Tensor-core teacher for bf16, H = 128, D a multiple of 64 up to 512, teacher rows up to 2048 wide: one query
// row per work item, q in TMEM, the selected compressed keys gathered (sparse loss) or tiled (dense loss).
bool tc_teacher_h128_supported(const Geo &g, bool bf16);
// The KL step taken inside the teacher (sparse loss, teacher width K): from the row's selected scores and its
// normalised teacher, the row's KL goes to row_loss and g to gslot (by slot, [rows][K]) and/or gkey (by key,
// row gd_row_of(...) of stride ncp, its visible range zeroed first); either may be null.  The teacher rows are
// then not written.
struct TeacherKl {
    const float *selscore;
    float *gslot;
    float *gkey;
    int ncp;
    float *row_loss;
};
cudaError_t launch_teacher_h128_tc(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *kv,
                                   const __nv_bfloat16 *kv_c, const float *sink, const int32_t *ids, float *teacher,
                                   const TeacherKl *kl, cudaStream_t st);
cudaError_t teacher_h128_read_clear_error(int *flag);

// One tiny kernel whose bounded wait (about 1 ms) on a barrier nothing arrives on runs out (k_selftest.cu), and
// the read-and-clear of the word it sets.
cudaError_t launch_bounded_wait_selftest(cudaStream_t st);
cudaError_t selftest_read_clear_error(int *flag);

// Reads and clears the tensor-core kernels' device error word (set when a kernel gives up a bounded
// wait on an mbarrier).  Synchronous: call after the stream has drained.
cudaError_t tc_read_clear_error(int *flag);

}  // namespace csa
