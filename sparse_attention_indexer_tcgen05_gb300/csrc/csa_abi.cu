// csa_abi.cu -- the C ABI of libcsa_indexer.so: argument checks, workspace plan and kernel dispatch.
//
// Every entry point validates its arguments on the host before anything is enqueued, never allocates
// device memory, never synchronises (except csa_check_device_status), and returns a csa_status.
#include "csa_internal.cuh"
#include "csa_tc.cuh"

#include <math.h>
#include <stdlib.h>
#include <string.h>

using namespace csa;

#include <atomic>

namespace csa {
static std::atomic<unsigned long long> g_launches{0};
void note_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }
}  // namespace csa

namespace {

thread_local const char *t_last_path = "none";

constexpr size_t kAlign = 256;
inline size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

// Host-side fault injection for the error paths (CSA_FAULT=<site>): the named entry returns the
// named status without enqueueing anything.  Sites: invalid_arg, unsupported, alignment, workspace,
// cuda, timeout.  Read on every call so a test can set and clear it.
csa_status injected_fault()
{
    const char *f = getenv("CSA_FAULT");
    if (f == nullptr || f[0] == 0) return CSA_OK;
    if (!strcmp(f, "invalid_arg")) return CSA_ERR_INVALID_ARG;
    if (!strcmp(f, "unsupported")) return CSA_ERR_UNSUPPORTED;
    if (!strcmp(f, "alignment")) return CSA_ERR_ALIGNMENT;
    if (!strcmp(f, "workspace")) return CSA_ERR_WORKSPACE;
    if (!strcmp(f, "cuda")) return CSA_ERR_CUDA;
    if (!strcmp(f, "timeout")) return CSA_ERR_TIMEOUT;
    return CSA_OK;
}

struct Plan {
    Geo g;
    int dtype;
    bool require_tc;      // refuse the CUDA-core kernels of the score, teacher and backward steps
    bool dense_rescore;   // dense loss with K below the key width: visible scores go to the workspace
    size_t off_cu_c, off_teacher, off_g, off_rowloss, off_dk, off_dense, off_tc, off_btc, off_ttc, total;
};

csa_status make_plan(const csa_params *p, Plan *P)
{
    if (p == nullptr) return CSA_ERR_INVALID_ARG;
    if (p->layout < CSA_SBHD || p->layout > CSA_THD) return CSA_ERR_INVALID_ARG;
    if (p->dtype != CSA_F32 && p->dtype != CSA_BF16) return CSA_ERR_INVALID_ARG;
    if (p->compress_ratio < 1 || p->window < 0 || p->topk < 1) return CSA_ERR_INVALID_ARG;
    if (p->heads < 1 || p->head_dim < 1 || p->idx_heads < 1 || p->idx_dim < 1) return CSA_ERR_INVALID_ARG;
    if (p->sparse_loss != 0 && p->sparse_loss != 1) return CSA_ERR_INVALID_ARG;
    if (p->reduction != 0 && p->reduction != 1) return CSA_ERR_INVALID_ARG;
    if (p->teacher_mode != CSA_TEACHER_FULL && p->teacher_mode != CSA_TEACHER_COMPRESSED_ONLY) return CSA_ERR_INVALID_ARG;
    if (p->require_tensor_cores != 0 && p->require_tensor_cores != 1) return CSA_ERR_INVALID_ARG;
    if (!isfinite(p->softmax_scale) || !isfinite(p->loss_coeff)) return CSA_ERR_INVALID_ARG;
    if (p->batch < 1 || p->seqlen < 0) return CSA_ERR_INVALID_ARG;

    Geo g;
    memset(&g, 0, sizeof g);
    g.layout = p->layout;
    g.B = p->batch;
    g.S = p->seqlen;
    g.ratio = p->compress_ratio;
    // the compressed-only teacher is the full one with no window and no sink
    g.window = p->teacher_mode == CSA_TEACHER_COMPRESSED_ONLY ? 0 : p->window;
    g.no_sink = p->teacher_mode == CSA_TEACHER_COMPRESSED_ONLY ? 1 : 0;
    g.H = p->heads;
    g.D = p->head_dim;
    g.HI = p->idx_heads;
    g.DI = p->idx_dim;
    g.scale = p->softmax_scale;
    g.sparse = p->sparse_loss;
    long long rows;
    if (p->layout == CSA_THD) {
        if (p->cu_seqlens_q == nullptr || p->max_seqlen_q < 0 || p->key_rows < 0) return CSA_ERR_INVALID_ARG;
        if (p->max_seqlen_q > p->seqlen) return CSA_ERR_INVALID_ARG;
        rows = p->seqlen;
        g.nc = 0;
        g.NC = p->max_seqlen_q / p->compress_ratio;
        g.key_rows = p->key_rows;
        g.cu_q = p->cu_seqlens_q;
        g.cu_real = p->cu_seqlens_q_unpadded ? p->cu_seqlens_q_unpadded : p->cu_seqlens_q;
    } else {
        rows = (long long)p->batch * p->seqlen;
        g.nc = p->seqlen / p->compress_ratio;
        g.NC = g.nc;
        long long kr = (long long)p->batch * g.nc;
        if (p->key_rows != 0 && p->key_rows != kr) return CSA_ERR_INVALID_ARG;
        g.key_rows = kr;
    }
    if (rows > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;
    g.rows = (int)rows;
    g.K = p->topk < g.NC ? p->topk : g.NC;
    g.TW = g.sparse ? g.K : g.NC;
    const double f = p->reduction == 0 ? (rows > 0 ? (double)p->loss_coeff / (double)rows : 0.0) : p->loss_coeff;
    g.factor = (float)f;
    // index arithmetic is 64-bit; per-row element counts must stay inside int
    if ((long long)g.HI * g.DI > 0x7fffffffLL || (long long)g.H * g.D > 0x7fffffffLL) return CSA_ERR_UNSUPPORTED;

    P->g = g;
    P->dtype = p->dtype;
    P->require_tc = p->require_tensor_cores != 0;
    P->dense_rescore = !g.sparse && g.K < g.NC;
    size_t off = 0;
    P->off_cu_c = off;
    off = align_up(off + sizeof(int) * (size_t)(p->layout == CSA_THD ? p->batch + 1 : 1));
    P->off_teacher = off;
    off = align_up(off + sizeof(float) * (size_t)rows * g.TW);
    // g by slot for the CUDA-core backward and the tensor-core one on long key axes, or g by key (inside the
    // tensor-core backward's region) for the tensor-core one on short key axes
    const bool tc_bwd = tc_bwd_supported(g, p->dtype == CSA_BF16);
    const bool by_key = tc_bwd && !tc_bwd_long(g);
    P->off_g = off;
    off = align_up(off + (by_key ? 0 : sizeof(float) * (size_t)rows * g.TW));
    P->off_rowloss = off;
    off = align_up(off + sizeof(float) * (size_t)(rows > 0 ? rows : 1));
    P->off_dk = off;
    off = align_up(off + sizeof(float) * (size_t)g.key_rows * g.DI);
    P->off_dense = off;
    off = align_up(off + (P->dense_rescore ? sizeof(float) * (size_t)rows * g.NC : 0));
    P->off_tc = off;
    off = align_up(off + tc_workspace_bytes(g));
    P->off_btc = off;
    off = align_up(off + (tc_bwd ? tc_bwd_workspace_bytes(g) : 0));
    P->off_ttc = off;
    off = align_up(off + tc_teacher_workspace_bytes(g));
    P->total = off;
    return CSA_OK;
}

inline bool aligned(const void *ptr, size_t a) { return ((uintptr_t)ptr & (a - 1)) == 0; }

// A tensor argument: must be non-null and 16-byte aligned whenever it holds at least one element.
inline csa_status need(const void *ptr, long long elems)
{
    if (elems <= 0) return CSA_OK;
    if (ptr == nullptr) return CSA_ERR_INVALID_ARG;
    return aligned(ptr, 16) ? CSA_OK : CSA_ERR_ALIGNMENT;
}

#define CSA_TRY(x)                                    \
    do {                                              \
        csa_status _s = (x);                          \
        if (_s != CSA_OK) return _s;                  \
    } while (0)

thread_local const char *t_last_cuda_error = "no error";
thread_local int32_t t_last_timeout_site = 0;

// A failed CUDA call ends the entry point with CSA_ERR_CUDA and leaves its message for csa_last_cuda_error.
#define CSA_CUDA(x)                                     \
    do {                                                \
        const cudaError_t csa_e_ = (x);                 \
        if (csa_e_ != cudaSuccess) {                    \
            t_last_cuda_error = cudaGetErrorString(csa_e_); \
            return CSA_ERR_CUDA;                        \
        }                                               \
    } while (0)

int g_max_smem = -1;

csa_status check_smem(size_t bytes)
{
    if (g_max_smem < 0) {
        int dev = 0;
        CSA_CUDA(cudaGetDevice(&dev));
        CSA_CUDA(cudaDeviceGetAttribute(&g_max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev));
    }
    return bytes <= (size_t)g_max_smem ? CSA_OK : CSA_ERR_UNSUPPORTED;
}

char *ws_at(void *ws, size_t off) { return static_cast<char *>(ws) + off; }

// With require_tensor_cores set: CSA_ERR_UNSUPPORTED, before anything is enqueued, when a step of the call would run
// a CUDA-core kernel for its contraction (the score, the teacher, or the backward, including the dense loss's
// rescoring of the visible keys).
csa_status check_required_tc(const Plan &P, bool fwd, bool teacher, bool bwd)
{
    if (!P.require_tc) return CSA_OK;
    const bool bf16 = P.dtype == CSA_BF16;
    if (fwd && !tc_score_supported(P.g, bf16)) return CSA_ERR_UNSUPPORTED;
    if (teacher && !tc_teacher_supported(P.g, bf16) && !tc_teacher_h128_supported(P.g, bf16)) return CSA_ERR_UNSUPPORTED;
    if (bwd && (!tc_bwd_supported(P.g, bf16) || P.dense_rescore)) return CSA_ERR_UNSUPPORTED;
    return CSA_OK;
}

// Per-call prologue shared by the three calls: THD compressed offsets into the workspace.
csa_status prologue(Plan &P, void *ws, cudaStream_t st)
{
    if (P.g.layout == CSA_THD) {
        int *cu_c = reinterpret_cast<int *>(ws_at(ws, P.off_cu_c));
        P.g.cu_c = cu_c;
        CSA_CUDA(launch_build_cu_c(P.g, cu_c, st));
    }
    return CSA_OK;
}

template <typename T>
csa_status run_fwd(Plan &P, const void *q_idx, const float *w, const void *k_idx, int32_t *ids, float *selscore,
                   float *dump, long long row0, long long nrows, void *ws, cudaStream_t st)
{
    CSA_TRY(prologue(P, ws, st));
    if (tc_score_supported(P.g, sizeof(T) == 2) && dump == nullptr) {
        t_last_path = "tcgen05";
        CSA_CUDA(launch_score_topk_tc(P.g, (const __nv_bfloat16 *)q_idx, w, (const __nv_bfloat16 *)k_idx, ids,
                                      selscore, ws_at(ws, P.off_tc), st));
        return CSA_OK;
    }
    if (tc_score_supported(P.g, sizeof(T) == 2) && dump != nullptr) {
        t_last_path = "tcgen05";
        CSA_CUDA(launch_score_dump_tc(P.g, (const __nv_bfloat16 *)q_idx, w, (const __nv_bfloat16 *)k_idx, dump,
                                      row0, nrows, ws_at(ws, P.off_tc), st));
        return CSA_OK;
    }
    CSA_TRY(check_smem(score_topk_generic_smem(P.g)));
    t_last_path = "generic";
    CSA_CUDA(launch_score_topk_generic<T>(P.g, (const T *)q_idx, w, (const T *)k_idx, ids, selscore, dump, row0,
                                          nrows, st));
    return CSA_OK;
}

template <typename T>
csa_status run_teacher(Plan &P, const void *q, const void *kv, const void *kv_c, const float *sink,
                       const int32_t *ids, float *teacher, void *ws, cudaStream_t st, const TeacherKl *kl = nullptr,
                       bool *kl_done = nullptr)
{
    if (kl_done != nullptr) *kl_done = false;
    if (tc_teacher_supported(P.g, sizeof(T) == 2)) {
        t_last_path = "tcgen05";
        CSA_CUDA(launch_teacher_tc(P.g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kv,
                                   (const __nv_bfloat16 *)kv_c, sink, ids, teacher, ws_at(ws, P.off_ttc), st));
        return CSA_OK;
    }
    if (tc_teacher_h128_supported(P.g, sizeof(T) == 2)) {
        t_last_path = "tcgen05";
        CSA_CUDA(launch_teacher_h128_tc(P.g, (const __nv_bfloat16 *)q, (const __nv_bfloat16 *)kv,
                                        (const __nv_bfloat16 *)kv_c, sink, ids, teacher, kl, st));
        if (kl_done != nullptr) *kl_done = kl != nullptr;
        return CSA_OK;
    }
    CSA_TRY(check_smem(teacher_generic_smem(P.g, sizeof(T) == 2)));
    t_last_path = "generic";
    CSA_CUDA(launch_teacher_generic<T>(P.g, (const T *)q, (const T *)kv, (const T *)kv_c, sink, ids, teacher, st));
    return CSA_OK;
}

template <typename T>
csa_status run_bwd(Plan &P, const void *q_idx, const float *w, const void *k_idx, const void *q, const void *kv,
                   const void *kv_c, const float *sink, const int32_t *ids, const float *selscore,
                   const float *teacher_in, float *loss, float *row_loss_out, void *dq_idx, float *dw,
                   void *dk_idx, void *ws, float *dk_acc, cudaStream_t st)
{
    CSA_TRY(prologue(P, ws, st));
    const Geo &g = P.g;
    float *gbuf = reinterpret_cast<float *>(ws_at(ws, P.off_g));
    float *row_loss = row_loss_out ? row_loss_out : reinterpret_cast<float *>(ws_at(ws, P.off_rowloss));
    const bool tc = tc_bwd_supported(g, sizeof(T) == 2);
    const bool by_key = tc && !tc_bwd_long(g);
    char *btc = ws_at(ws, P.off_btc);
    float *gd = by_key ? tc_bwd_gd(g, btc) : nullptr;
    // the tensor-core backward on short key axes reads g by key only; the slot-layout rows serve the CUDA-core
    // backward and the tensor-core one on long key axes
    float *g_slot = by_key ? nullptr : gbuf;
    const int ncp = by_key ? tc_bwd_ncp(g) : 0;
    const float *teacher = teacher_in;
    bool kl_done = false;
    if (teacher == nullptr) {
        // with the sparse loss the 128-head teacher takes the KL step itself (its rows then never go to memory)
        const TeacherKl kl = {selscore, g_slot, gd, ncp, row_loss};
        const bool fuse = g.sparse && !P.dense_rescore && g.TW == g.K;
        float *tbuf = reinterpret_cast<float *>(ws_at(ws, P.off_teacher));
        CSA_TRY(run_teacher<T>(P, q, kv, kv_c, sink, ids, tbuf, ws, st, fuse ? &kl : nullptr, &kl_done));
        teacher = tbuf;
    }
    if (!kl_done) {
        const float *dense_scores = nullptr;
        if (P.dense_rescore) {
            float *ds = reinterpret_cast<float *>(ws_at(ws, P.off_dense));
            CSA_TRY(check_smem(score_topk_generic_smem(g)));
            CSA_CUDA(launch_score_topk_generic<T>(g, (const T *)q_idx, w, (const T *)k_idx, nullptr, nullptr, ds, 0,
                                                  g.rows, st));
            dense_scores = ds;
        }
        CSA_CUDA(launch_kl(g, ids, selscore, dense_scores, teacher, g_slot, row_loss, gd, ncp, st));
    }
    if (g.key_rows * g.DI > 0)
        CSA_CUDA(cudaMemsetAsync(dk_acc, 0, sizeof(float) * (size_t)g.key_rows * g.DI, st));
    if (tc) {
        t_last_path = "tcgen05";
        CSA_CUDA(launch_bwd_tc(g, (const __nv_bfloat16 *)q_idx, w, (const __nv_bfloat16 *)k_idx, (__nv_bfloat16 *)dq_idx,
                               dw, dk_acc, btc, ids, gbuf, st));
    } else {
        CSA_TRY(check_smem(grad_generic_smem(g)));
        t_last_path = "generic";
        CSA_CUDA(launch_grad_generic<T>(g, (const T *)q_idx, w, (const T *)k_idx, ids, gbuf, (T *)dq_idx, dw, dk_acc,
                                        st));
    }
    CSA_CUDA(launch_finalize<T>(g, dk_acc, (T *)dk_idx, row_loss, loss, st));
    return CSA_OK;
}

}  // namespace

extern "C" {

int32_t csa_topk_width(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.g.K : -1;
}

int32_t csa_key_width(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.g.NC : -1;
}

int32_t csa_teacher_width(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.g.TW : -1;
}

int64_t csa_rows(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.g.rows : -1;
}

int64_t csa_compressed_rows(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.g.key_rows : -1;
}

size_t csa_workspace_size(const csa_params *p)
{
    Plan P;
    return make_plan(p, &P) == CSA_OK ? P.total : 0;
}

csa_status csa_indexer_fwd(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                           int32_t *ids_out, float *selscore_out, void *workspace, size_t workspace_bytes,
                           void *stream)
{
    CSA_TRY(injected_fault());
    Plan P;
    CSA_TRY(make_plan(p, &P));
    const Geo &g = P.g;
    CSA_TRY(need(q_idx, (long long)g.rows * g.HI * g.DI));
    CSA_TRY(need(w, (long long)g.rows * g.HI));
    CSA_TRY(need(k_idx, g.key_rows * g.DI));
    CSA_TRY(need(ids_out, (long long)g.rows * g.K));
    CSA_TRY(need(selscore_out, (long long)g.rows * g.K));
    if (workspace_bytes < P.total || (P.total > 0 && workspace == nullptr)) return CSA_ERR_WORKSPACE;
    CSA_TRY(check_required_tc(P, true, false, false));
    if (g.rows == 0) return CSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (P.dtype == CSA_BF16)
        return run_fwd<__nv_bfloat16>(P, q_idx, w, k_idx, ids_out, selscore_out, nullptr, 0, 0, workspace, st);
    return run_fwd<float>(P, q_idx, w, k_idx, ids_out, selscore_out, nullptr, 0, 0, workspace, st);
}

csa_status csa_scores_debug(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                            int64_t row_begin, int64_t row_count, float *scores_out, void *workspace,
                            size_t workspace_bytes, void *stream)
{
    CSA_TRY(injected_fault());
    Plan P;
    CSA_TRY(make_plan(p, &P));
    const Geo &g = P.g;
    if (row_begin < 0 || row_count < 0 || row_begin + row_count > g.rows) return CSA_ERR_INVALID_ARG;
    CSA_TRY(need(q_idx, (long long)g.rows * g.HI * g.DI));
    CSA_TRY(need(w, (long long)g.rows * g.HI));
    CSA_TRY(need(k_idx, g.key_rows * g.DI));
    CSA_TRY(need(scores_out, row_count * g.NC));
    if (workspace_bytes < P.total || (P.total > 0 && workspace == nullptr)) return CSA_ERR_WORKSPACE;
    CSA_TRY(check_required_tc(P, true, false, false));
    if (row_count == 0 || g.NC == 0) return CSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (P.dtype == CSA_BF16)
        return run_fwd<__nv_bfloat16>(P, q_idx, w, k_idx, nullptr, nullptr, scores_out, row_begin, row_count,
                                      workspace, st);
    return run_fwd<float>(P, q_idx, w, k_idx, nullptr, nullptr, scores_out, row_begin, row_count, workspace, st);
}

csa_status csa_teacher(const csa_params *p, const void *q, const void *kv, const void *kv_c, const float *sink,
                       const int32_t *ids, float *teacher_out, void *workspace, size_t workspace_bytes, void *stream)
{
    CSA_TRY(injected_fault());
    Plan P;
    CSA_TRY(make_plan(p, &P));
    const Geo &g = P.g;
    CSA_TRY(need(q, (long long)g.rows * g.H * g.D));
    CSA_TRY(need(kv, (long long)g.rows * g.D));
    CSA_TRY(need(kv_c, g.key_rows * g.D));
    CSA_TRY(need(sink, g.H));
    CSA_TRY(need(ids, (long long)g.rows * g.K));
    CSA_TRY(need(teacher_out, (long long)g.rows * g.TW));
    if (workspace_bytes < P.total || (P.total > 0 && workspace == nullptr)) return CSA_ERR_WORKSPACE;
    CSA_TRY(check_required_tc(P, false, true, false));
    if (g.rows == 0 || g.TW == 0) return CSA_OK;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CSA_TRY(prologue(P, workspace, st));
    if (P.dtype == CSA_BF16) return run_teacher<__nv_bfloat16>(P, q, kv, kv_c, sink, ids, teacher_out, workspace, st);
    return run_teacher<float>(P, q, kv, kv_c, sink, ids, teacher_out, workspace, st);
}

csa_status csa_teacher_from_lse(const csa_params *p, const void *q, const void *kv_c, const float *lse_nc,
                                const int32_t *ids, float *teacher_out, void *workspace, size_t workspace_bytes,
                                void *stream)
{
    CSA_TRY(injected_fault());
    Plan P;
    CSA_TRY(make_plan(p, &P));
    Geo &g = P.g;
    CSA_TRY(need(q, (long long)g.rows * g.H * g.D));
    CSA_TRY(need(kv_c, g.key_rows * g.D));
    CSA_TRY(need(lse_nc, (long long)g.rows * g.H));
    CSA_TRY(need(ids, (long long)g.rows * g.K));
    CSA_TRY(need(teacher_out, (long long)g.rows * g.TW));
    if (workspace_bytes < P.total || (P.total > 0 && workspace == nullptr)) return CSA_ERR_WORKSPACE;
    CSA_TRY(check_required_tc(P, false, true, false));
    if (g.rows == 0 || g.TW == 0) return CSA_OK;
    // the given log-sum-exp carries the whole non-compressed part of each head's denominator
    g.window = 0;
    g.no_sink = 0;
    g.lse_nc = lse_nc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    CSA_TRY(prologue(P, workspace, st));
    // kv is never read without a window: kv_c stands in for it
    if (P.dtype == CSA_BF16)
        return run_teacher<__nv_bfloat16>(P, q, kv_c, kv_c, nullptr, ids, teacher_out, workspace, st);
    return run_teacher<float>(P, q, kv_c, kv_c, nullptr, ids, teacher_out, workspace, st);
}

csa_status csa_indexer_bwd(const csa_params *p, const void *q_idx, const float *w, const void *k_idx, const void *q,
                           const void *kv, const void *kv_c, const float *sink, const int32_t *ids,
                           const float *selscore, const float *teacher_or_null, float *loss_out,
                           float *row_loss_out, void *dq_idx, float *dw, void *dk_idx, void *workspace,
                           size_t workspace_bytes, void *stream)
{
    CSA_TRY(injected_fault());
    Plan P;
    CSA_TRY(make_plan(p, &P));
    const Geo &g = P.g;
    CSA_TRY(need(q_idx, (long long)g.rows * g.HI * g.DI));
    CSA_TRY(need(w, (long long)g.rows * g.HI));
    CSA_TRY(need(k_idx, g.key_rows * g.DI));
    if (teacher_or_null == nullptr) {
        CSA_TRY(need(q, (long long)g.rows * g.H * g.D));
        CSA_TRY(need(kv, (long long)g.rows * g.D));
        CSA_TRY(need(kv_c, g.key_rows * g.D));
        CSA_TRY(need(sink, g.H));
    } else {
        CSA_TRY(need(teacher_or_null, (long long)g.rows * g.TW));
    }
    CSA_TRY(need(ids, (long long)g.rows * g.K));
    CSA_TRY(need(selscore, (long long)g.rows * g.K));
    if (loss_out == nullptr) return CSA_ERR_INVALID_ARG;
    if (!aligned(loss_out, 4)) return CSA_ERR_ALIGNMENT;
    if (row_loss_out != nullptr && !aligned(row_loss_out, 4)) return CSA_ERR_ALIGNMENT;
    CSA_TRY(need(dq_idx, (long long)g.rows * g.HI * g.DI));
    CSA_TRY(need(dw, (long long)g.rows * g.HI));
    CSA_TRY(need(dk_idx, g.key_rows * g.DI));
    if (workspace_bytes < P.total || (P.total > 0 && workspace == nullptr)) return CSA_ERR_WORKSPACE;
    CSA_TRY(check_required_tc(P, false, teacher_or_null == nullptr, true));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    float *dk_acc = reinterpret_cast<float *>(ws_at(workspace, P.off_dk));
    if (P.dtype == CSA_BF16)
        return run_bwd<__nv_bfloat16>(P, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore, teacher_or_null,
                                      loss_out, row_loss_out, dq_idx, dw, dk_idx, workspace, dk_acc, st);
    return run_bwd<float>(P, q_idx, w, k_idx, q, kv, kv_c, sink, ids, selscore, teacher_or_null, loss_out,
                          row_loss_out, dq_idx, dw, dk_idx, workspace, dk_acc, st);
}

csa_status csa_check_device_status(void *stream)
{
    CSA_TRY(injected_fault());
    CSA_CUDA(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    int flag = 0, flag2 = 0;
    CSA_CUDA(tc_read_clear_error(&flag));
    CSA_CUDA(selftest_read_clear_error(&flag2));
    if (flag == 0 && flag2 == 0) return CSA_OK;
    t_last_timeout_site = flag != 0 ? flag : 900 + flag2;
    return CSA_ERR_TIMEOUT;
}

int32_t csa_last_timeout_site(void) { return t_last_timeout_site; }

csa_status csa_selftest_bounded_wait(void *stream)
{
    CSA_TRY(injected_fault());
    CSA_CUDA(launch_bounded_wait_selftest(static_cast<cudaStream_t>(stream)));
    return CSA_OK;
}

const char *csa_last_path(void) { return t_last_path; }

const char *csa_last_cuda_error(void) { return t_last_cuda_error; }

uint64_t csa_kernel_launches(void) { return (uint64_t)g_launches.load(std::memory_order_relaxed); }

const char *csa_status_string(csa_status s)
{
    switch (s) {
    case CSA_OK: return "CSA_OK";
    case CSA_ERR_INVALID_ARG: return "CSA_ERR_INVALID_ARG: null, negative or inconsistent argument";
    case CSA_ERR_UNSUPPORTED: return "CSA_ERR_UNSUPPORTED: shape or dtype combination not implemented";
    case CSA_ERR_ALIGNMENT: return "CSA_ERR_ALIGNMENT: tensor pointer not 16-byte aligned";
    case CSA_ERR_WORKSPACE: return "CSA_ERR_WORKSPACE: workspace smaller than csa_workspace_size()";
    case CSA_ERR_CUDA: return "CSA_ERR_CUDA: a CUDA runtime call failed";
    case CSA_ERR_TIMEOUT: return "CSA_ERR_TIMEOUT: a kernel gave up a bounded wait";
    }
    return "CSA_ERR_UNKNOWN";
}

}  // extern "C"
