/*
 * csa_indexer.h -- C ABI of the GB300 (sm_103a) CSA Lightning-Indexer training step.
 *
 * The step (one pass of the hot path):
 *   1. indexer scores  I[t,s] = sum_j w[t,j] * max(0, q_idx[t,j] . k_idx[s])  over the compressed keys
 *      that are causally visible to row t;
 *   2. per-row top-k of I with global key ids;
 *   3. the full-CSA teacher t over the selected compressed keys, whose per-head denominator holds the
 *      attention sink, the sliding window of original KV and the selected compressed KV together;
 *   4. KL(t || softmax of I over the same support);
 *   5. the indexer backward: dQ_idx, dW, dK_idx.
 *
 * Sources, cited by page title and section:
 *   [BUG] "[Bug] DSV4 unfused CSA indexer loss uses a compressed-only teacher instead of the full CSA
 *         attention distribution" (Megatron-LM issue #5776), with its code excerpts (csa.py, dsa.py,
 *         dsa_kernels.py) and the follow-up proposal and review comments.
 *   [PR]  "Megatron-LM PR #8539" (cuDNN frontend 1.26 default changes).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers, except where a comment says otherwise.  The caller owns
 *     every buffer; the library never allocates device memory and never synchronises the stream
 *     (except csa_check_device_status, which exists to do exactly that).  Work is enqueued on `stream`
 *     (a cudaStream_t; NULL is the legacy default stream) in order.
 *   - Inputs are const and never written.  Outputs are fully overwritten.
 *   - Errors are returned, never trapped: invalid arguments are rejected before anything is enqueued,
 *     and unsupported shape/dtype combinations fail closed (no silent fallback).
 *   - "value" tensors (q_idx, k_idx, q, kv, kv_c and the gradients dq_idx, dk_idx) share the element type
 *     csa_params.dtype (fp32 or bf16); w, sink, selscore, teacher, dw and the loss are always fp32.
 *
 * Layouts ([BUG] sec. 1 and sec. 2 excerpts: [sq, b, np, hn] for queries, [sk, b, np, hn] for keys):
 *   SBHD: q_idx [S, B, H_I, D_I]   w [S, B, H_I]   q [S, B, H, D]   kv [S, B, D]
 *         k_idx [n_c, B, D_I]      kv_c [n_c, B, D]                      (n_c = S / compress_ratio)
 *   BSHD: the same with the first two dimensions swapped ([B, S, ...], [B, n_c, ...]).
 *   THD:  q_idx [T, H_I, D_I] ... kv [T, D]; k_idx [T_c, D_I], kv_c [T_c, D].  Segment b holds rows
 *         cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 (physical; trailing padding may be absorbed into the last
 *         segment).  Its real length L_b comes from cu_seqlens_q_unpadded (or cu_seqlens_q when NULL); rows
 *         at positions >= L_b are padding.  Its compressed keys are rows cu_c[b] .. cu_c[b] + L_b/r - 1 of
 *         k_idx / kv_c with cu_c = [0, cumsum(L_b / r)] built from the UNPADDED lengths ([BUG] sec. 1 THD
 *         excerpt: compressed cu_seqlens rebuilt from unpadded Q lengths); compressed rows produced by the
 *         padding may follow and are never read.
 *   kv and kv_c are single-head (MQA) tensors shared by every main-attention head.
 *
 * Row semantics (row t of segment b at 1-based position i; r = compress_ratio):
 *   visible keys    j < i / r (integer division) -- the compressed causal mask of [BUG] sec. 1 excerpt
 *                   (where(arange(n_c) >= positions // ratio, -inf, 0)), anchored per segment;
 *   K               = min(topk, n_c) (SBHD/BSHD) or min(topk, max_seqlen_q / r) (THD, longest unpadded segment)
 *                     ([BUG] sec. 1 excerpts: min(index_topk, n_compressed / max_seqlen_compressed));
 *   selection       the k_t = min(K, v_t) largest scores, ties to the lower key index (-0.0 == +0.0);
 *   global ids      b * n_c + j (SBHD/BSHD) or cu_c[b] + j (THD) ([PR] item 1: global ids b*S_k + local);
 *   id slot order   ascending id, then -1 pads ([BUG] sec. 3 excerpt: invalid slots are -1);
 *   window          the W original positions ending at and including the query, cut at the segment start;
 *   padding rows    ids -1, scores -inf, teacher 0, loss 0, gradients 0 ([BUG] fused-path excerpt:
 *                   padding_row_mask); they still count in the mean's divisor (the review comment on the
 *                   physical total_q divisor).
 */
#ifndef CSA_INDEXER_H
#define CSA_INDEXER_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    CSA_OK = 0,
    CSA_ERR_INVALID_ARG = 1,   /* null/negative/inconsistent argument */
    CSA_ERR_UNSUPPORTED = 2,   /* valid but not implemented (shape beyond a kernel's limit, ...) */
    CSA_ERR_ALIGNMENT = 3,     /* a pointer is not aligned to its element type (16 B for value tensors) */
    CSA_ERR_WORKSPACE = 4,     /* workspace smaller than csa_workspace_size() */
    CSA_ERR_CUDA = 5,          /* a CUDA runtime call failed (launch error, no device, ...) */
    CSA_ERR_TIMEOUT = 6        /* a kernel gave up a bounded wait (reported by csa_check_device_status) */
} csa_status;

typedef enum { CSA_SBHD = 0, CSA_BSHD = 1, CSA_THD = 2 } csa_layout;
typedef enum { CSA_F32 = 0, CSA_BF16 = 1 } csa_dtype;

/* Which teacher the loss distils ([BUG] "Paper reference" and sec. 3 for the full one; sec. 1, the
 * compressed-only teacher the issue reports as the bug).
 *   CSA_TEACHER_FULL: each head's denominator takes the sink, the sliding window and the selected
 *     compressed keys together (Z_h = e^{a_h} + sum_C e^{c_hj} + sum_W e^{w_hr}).
 *   CSA_TEACHER_COMPRESSED_ONLY: a per-head softmax over the compressed support alone (no sink, no
 *     window), i.e. the teacher the issue shows to be wrong; kept as an A/B negative control.  kv and
 *     sink are still validated but not read. */
typedef enum { CSA_TEACHER_FULL = 0, CSA_TEACHER_COMPRESSED_ONLY = 1 } csa_teacher_mode;

/* Geometry and flags of one step.  A plain struct read on the host; the two cu_seqlens pointers are
 * device pointers.  Megatron's flags map as: index_topk -> topk, dsa_indexer_use_sparse_loss ->
 * sparse_loss, calculate_per_token_loss -> reduction = 1, dsa_indexer_loss_coeff -> loss_coeff
 * ([BUG] sec. 1 excerpt, the FusedDSAIndexerLoss.apply call). */
typedef struct {
    int32_t layout;                       /* csa_layout */
    int32_t dtype;                        /* csa_dtype of the value tensors */
    int32_t batch;                        /* SBHD/BSHD: sequences B.  THD: number of segments */
    int32_t seqlen;                       /* SBHD/BSHD: sequence length S.  THD: physical rows T */
    const int32_t *cu_seqlens_q;          /* THD: device [batch+1], physical offsets (non-decreasing) */
    const int32_t *cu_seqlens_q_unpadded; /* THD: device [batch+1] or NULL; real lengths <= physical */
    int32_t max_seqlen_q;                 /* THD: host-known longest UNPADDED segment (no device sync); the
                                             key width is max_seqlen_q / r (padding rows see no keys) */
    int32_t key_rows;                     /* THD: rows of k_idx / kv_c (T_c).  SBHD/BSHD: 0 or B * (S / r) */
    int32_t compress_ratio;               /* r >= 1 */
    int32_t window;                       /* W >= 0 original-KV positions (query included) */
    int32_t topk;                         /* >= 1; clamped to the key width (see K above) */
    int32_t heads, head_dim;              /* main attention: H, D */
    int32_t idx_heads, idx_dim;           /* indexer: H_I, D_I */
    float softmax_scale;                  /* main-attention scale sigma.  The indexer's own scale must be
                                             folded into w by the caller ([BUG] sec. 1 excerpt,
                                             weights_for_unfused = weights.float() * softmax_scale) */
    int32_t sparse_loss;                  /* 1: support C = selected keys.  0: C = every visible key */
    int32_t reduction;                    /* 0: mean over physical rows.  1: sum (per-token loss) */
    float loss_coeff;                     /* multiplies the loss and every gradient */
    int32_t teacher_mode;                 /* csa_teacher_mode; 0 (full CSA) when zero-initialised */
    int32_t require_tensor_cores;         /* 1: a call that the tcgen05 kernels do not take (fp32 values, or a
                                             shape outside their limits) returns CSA_ERR_UNSUPPORTED instead of
                                             running the CUDA-core kernels.  0 (default): it runs them, and
                                             csa_last_path reports "generic". */
} csa_params;

/* ------------------------------------------------------------------ sizes (host only, no CUDA call) */

/* K: width of ids / selscore rows.  Returns -1 on invalid params. */
int32_t csa_topk_width(const csa_params *p);

/* Width of the dense compressed-key axis: n_c (SBHD/BSHD) or max_seqlen_q / r (THD).  -1 if invalid. */
int32_t csa_key_width(const csa_params *p);

/* Width of teacher rows: K slots aligned to ids (sparse), or the dense key axis indexed by local key
 * (dense loss).  -1 if invalid. */
int32_t csa_teacher_width(const csa_params *p);

/* Number of query rows (B*S or T) and of compressed key rows.  -1 if invalid. */
int64_t csa_rows(const csa_params *p);
int64_t csa_compressed_rows(const csa_params *p);

/* Bytes of device workspace each call needs (the largest of the three calls).  0 on invalid params. */
size_t csa_workspace_size(const csa_params *p);

/* ------------------------------------------------------------------ the step */

/* Steps 1-2: indexer scores over the visible compressed keys, fused with the top-k; the score matrix is
 * never written to memory.
 *   q_idx [rows, H_I, D_I] (layout order), w [rows, H_I] fp32, k_idx [compressed rows, D_I]
 *   -> ids_out [rows, K] int32 (global ids, ascending, -1 pads),
 *      selscore_out [rows, K] fp32 (I of each selected key, -inf in pad slots).
 * Row order of outputs is the layout's row order (SBHD: s*B+b, BSHD: b*S+s, THD: t).
 * Source: [BUG] sec. 1 excerpt (mask, min(topk, n_c)), sec. 3 excerpt (valid slots), [PR] item 1. */
csa_status csa_indexer_fwd(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                           int32_t *ids_out, float *selscore_out,
                           void *workspace, size_t workspace_bytes, void *stream);

/* Step 3: the full-CSA teacher for given ids ([BUG] "Paper reference": Z_h and t_j equations; the
 * follow-up proposal's factored form u_h, l_h, p_hj; sec. 3: window + compressed + sink share one
 * denominator):
 *   c_hj = sigma q[t,h].kv_c[j] (j in C), w_hr = sigma q[t,h].kv[r] (r in the window), a_h = sink[h]
 *   l_h  = log(exp(a_h) + sum_C exp(c_hj) + sum_W exp(w_hr))
 *   t_j  = sum_h exp(c_hj - l_h) / max(sum_{k in C} sum_h exp(c_hk - l_h), 1e-10)
 *   q [rows, H, D], kv [rows, D], kv_c [compressed rows, D], sink [H] fp32, ids [rows, K]
 *   -> teacher_out [rows, teacher_width] fp32 (0 in slots outside C). */
csa_status csa_teacher(const csa_params *p, const void *q, const void *kv, const void *kv_c,
                       const float *sink, const int32_t *ids, float *teacher_out,
                       void *workspace, size_t workspace_bytes, void *stream);

/* Step 3 from a given non-compressed log-sum-exp ([BUG] follow-up proposal: take u_h, the log-sum-exp of the
 * sink and the window logits, from the attention forward (non_compressed_lse) instead of recomputing the
 * window):
 *   u_h  = lse_nc[t,h] = log(exp(a_h) + sum_W exp(w_hr))          (given; natural log; -inf for neither)
 *   l_h  = log(exp(u_h) + sum_C exp(c_hj)),  t_j as in csa_teacher
 *   q [rows, H, D], kv_c [compressed rows, D], lse_nc [rows, H] fp32 (row order of the layout), ids [rows, K]
 *   -> teacher_out [rows, teacher_width] fp32.
 * No window logit is computed; p->window and p->teacher_mode are ignored (lse_nc carries the whole
 * non-compressed part).  Same workspace as csa_teacher; same validation and errors (lse_nc: 16-byte aligned,
 * non-null when rows > 0). */
csa_status csa_teacher_from_lse(const csa_params *p, const void *q, const void *kv_c, const float *lse_nc,
                                const int32_t *ids, float *teacher_out, void *workspace, size_t workspace_bytes,
                                void *stream);

/* Steps 3-5: teacher (recomputed when teacher_or_null is NULL), KL and the indexer gradients.
 *   p_s   = softmax over C of the scores (selscore from csa_indexer_fwd; dense loss with K below the key
 *           width recomputes the visible scores into the workspace)
 *   L_t   = sum_{s in C} t_s (log(t_s + 1e-10) - log(p_s + 1e-10))      ([BUG] sec. 2 excerpt; the review
 *           keeps log(x + 1e-10), not a clamp to tiny)
 *   loss  = loss_coeff * sum_t L_t / rows (mean) or loss_coeff * sum_t L_t (sum)
 *   g_ts  = dloss/dI_ts = f * p_s (A - t_s / (p_s + 1e-10)),  A = sum_k t_k p_k / (p_k + 1e-10)
 *   dw     [rows, H_I] fp32 = sum_s g_ts max(0, x_tjs)
 *   dq_idx [rows, H_I, D_I] = sum_s g_ts w_tj 1[x_tjs > 0] k_idx[s]
 *   dk_idx [compressed rows, D_I] = sum_t sum_j g_ts w_tj 1[x_tjs > 0] q_idx[t,j]   (rows never selected: 0)
 * with x_tjs = q_idx[t,j].k_idx[s].  No gradient flows to q, kv, kv_c or the sink (the follow-up
 * proposal: teacher-side inputs stay detached).  loss_out is one device fp32; row_loss_out (optional, NULL to
 * skip) receives the unscaled per-row KL L_t [rows] fp32 (0 for padding rows and rows without keys).
 * With teacher_or_null NULL, 128 main heads and the sparse loss, the KL step runs inside the teacher kernel, which
 * reduces a row's maximum and normaliser in another order than the separate KL kernel that a given teacher takes:
 * the two calls then agree to fp32 rounding (and the bf16 outputs to a unit in the last place), not bit for bit. */
csa_status csa_indexer_bwd(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                           const void *q, const void *kv, const void *kv_c, const float *sink,
                           const int32_t *ids, const float *selscore, const float *teacher_or_null,
                           float *loss_out, float *row_loss_out, void *dq_idx, float *dw, void *dk_idx,
                           void *workspace, size_t workspace_bytes, void *stream);

/* ------------------------------------------------------------------ backward without a workspace */

/* Size of the library's built-in device scratch used by csa_indexer_bwd_noalloc: 64 MiB. */
#define CSA_NOALLOC_SCRATCH_BYTES (64u << 20)

/* The same computation as csa_indexer_bwd (same arguments and outputs), for callers that cannot allocate
 * device memory and so cannot pass a workspace -- for example code running where the host application owns
 * every device allocation, or a process that must not call cudaMalloc once it is running.  The paper has no
 * counterpart to this call; it exists only for those callers.
 *   - Scratch: a fixed device array of CSA_NOALLOC_SCRATCH_BYTES inside the library.  Every GPU on which the
 *     library's device code is loaded holds it until the process exits.  Nothing is allocated or freed.
 *   - Limit: returns CSA_ERR_WORKSPACE, without enqueueing anything, when csa_workspace_size(p) exceeds
 *     CSA_NOALLOC_SCRATCH_BYTES (the bshd_bf16 workload needs about 49 MiB).
 *   - Set-up: the first call on a device looks up the array's device address (cudaGetSymbolAddress) with that
 *     device current; make that first call before any stream capture.
 *   - Sharing: every call on a device uses the same array, which keeps whatever the last call left there; the
 *     call zeroes what must start at zero (the dK accumulator) itself.  Calls whose work overlaps on the GPU
 *     (different streams, or different host threads) race on the array and must be serialised by the caller. */
/*   - Device resets: the looked-up address belongs to the device's primary context; after cudaDeviceReset (or
 *     anything else that destroys that context) the library would keep using the old address, so do not call
 *     csa_indexer_bwd_noalloc again on a device that was reset in the same process. */
csa_status csa_indexer_bwd_noalloc(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                                   const void *q, const void *kv, const void *kv_c, const float *sink,
                                   const int32_t *ids, const float *selscore, const float *teacher_or_null,
                                   float *loss_out, float *row_loss_out, void *dq_idx, float *dw, void *dk_idx,
                                   void *stream);

/* ------------------------------------------------------------------ diagnostics */

/* Test aid: the fp32 scores exactly as csa_indexer_fwd computes them, for rows
 * [row_begin, row_begin + row_count) -> scores_out [row_count, key width] (-inf where not visible).
 * Writes the score rows it is asked for, so keep row_count small. */
csa_status csa_scores_debug(const csa_params *p, const void *q_idx, const float *w, const void *k_idx,
                            int64_t row_begin, int64_t row_count, float *scores_out,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Synchronises `stream`, then reads and clears the library's device error word (set by a kernel that
 * gave up a bounded wait).  Returns CSA_ERR_TIMEOUT if it was set, CSA_ERR_CUDA on a CUDA error. */
csa_status csa_check_device_status(void *stream);

/* Test aid for the device-side timeout reporting: enqueues one tiny kernel that waits, with the same bounded
 * wait the tensor-core kernels use but a limit of about 1 ms, on a barrier nothing arrives on.  The wait runs
 * out, the kernel records the expiry in the library's device error word and returns; no copy or MMA is in
 * flight.  The next csa_check_device_status on the stream returns CSA_ERR_TIMEOUT (and clears the word); the
 * CUDA context stays usable.  The pages have no counterpart to this call. */
csa_status csa_selftest_bounded_wait(void *stream);

/* Where the last timeout that csa_check_device_status reported on this host thread happened, as
 * 100 x kernel + wait site: kernel 1 the score / top-k kernel, 2 the backward, 3 the 64-head teacher, 4 the
 * 128-head teacher, 5 the gathered row-owner backward, 9 the bounded-wait self-test; site 99 is a drain of the
 * kernel's own copies that ran out after an abort.  0 before the first timeout; not cleared by later calls. */
int32_t csa_last_timeout_site(void);

/* Name of the last kernel path csa_indexer_fwd, csa_teacher, csa_teacher_from_lse or csa_indexer_bwd chose
 * on this host thread ("tcgen05", "generic", ...; for csa_indexer_bwd, its backward's).  Static string. */
const char *csa_last_path(void);

/* Message of the last CUDA runtime error that ended a call of this library with CSA_ERR_CUDA on this host
 * thread ("no error" before the first).  Static string; not cleared by later successful calls. */
const char *csa_last_cuda_error(void);

/* Number of CUDA kernels this library has launched in the process so far (all devices, all threads). */
uint64_t csa_kernel_launches(void);

const char *csa_status_string(csa_status s);

#ifdef __cplusplus
}
#endif

#endif /* CSA_INDEXER_H */
