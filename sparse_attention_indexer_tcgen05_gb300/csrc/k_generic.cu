// k_generic.cu -- CUDA-core kernels of the CSA indexer step for any shape and both value dtypes.
//
// These are the correct-first path: one CTA per query row, fp32 arithmetic on CUDA cores, shared
// memory for the row's operands.  They serve every shape the tensor-core kernels do not take (fp32
// mode, small or odd head counts), unless the caller sets csa_params.require_tensor_cores.  Both paths
// are tested against the float64 oracle.
//
// Sources, by page title and section:
//   [BUG] "[Bug] DSV4 unfused CSA indexer loss uses a compressed-only teacher instead of the full CSA
//         attention distribution" (Megatron-LM issue #5776) and its comments.
//   [PR]  "Megatron-LM PR #8539".
#include "csa_internal.cuh"

#include <math.h>

namespace csa {

static constexpr int kThreads = 256;
static constexpr int kWarps = kThreads / 32;
static constexpr float kEps = 1e-10f;   // [BUG] sec. 2 excerpt: clamp(min=1e-10), log(x + 1e-10)

// ------------------------------------------------------------------ THD compressed offsets

// cu_c = [0, cumsum(real_len // r)]: compressed cu_seqlens rebuilt from the unpadded lengths
// ([BUG] sec. 1 THD excerpt).  Segments are few; one thread walks them.
__global__ void build_cu_c_kernel(const int *cu_real, int nseg, int ratio, int *cu_c)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    cu_c[0] = 0;
    for (int b = 0; b < nseg; b++) {
        int len = cu_real[b + 1] - cu_real[b];
        acc += len > 0 ? len / ratio : 0;
        cu_c[b + 1] = acc;
    }
}

cudaError_t launch_build_cu_c(const Geo &g, int *cu_c, cudaStream_t st)
{
    build_cu_c_kernel<<<1, 32, 0, st>>>(g.cu_real, g.B, g.ratio, cu_c);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ block helpers

// Exclusive prefix count of `flag` over the block in thread order, and the block total.
__device__ __forceinline__ int block_excl_count(bool flag, int *warp_tot, int &total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    unsigned bal = __ballot_sync(0xffffffffu, flag);
    int in_warp = __popc(bal & ((1u << lane) - 1u));
    if (lane == 0) warp_tot[wid] = __popc(bal);
    __syncthreads();
    int before = 0, tot = 0;
    for (int i = 0; i < (int)(blockDim.x >> 5); i++) {
        int c = warp_tot[i];
        before += i < wid ? c : 0;
        tot += c;
    }
    __syncthreads();
    total = tot;
    return before + in_warp;
}

__device__ __forceinline__ float block_reduce(float x, float *red, bool is_max)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    x = is_max ? warp_max(x) : warp_sum(x);
    if (lane == 0) red[wid] = x;
    __syncthreads();
    float r = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); i++) r = is_max ? fmaxf(r, red[i]) : r + red[i];
    __syncthreads();
    return r;
}

// ------------------------------------------------------------------ steps 1-2: score + top-k

size_t score_topk_generic_smem(const Geo &g)
{
    return sizeof(float) * ((size_t)g.HI * (g.DI + 1) + g.HI + (size_t)kWarps * g.DI + (size_t)(g.NC > 0 ? g.NC : 1));
}

// One CTA per query row.  Scores of the row's visible keys are kept in shared memory only; the
// k-th largest is found by a 4-pass radix select on order-preserving keys, and the selection is
// written in ascending key order by a stable block compaction (ties: lower index first).
template <typename T>
__global__ void __launch_bounds__(kThreads)
score_topk_generic_kernel(Geo g, const T *__restrict__ q_idx, const float *__restrict__ w,
                          const T *__restrict__ k_idx, int32_t *__restrict__ ids, float *__restrict__ selscore,
                          float *__restrict__ dump, long long dump_row0, long long dump_rows)
{
    extern __shared__ float smem[];
    const int HI = g.HI, DI = g.DI, DP = DI + 1;
    float *qs = smem;                       // [HI][DI+1]
    float *wsm = qs + (size_t)HI * DP;      // [HI]
    float *kb_all = wsm + HI;               // [warps][DI]
    float *sc = kb_all + (size_t)kWarps * DI;  // [NC]
    __shared__ uint32_t hist[256];
    __shared__ int warp_tot[kWarps];
    __shared__ uint32_t s_prefix, s_rem;

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float *kb = kb_all + (size_t)wid * DI;

    for (long long r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const bool dumping = dump != nullptr && r >= dump_row0 && r < dump_row0 + dump_rows;
        if (ids == nullptr && !dumping) continue;
        const Row R = decode_row(g, r);
        const int v = R.v;
        if (v > 0) {
            for (int e = tid; e < HI * DI; e += kThreads)
                qs[(e / DI) * DP + e % DI] = ldf(q_idx, r * HI * DI + e);
            for (int e = tid; e < HI; e += kThreads) wsm[e] = __ldg(w + r * HI + e);
            __syncthreads();
            // I[t,j] = sum_h w[t,h] * max(0, q_idx[t,h] . k_idx[j]) over the visible keys j < v
            for (int j = wid; j < v; j += kWarps) {
                const long long kr = key_row(g, key_gid(g, R, j));
                for (int d = lane; d < DI; d += 32) kb[d] = ldf(k_idx, kr * DI + d);
                __syncwarp();
                float acc = 0.f;
                for (int h = lane; h < HI; h += 32) {
                    const float *qh = qs + (size_t)h * DP;
                    float x = 0.f;
                    for (int d = 0; d < DI; d++) x = fmaf(qh[d], kb[d], x);
                    acc = fmaf(wsm[h], fmaxf(x, 0.f), acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) sc[j] = acc;
                __syncwarp();
            }
        }
        __syncthreads();
        if (dumping) {
            float *out = dump + (r - dump_row0) * (long long)g.NC;
            for (int j = tid; j < g.NC; j += kThreads) out[j] = j < v ? sc[j] : -INFINITY;
        }
        if (ids != nullptr) {
            const int K = g.K;
            const int k = v < K ? v : K;
            int32_t *orow = ids + r * K;
            float *srow = selscore + r * K;
            if (k > 0) {
                // radix select: exact key of the k-th largest score, and how many equal keys to take
                if (tid == 0) { s_prefix = 0u; s_rem = (uint32_t)k; }
                uint32_t mask = 0u;
                for (int shift = 24; shift >= 0; shift -= 8) {
                    hist[tid] = 0u;  // kThreads == 256 bins
                    __syncthreads();
                    const uint32_t prefix = s_prefix;
                    for (int j = tid; j < v; j += kThreads) {
                        uint32_t u = score_key(sc[j]);
                        if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1u);
                    }
                    __syncthreads();
                    if (tid == 0) {
                        uint32_t rem = s_rem;
                        int dgt = 255;
                        for (; dgt > 0; --dgt) {
                            if (hist[dgt] >= rem) break;
                            rem -= hist[dgt];
                        }
                        s_prefix = prefix | ((uint32_t)dgt << shift);
                        s_rem = rem;
                    }
                    __syncthreads();
                    mask |= 255u << shift;
                }
                const uint32_t thr = s_prefix;
                const int need_eq = (int)s_rem;
                int base_eq = 0, base_sel = 0;
                for (int j0 = 0; j0 < v; j0 += kThreads) {
                    const int j = j0 + tid;
                    const uint32_t u = j < v ? score_key(sc[j]) : 0u;
                    const bool gt = j < v && u > thr;
                    const bool eq = j < v && u == thr;
                    int tot_eq, tot_sel;
                    const int eq_rank = base_eq + block_excl_count(eq, warp_tot, tot_eq);
                    const bool sel = gt || (eq && eq_rank < need_eq);
                    const int pos = base_sel + block_excl_count(sel, warp_tot, tot_sel);
                    if (sel) {
                        orow[pos] = (int32_t)key_gid(g, R, j);
                        srow[pos] = sc[j];
                    }
                    base_eq += tot_eq;
                    base_sel += tot_sel;
                }
            }
            for (int s = k + tid; s < K; s += kThreads) {
                orow[s] = -1;
                srow[s] = -INFINITY;
            }
        }
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_score_topk_generic(const Geo &g, const T *q_idx, const float *w, const T *k_idx,
                                      int32_t *ids, float *selscore, float *dump, long long dump_row0,
                                      long long dump_rows, cudaStream_t st)
{
    if (g.rows == 0) return cudaSuccess;
    size_t smem = score_topk_generic_smem(g);
    cudaError_t e = cudaFuncSetAttribute(score_topk_generic_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int grid = g.rows < 65535 * 8 ? g.rows : 65535 * 8;
    score_topk_generic_kernel<T><<<grid, kThreads, smem, st>>>(g, q_idx, w, k_idx, ids, selscore, dump,
                                                               dump_row0, dump_rows);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ step 3: teacher

static __host__ __device__ inline int q_stride(int D, bool bf16) { return bf16 ? D + 2 : D + 1; }

size_t teacher_generic_smem(const Geo &g, bool bf16)
{
    size_t q_bytes = (size_t)g.H * q_stride(g.D, bf16) * (bf16 ? 2 : 4);
    q_bytes = (q_bytes + 15) & ~(size_t)15;
    size_t cap = (size_t)(g.TW > 0 ? g.TW : 1);
    return q_bytes + sizeof(float) * ((size_t)kWarps * g.D + 2 * (size_t)kWarps * g.H + g.H + cap);
}

// Support slot -> global key id of the row, or -1 when the slot is not in C.  Sparse: the slot's id,
// accepted only when it is a visible key of this row (ids outside that range are treated as invalid,
// so a bad id can never address memory outside the row's keys).  Dense: slot j is local key j.
__device__ __forceinline__ long long support_gid(const Geo &g, const Row &R, const int32_t *row_ids, int slot)
{
    if (g.sparse) {
        if (slot >= g.K) return -1;
        long long id = row_ids[slot];
        long long lo = key_gid(g, R, 0);
        return (id >= lo && id < lo + R.v) ? id : -1;
    }
    return slot < R.v ? key_gid(g, R, slot) : -1;
}

// One CTA per query row.  Pass 1 computes every logit of the row's support C and its window W with an
// online per-head max/sum, then folds in the sink: l_h = log(exp(a_h) + sum_C exp(c) + sum_W exp(w)).
// Pass 2 recomputes the compressed logits and forms T_j = sum_h exp(c_hj - l_h); the row is then
// L1-normalised ([BUG] "Paper reference" equations; the follow-up proposal's u_h / l_h form).
template <typename T>
__global__ void __launch_bounds__(kThreads)
teacher_generic_kernel(Geo g, const T *__restrict__ q, const T *__restrict__ kv, const T *__restrict__ kv_c,
                       const float *__restrict__ sink, const int32_t *__restrict__ ids, float *__restrict__ teacher)
{
    extern __shared__ __align__(16) unsigned char tsm[];
    const bool bf16 = sizeof(T) == 2;
    const int H = g.H, D = g.D, QS = q_stride(D, bf16);
    size_t q_bytes = (size_t)H * QS * sizeof(T);
    q_bytes = (q_bytes + 15) & ~(size_t)15;
    T *qs = reinterpret_cast<T *>(tsm);
    float *kb_all = reinterpret_cast<float *>(tsm + q_bytes);  // [warps][D]
    float *st_m = kb_all + (size_t)kWarps * D;                 // [warps][H]
    float *st_s = st_m + (size_t)kWarps * H;                   // [warps][H]
    float *ell = st_s + (size_t)kWarps * H;                    // [H]
    float *Tacc = ell + H;                                     // [TW]
    __shared__ float red[kWarps];

    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float *kb = kb_all + (size_t)wid * D;
    const int TW = g.TW;

    for (long long r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const Row R = decode_row(g, r);
        float *trow = teacher + r * TW;
        if (R.v == 0) {
            for (int s = tid; s < TW; s += kThreads) trow[s] = 0.f;
            continue;
        }
        const int32_t *row_ids = ids + r * g.K;
        const int nslots = g.sparse ? g.K : R.v;
        int p0 = R.s - g.window + 1;
        if (p0 < 0) p0 = 0;
        const int nW = g.window > 0 ? R.s - p0 + 1 : 0;
        for (int e = tid; e < H * D; e += kThreads) qs[(e / D) * QS + e % D] = q[r * H * D + e];
        for (int e = tid; e < kWarps * H; e += kThreads) { st_m[e] = -INFINITY; st_s[e] = 0.f; }
        __syncthreads();

        // pass 1: online per-head max / sum over C and W
        for (int it = wid; it < nslots + nW; it += kWarps) {
            const T *src;
            if (it < nslots) {
                long long gid = support_gid(g, R, row_ids, it);
                if (gid < 0) continue;
                src = kv_c + key_row(g, gid) * D;
            } else {
                src = kv + q_row(g, R, p0 + (it - nslots)) * D;
            }
            for (int d = lane; d < D; d += 32) kb[d] = ldf(src, d);
            __syncwarp();
            for (int h = lane; h < H; h += 32) {
                const T *qh = qs + (size_t)h * QS;
                float x = 0.f;
                for (int d = 0; d < D; d++) x = fmaf(lds(qh, d), kb[d], x);
                x *= g.scale;
                float m = st_m[wid * H + h], s = st_s[wid * H + h];
                if (x > m) { s = s * __expf(m - x) + 1.f; m = x; }
                else s += __expf(x - m);
                st_m[wid * H + h] = m;
                st_s[wid * H + h] = s;
            }
            __syncwarp();
        }
        __syncthreads();
        for (int h = tid; h < H; h += kThreads) {
            float m = -INFINITY;
            for (int k = 0; k < kWarps; k++) m = fmaxf(m, st_m[k * H + h]);
            const float a = g.lse_nc != nullptr ? g.lse_nc[r * H + h] : (g.no_sink ? -INFINITY : sink[h]);
            const float M = fmaxf(m, a);
            float s = 0.f;
            if (M != -INFINITY) {
                for (int k = 0; k < kWarps; k++)
                    if (st_m[k * H + h] != -INFINITY) s += st_s[k * H + h] * __expf(st_m[k * H + h] - M);
                if (a != -INFINITY) s += __expf(a - M);
            }
            ell[h] = M + logf(s);
        }
        __syncthreads();

        // pass 2: T_j = sum_h exp(c_hj - l_h) for the compressed support
        for (int it = wid; it < TW; it += kWarps) {
            long long gid = it < nslots ? support_gid(g, R, row_ids, it) : -1;
            if (gid < 0) {
                if (lane == 0) Tacc[it] = 0.f;
                continue;
            }
            const T *src = kv_c + key_row(g, gid) * D;
            for (int d = lane; d < D; d += 32) kb[d] = ldf(src, d);
            __syncwarp();
            float acc = 0.f;
            for (int h = lane; h < H; h += 32) {
                const T *qh = qs + (size_t)h * QS;
                float x = 0.f;
                for (int d = 0; d < D; d++) x = fmaf(lds(qh, d), kb[d], x);
                acc += __expf(x * g.scale - ell[h]);
            }
            acc = warp_sum(acc);
            if (lane == 0) Tacc[it] = acc;
            __syncwarp();
        }
        __syncthreads();
        float part = 0.f;
        for (int s = tid; s < TW; s += kThreads) part += Tacc[s];
        float S = block_reduce(part, red, false);
        S = fmaxf(S, kEps);
        for (int s = tid; s < TW; s += kThreads) trow[s] = Tacc[s] / S;
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_teacher_generic(const Geo &g, const T *q, const T *kv, const T *kv_c, const float *sink,
                                   const int32_t *ids, float *teacher, cudaStream_t st)
{
    if (g.rows == 0 || g.TW == 0) return cudaSuccess;
    size_t smem = teacher_generic_smem(g, sizeof(T) == 2);
    cudaError_t e = cudaFuncSetAttribute(teacher_generic_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int grid = g.rows < 65535 * 8 ? g.rows : 65535 * 8;
    teacher_generic_kernel<T><<<grid, kThreads, smem, st>>>(g, q, kv, kv_c, sink, ids, teacher);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ step 4: KL and dL/dI

// One CTA per query row.  p = softmax over C of the scores, L_t = sum t (log(t+eps) - log(p+eps)) and
// g_s = f * p_s (A - t_s/(p_s+eps)) with A = sum_k t_k p_k/(p_k+eps): the exact derivative of the
// eps-guarded KL of [BUG] sec. 2 excerpt.  gbuf uses the teacher's slot layout.
// With gd != nullptr it also writes g by key: gd[prow][j] for the row's visible keys j < v (0 off the support),
// row stride ncp; what lies beyond v is left as it is.  Rows are ordered by position within each sequence
// (prow = b S + s for SBHD, the row itself otherwise), so the two rows of a position pair are adjacent.

__global__ void __launch_bounds__(kThreads)
kl_kernel(Geo g, const int32_t *__restrict__ ids, const float *__restrict__ selscore,
          const float *__restrict__ dense_scores, const float *__restrict__ teacher, float *__restrict__ gbuf,
          float *__restrict__ row_loss, float *__restrict__ gd, int ncp)
{
    __shared__ float red[kWarps];
    const int tid = threadIdx.x;
    const int TW = g.TW;
    for (long long r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const Row R = decode_row(g, r);
        const int32_t *row_ids = ids + r * g.K;
        const float *trow = teacher + r * TW;
        float *grow = gbuf != nullptr ? gbuf + r * TW : nullptr;
        float *drow = gd != nullptr ? gd + gd_row_of(g, R.b, R.s, r) * ncp : nullptr;
        if (drow != nullptr) {
            for (int j = tid; j < R.v; j += kThreads) drow[j] = 0.f;
            __syncthreads();
        }
        // score of support slot s, or -inf when s is not in C
        auto score_of = [&](int s) -> float {
            if (s >= TW) return -INFINITY;
            if (g.sparse) return support_gid(g, R, row_ids, s) >= 0 ? selscore[r * g.K + s] : -INFINITY;
            if (s >= R.v) return -INFINITY;
            return dense_scores ? dense_scores[r * g.NC + s] : selscore[r * g.K + s];
        };
        float m = -INFINITY;
        for (int s = tid; s < TW; s += kThreads) m = fmaxf(m, score_of(s));
        m = block_reduce(m, red, true);
        if (m == -INFINITY) {  // empty support: no loss, no gradient
            if (grow != nullptr)
                for (int s = tid; s < TW; s += kThreads) grow[s] = 0.f;
            if (tid == 0) row_loss[r] = 0.f;
            continue;
        }
        const long long lo = key_gid(g, R, 0);
        float z = 0.f;
        for (int s = tid; s < TW; s += kThreads) {
            float x = score_of(s);
            z += x == -INFINITY ? 0.f : __expf(x - m);
        }
        z = block_reduce(z, red, false);
        const float inv_z = 1.f / z;
        float A = 0.f, L = 0.f;
        for (int s = tid; s < TW; s += kThreads) {
            float x = score_of(s);
            if (x == -INFINITY) continue;
            float p = __expf(x - m) * inv_z;
            float t = trow[s];
            A += t * p / (p + kEps);
            L += t * (logf(t + kEps) - logf(p + kEps));
        }
        A = block_reduce(A, red, false);
        L = block_reduce(L, red, false);
        for (int s = tid; s < TW; s += kThreads) {
            float x = score_of(s);
            float gv = 0.f;
            if (x != -INFINITY) {
                float p = __expf(x - m) * inv_z;
                gv = g.factor * p * (A - trow[s] / (p + kEps));
                if (drow != nullptr) drow[g.sparse ? (int)(row_ids[s] - lo) : s] = gv;
            }
            if (grow != nullptr) grow[s] = gv;
        }
        if (tid == 0) row_loss[r] = L;
    }
}

// The same step for the sparse support with K <= 512 slots (teacher width K): one warp per row, the row's
// ids, scores and teacher values held in registers (slot s = lane + 32 i, coalesced), warp reductions.
// The same step for the sparse support with K <= 512 slots (teacher width K): one warp per row, the row's
// scores, teacher values and key offsets held in registers (slot s = lane + 32 i, coalesced); the row's
// arithmetic is kl_row_warp.  gbuf may be null (the tensor-core backward reads gd only).
__global__ void __launch_bounds__(kThreads)
kl_warp_kernel(Geo g, const int32_t *__restrict__ ids, const float *__restrict__ selscore,
               const float *__restrict__ teacher, float *__restrict__ gbuf, float *__restrict__ row_loss,
               float *__restrict__ gd, int ncp)
{
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * kWarps;
    const int K = g.K;
    for (long long r = (long long)blockIdx.x * kWarps + (threadIdx.x >> 5); r < g.rows; r += nwarps) {
        const Row R = decode_row(g, r);
        const long long lo = key_gid(g, R, 0);
        const int32_t *row_ids = ids + r * K;
        const float *srow = selscore + r * K;
        const float *trow = teacher + r * K;
        int jj[kKlPer];
        float x[kKlPer], t[kKlPer];
#pragma unroll
        for (int i = 0; i < kKlPer; i++) {  // every load issued before any is used
            const int s = lane + 32 * i;
            const bool in = s < K;
            jj[i] = in ? __ldg(row_ids + s) : -1;
            x[i] = in ? __ldg(srow + s) : 0.f;
            t[i] = in ? __ldg(trow + s) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kKlPer; i++) {
            const long long j = jj[i] >= 0 ? (long long)jj[i] - lo : -1;
            jj[i] = (j >= 0 && j < R.v) ? (int)j : -1;
        }
        float *grow = gbuf != nullptr ? gbuf + r * K : nullptr;
        float *drow = gd != nullptr ? gd + gd_row_of(g, R.b, R.s, r) * ncp : nullptr;
        const float L = kl_row_warp(g, lane, K, R.v, jj, x, t, grow, drow);
        if (lane == 0) row_loss[r] = L;
    }
}

// The same step for the sparse support with 512 < K <= 4096 slots: one CTA of 256 threads per row, the row's
// ids, scores and teacher values held in registers (slot s = tid + 256 i, coalesced), so the row is read once;
// block reductions for the max, the normaliser and the pair (A, L); the arithmetic of kl_row_warp.
constexpr int kKlBlkPer = 16;  // slots per thread: K <= 4096
__global__ void __launch_bounds__(kThreads)
kl_block_kernel(Geo g, const int32_t *__restrict__ ids, const float *__restrict__ selscore,
                const float *__restrict__ teacher, float *__restrict__ gbuf, float *__restrict__ row_loss,
                float *__restrict__ gd, int ncp)
{
    __shared__ float red[2][kWarps];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int K = g.K;
    for (long long r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const Row R = decode_row(g, r);
        const long long lo = key_gid(g, R, 0);
        int jj[kKlBlkPer];
        float x[kKlBlkPer], t[kKlBlkPer];
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++) {  // every load issued before any is used
            const int s = tid + kThreads * i;
            const bool in = s < K;
            jj[i] = in ? __ldg(ids + r * K + s) : -1;
            x[i] = in ? __ldg(selscore + r * K + s) : 0.f;
            t[i] = in ? __ldg(teacher + r * K + s) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++) {
            const long long j = jj[i] >= 0 ? (long long)jj[i] - lo : -1;
            jj[i] = (j >= 0 && j < R.v) ? (int)j : -1;
        }
        float *grow = gbuf != nullptr ? gbuf + r * K : nullptr;
        float *drow = gd != nullptr ? gd + gd_row_of(g, R.b, R.s, r) * ncp : nullptr;
        if (drow != nullptr)  // zero the visible range
            for (int j = tid; j < R.v; j += kThreads) drow[j] = 0.f;
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++)
            if (jj[i] >= 0) m = fmaxf(m, x[i]);
        m = block_reduce(m, red[0], true);  // its barriers also order the zeroing above before the writes below
        if (m == -INFINITY) {  // empty support: no loss, no gradient
            if (grow != nullptr)
#pragma unroll
                for (int i = 0; i < kKlBlkPer; i++)
                    if (tid + kThreads * i < K) grow[tid + kThreads * i] = 0.f;
            if (tid == 0) row_loss[r] = 0.f;
            continue;
        }
        float z = 0.f;
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++) {
            x[i] = jj[i] >= 0 ? __expf(x[i] - m) : 0.f;
            z += x[i];
        }
        z = block_reduce(z, red[0], false);
        const float inv_z = 1.f / z;
        float A = 0.f, L = 0.f;
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++) {
            if (jj[i] < 0) continue;
            const float p = x[i] * inv_z;
            A += t[i] * p / (p + kKlEps);
            L += t[i] * (logf(t[i] + kKlEps) - logf(p + kKlEps));
        }
        // A and L in one block reduction
        A = warp_sum(A);
        L = warp_sum(L);
        if (lane == 0) {
            red[0][wid] = A;
            red[1][wid] = L;
        }
        __syncthreads();
        A = 0.f;
        L = 0.f;
        for (int w = 0; w < kWarps; w++) {
            A += red[0][w];
            L += red[1][w];
        }
        __syncthreads();
#pragma unroll
        for (int i = 0; i < kKlBlkPer; i++) {
            const int s = tid + kThreads * i;
            if (s >= K) continue;
            const float p = x[i] * inv_z;
            const float gv = jj[i] >= 0 ? g.factor * p * (A - t[i] / (p + kKlEps)) : 0.f;
            if (grow != nullptr) grow[s] = gv;
            if (drow != nullptr && jj[i] >= 0) drow[jj[i]] = gv;
        }
        if (tid == 0) row_loss[r] = L;
    }
}

cudaError_t launch_kl(const Geo &g, const int32_t *ids, const float *selscore, const float *dense_scores,
                      const float *teacher, float *gbuf, float *row_loss, float *gd, int ncp, cudaStream_t st)
{
    if (g.rows == 0) return cudaSuccess;
    if (g.sparse && dense_scores == nullptr && g.TW == g.K && g.K <= 32 * kKlPer) {
        const long long blocks = (g.rows + kWarps - 1) / kWarps;
        const int grid = blocks < 152 * 16 ? (int)blocks : 152 * 16;
        kl_warp_kernel<<<grid, kThreads, 0, st>>>(g, ids, selscore, teacher, gbuf, row_loss, gd, ncp);
        note_launches(1);
        return cudaGetLastError();
    }
    if (g.sparse && dense_scores == nullptr && g.TW == g.K && g.K <= kThreads * kKlBlkPer) {
        // as many CTAs as can be resident (each loops over rows): no late wave of CTAs at the end
        int dev = 0, sms = 0, per_sm = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kl_block_kernel, kThreads, 0);
        if (e != cudaSuccess) return e;
        const long long resident = (long long)sms * (per_sm > 0 ? per_sm : 1);
        const int grid = g.rows < resident ? g.rows : (int)resident;
        kl_block_kernel<<<grid, kThreads, 0, st>>>(g, ids, selscore, teacher, gbuf, row_loss, gd, ncp);
        note_launches(1);
        return cudaGetLastError();
    }
    int grid = g.rows < 65535 * 8 ? g.rows : 65535 * 8;
    kl_kernel<<<grid, kThreads, 0, st>>>(g, ids, selscore, dense_scores, teacher, gbuf, row_loss, gd, ncp);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ step 5: gradients

size_t grad_generic_smem(const Geo &g)
{
    return sizeof(float) * ((size_t)g.HI * (g.DI + 1) + g.HI + (size_t)g.HI * g.DI + g.HI + (size_t)kWarps * g.DI +
                            (size_t)kWarps * g.HI);
}

// One CTA per query row; one warp per support key at a time.  For each key s with g_s != 0:
//   x_j = q_idx[t,j].k_idx[s];  c_j = g_s w_j 1[x_j > 0]
//   dW[t,j] += g_s max(x_j, 0);  dQ[t,j] += c_j k_idx[s];  dK[s] += sum_j c_j q_idx[t,j]  (fp32 atomics)
template <typename T>
__global__ void __launch_bounds__(kThreads)
grad_generic_kernel(Geo g, const T *__restrict__ q_idx, const float *__restrict__ w, const T *__restrict__ k_idx,
                    const int32_t *__restrict__ ids, const float *__restrict__ gbuf, T *__restrict__ dq_idx,
                    float *__restrict__ dw, float *__restrict__ dk_acc)
{
    extern __shared__ float gsm[];
    const int HI = g.HI, DI = g.DI, DP = DI + 1;
    float *qs = gsm;                        // [HI][DI+1]
    float *wsm = qs + (size_t)HI * DP;      // [HI]
    float *dqs = wsm + HI;                  // [HI][DI]
    float *dws = dqs + (size_t)HI * DI;     // [HI]
    float *kb_all = dws + HI;               // [warps][DI]
    float *cf_all = kb_all + (size_t)kWarps * DI;  // [warps][HI]
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    float *kb = kb_all + (size_t)wid * DI;
    float *cf = cf_all + (size_t)wid * HI;
    const int TW = g.TW;

    for (long long r = blockIdx.x; r < g.rows; r += gridDim.x) {
        const Row R = decode_row(g, r);
        for (int e = tid; e < HI * DI; e += kThreads) {
            qs[(e / DI) * DP + e % DI] = ldf(q_idx, r * HI * DI + e);
            dqs[e] = 0.f;
        }
        for (int e = tid; e < HI; e += kThreads) { wsm[e] = __ldg(w + r * HI + e); dws[e] = 0.f; }
        __syncthreads();
        if (R.v > 0) {
            const int32_t *row_ids = ids + r * g.K;
            const float *grow = gbuf + r * TW;
            for (int s = wid; s < TW; s += kWarps) {
                const float gs = grow[s];
                if (gs == 0.f) continue;
                const long long gid = support_gid(g, R, row_ids, s);
                if (gid < 0) continue;
                const long long kr = key_row(g, gid);
                for (int d = lane; d < DI; d += 32) kb[d] = ldf(k_idx, kr * DI + d);
                __syncwarp();
                for (int h = lane; h < HI; h += 32) {
                    const float *qh = qs + (size_t)h * DP;
                    float x = 0.f;
                    for (int d = 0; d < DI; d++) x = fmaf(qh[d], kb[d], x);
                    const bool on = x > 0.f;
                    cf[h] = on ? gs * wsm[h] : 0.f;
                    if (on) atomicAdd(&dws[h], gs * x);
                }
                __syncwarp();
                if ((DI & 3) == 0) {
                    // four consecutive d per lane: one vector reduction per lane into dK
                    for (int d0 = lane * 4; d0 < DI; d0 += 128) {
                        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
                        for (int h = 0; h < HI; h++) {
                            const float c = cf[h];
                            if (c == 0.f) continue;
                            const float *qh = qs + (size_t)h * DP + d0;
                            acc.x = fmaf(c, qh[0], acc.x);
                            acc.y = fmaf(c, qh[1], acc.y);
                            acc.z = fmaf(c, qh[2], acc.z);
                            acc.w = fmaf(c, qh[3], acc.w);
                            float *dqh = dqs + (size_t)h * DI + d0;
                            atomicAdd(dqh + 0, c * kb[d0 + 0]);
                            atomicAdd(dqh + 1, c * kb[d0 + 1]);
                            atomicAdd(dqh + 2, c * kb[d0 + 2]);
                            atomicAdd(dqh + 3, c * kb[d0 + 3]);
                        }
                        atomicAdd(reinterpret_cast<float4 *>(dk_acc + kr * DI + d0), acc);
                    }
                } else {
                    for (int d = lane; d < DI; d += 32) {
                        float acc = 0.f;
                        const float kd = kb[d];
                        for (int h = 0; h < HI; h++) {
                            const float c = cf[h];
                            if (c != 0.f) {
                                acc = fmaf(c, qs[(size_t)h * DP + d], acc);
                                atomicAdd(&dqs[(size_t)h * DI + d], c * kd);
                            }
                        }
                        atomicAdd(&dk_acc[kr * DI + d], acc);
                    }
                }
                __syncwarp();
            }
        }
        __syncthreads();
        for (int e = tid; e < HI * DI; e += kThreads) dq_idx[r * HI * DI + e] = from_f<T>(dqs[e]);
        for (int e = tid; e < HI; e += kThreads) dw[r * HI + e] = dws[e];
        __syncthreads();
    }
}

template <typename T>
cudaError_t launch_grad_generic(const Geo &g, const T *q_idx, const float *w, const T *k_idx, const int32_t *ids,
                                const float *gbuf, T *dq_idx, float *dw, float *dk_acc, cudaStream_t st)
{
    if (g.rows == 0) return cudaSuccess;
    size_t smem = grad_generic_smem(g);
    cudaError_t e = cudaFuncSetAttribute(grad_generic_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    int grid = g.rows < 65535 * 8 ? g.rows : 65535 * 8;
    grad_generic_kernel<T><<<grid, kThreads, smem, st>>>(g, q_idx, w, k_idx, ids, gbuf, dq_idx, dw, dk_acc);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ finalize

template <typename T>
__global__ void dk_convert_kernel(const float *__restrict__ acc, T *__restrict__ out, long long n)
{
    for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x)
        out[i] = from_f<T>(acc[i]);
}

// loss = f * sum_t L_t, summed in a fixed order (deterministic)
__global__ void __launch_bounds__(1024) loss_reduce_kernel(const float *__restrict__ row_loss, long long rows,
                                                           float factor, float *__restrict__ loss)
{
    __shared__ float red[32];
    float acc = 0.f;
    for (long long i = threadIdx.x; i < rows; i += blockDim.x) acc += row_loss[i];
    acc = warp_sum(acc);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x < 32) {
        float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
        v = warp_sum(v);
        if (threadIdx.x == 0) loss[0] = factor * v;
    }
}

template <typename T>
cudaError_t launch_finalize(const Geo &g, const float *dk_acc, T *dk_idx, const float *row_loss, float *loss,
                            cudaStream_t st)
{
    long long n = g.key_rows * g.DI;
    if (n > 0) {
        long long blocks = (n + 255) / 256;
        int grid = blocks < 152 * 16 ? (int)blocks : 152 * 16;
        dk_convert_kernel<T><<<grid, 256, 0, st>>>(dk_acc, dk_idx, n);
        note_launches(1);
    }
    loss_reduce_kernel<<<1, 1024, 0, st>>>(row_loss, g.rows, g.factor, loss);
    note_launches(1);
    return cudaGetLastError();
}

// ------------------------------------------------------------------ instantiations

#define CSA_INST(T)                                                                                           \
    template cudaError_t launch_score_topk_generic<T>(const Geo &, const T *, const float *, const T *,      \
                                                      int32_t *, float *, float *, long long, long long,      \
                                                      cudaStream_t);                                          \
    template cudaError_t launch_teacher_generic<T>(const Geo &, const T *, const T *, const T *,             \
                                                   const float *, const int32_t *, float *, cudaStream_t);    \
    template cudaError_t launch_grad_generic<T>(const Geo &, const T *, const float *, const T *,            \
                                                const int32_t *, const float *, T *, float *, float *,        \
                                                cudaStream_t);                                                \
    template cudaError_t launch_finalize<T>(const Geo &, const float *, T *, const float *, float *, cudaStream_t);
CSA_INST(float)
CSA_INST(__nv_bfloat16)

}  // namespace csa
