// csa_internal.cuh -- device-side geometry and helpers shared by the CSA indexer kernels.
//
// Row geometry follows the layouts of the C ABI (include/csa_indexer.h): a query row t sits in
// segment b at 0-based position s (1-based i = s + 1) and sees the compressed keys j < i / r
// ("[Bug] DSV4 unfused CSA indexer loss ..." (Megatron-LM issue #5776), sec. 1 excerpt: the
// compressed causal mask where(arange(n_c) >= positions // ratio, -inf, 0), anchored per segment).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/csa_indexer.h"

namespace csa {

// Everything a kernel needs to place a row, a key or a window position.
struct Geo {
    int layout;        // CSA_SBHD / CSA_BSHD / CSA_THD
    int B;             // sequences (SBHD/BSHD) or segments (THD)
    int S;             // sequence length (SBHD/BSHD) or physical rows (THD)
    int rows;          // query rows
    int nc;            // compressed keys per sequence (SBHD/BSHD); unused in THD
    int ratio, window;
    int K;             // top-k width
    int NC;            // dense key width
    int TW;            // teacher width
    int H, D, HI, DI;
    long long key_rows;
    float scale;       // sigma
    int sparse;
    int no_sink;       // compressed-only teacher: the sink term is dropped (and the window is 0)
    const float *lse_nc; // teacher from a given non-compressed log-sum-exp [rows][H] (natural log): it replaces
                         // the sink term, and the window is 0; null otherwise
    float factor;      // loss_coeff / rows (mean) or loss_coeff (sum)
    const int *cu_q;   // THD physical offsets
    const int *cu_real;// THD unpadded offsets (== cu_q when none given)
    const int *cu_c;   // THD compressed offsets (built on device from cu_real)
};

struct Row {
    int b, s, len, v;
    bool pad;
    long long c_base;  // THD: first compressed row of the segment
};

__device__ __forceinline__ Row decode_row(const Geo &g, long long r)
{
    Row R;
    R.c_base = 0;
    if (g.layout == CSA_SBHD) {
        R.s = (int)(r / g.B);
        R.b = (int)(r % g.B);
        R.len = g.S;
    } else if (g.layout == CSA_BSHD) {
        R.b = (int)(r / g.S);
        R.s = (int)(r % g.S);
        R.len = g.S;
    } else {
        // largest b with cu_q[b] <= r (empty segments resolve to the last of equal offsets)
        int lo = 0, hi = g.B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (__ldg(g.cu_q + mid) <= r) lo = mid; else hi = mid - 1;
        }
        R.b = lo;
        R.s = (int)(r - __ldg(g.cu_q + lo));
        R.len = __ldg(g.cu_real + lo + 1) - __ldg(g.cu_real + lo);
        R.c_base = __ldg(g.cu_c + lo);
    }
    R.pad = R.s >= R.len;
    int v = R.pad ? 0 : (R.s + 1) / g.ratio;
    // guards against inconsistent caller metadata (max_seqlen_q, key_rows): a row never addresses more
    // keys than the dense key axis holds, nor compressed rows past the end of k_idx / kv_c
    if (v > g.NC) v = g.NC;
    if (g.layout == CSA_THD && R.c_base + v > g.key_rows) v = R.c_base < g.key_rows ? (int)(g.key_rows - R.c_base) : 0;
    R.v = v;
    return R;
}

// memory row of original position p of the row's segment (query-like tensors)
__device__ __forceinline__ long long q_row(const Geo &g, const Row &R, int p)
{
    if (g.layout == CSA_SBHD) return (long long)p * g.B + R.b;
    if (g.layout == CSA_BSHD) return (long long)R.b * g.S + p;
    return (long long)__ldg(g.cu_q + R.b) + p;
}

// global id of the row's local compressed key j
__device__ __forceinline__ long long key_gid(const Geo &g, const Row &R, int j)
{
    if (g.layout == CSA_THD) return R.c_base + j;
    return (long long)R.b * g.nc + j;
}

// memory row of the compressed key with global id gid
__device__ __forceinline__ long long key_row(const Geo &g, long long gid)
{
    if (g.layout == CSA_SBHD) return (gid % g.nc) * g.B + gid / g.nc;
    return gid;
}

template <typename T> __device__ __forceinline__ float ldf(const T *p, long long i);
template <> __device__ __forceinline__ float ldf<float>(const float *p, long long i) { return __ldg(p + i); }
template <> __device__ __forceinline__ float ldf<__nv_bfloat16>(const __nv_bfloat16 *p, long long i)
{
    return __bfloat162float(p[i]);
}

// plain (non-.nc) load, valid for shared memory as well as global
template <typename T> __device__ __forceinline__ float lds(const T *p, int i);
template <> __device__ __forceinline__ float lds<float>(const float *p, int i) { return p[i]; }
template <> __device__ __forceinline__ float lds<__nv_bfloat16>(const __nv_bfloat16 *p, int i)
{
    return __bfloat162float(p[i]);
}

template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Order-preserving map of an fp32 score to uint32 (larger score -> larger key); -0.0 maps like +0.0.
__device__ __forceinline__ uint32_t score_key(float x)
{
    uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float warp_sum(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float warp_max(float x)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

// ------------------------------------------------------------------ KL of one row, held by one warp
// ([BUG] sec. 2 excerpt: p = softmax of the indexer scores over the support C, L = sum t (log(t + eps) -
// log(p + eps)); g_s = f p_s (A - t_s / (p_s + eps)) with A = sum_k t_k p_k / (p_k + eps), the exact derivative
// of that eps-guarded KL.)  Slot s = lane + 32 i holds the score x[i], the teacher value t[i] and the key's
// offset jj[i] within the row's visible range (-1 off the support).  Writes g by slot (grow, may be null) and
// by key (drow over [0, v), zeroed first; may be null) and returns L (0 for an empty support).
constexpr int kKlPer = 16;          // slots per lane: K <= 512
constexpr float kKlEps = 1e-10f;    // [BUG] sec. 2 excerpt: log(x + 1e-10)
__device__ __forceinline__ float kl_row_warp(const Geo &g, int lane, int K, int v, const int (&jj)[kKlPer],
                                             float (&x)[kKlPer], const float (&t)[kKlPer], float *grow, float *drow)
{
    if (drow != nullptr) {  // zero the visible range (16-byte stores: the row stride is a multiple of 4)
        for (int j4 = lane; 4 * j4 < v; j4 += 32) reinterpret_cast<float4 *>(drow)[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
        __syncwarp();
    }
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < kKlPer; i++)
        if (jj[i] >= 0) m = fmaxf(m, x[i]);
    m = warp_max(m);
    if (m == -INFINITY) {  // empty support: no loss, no gradient
        if (grow != nullptr) {
#pragma unroll
            for (int i = 0; i < kKlPer; i++)
                if (lane + 32 * i < K) grow[lane + 32 * i] = 0.f;
        }
        return 0.f;
    }
    float z = 0.f;
#pragma unroll
    for (int i = 0; i < kKlPer; i++) {
        x[i] = jj[i] >= 0 ? __expf(x[i] - m) : 0.f;
        z += x[i];
    }
    z = warp_sum(z);
    const float inv_z = 1.f / z;
    float A = 0.f, L = 0.f;
#pragma unroll
    for (int i = 0; i < kKlPer; i++) {
        if (jj[i] < 0) continue;
        const float p = x[i] * inv_z;
        A += t[i] * p / (p + kKlEps);
        L += t[i] * (logf(t[i] + kKlEps) - logf(p + kKlEps));
    }
    A = warp_sum(A);
    L = warp_sum(L);
#pragma unroll
    for (int i = 0; i < kKlPer; i++) {
        const int s = lane + 32 * i;
        if (s >= K) continue;
        const float p = x[i] * inv_z;
        const float gv = jj[i] >= 0 ? g.factor * p * (A - t[i] / (p + kKlEps)) : 0.f;
        if (grow != nullptr) grow[s] = gv;
        if (drow != nullptr && jj[i] >= 0) drow[jj[i]] = gv;
    }
    return L;
}

// Row of the by-key gradient rows gd: position-major within each sequence (b S + s for SBHD, the row itself
// otherwise), so the two rows of a position pair are adjacent.
__device__ __forceinline__ long long gd_row_of(const Geo &g, int b, int s, long long r)
{
    return g.layout == CSA_SBHD ? (long long)b * g.S + s : r;
}

// Count of kernel launches made by the library in this process (diagnostics; see csa_kernel_launches).
void note_launches(int n);

// ---------------------------------------------------------------- launchers (k_generic.cu)

cudaError_t launch_build_cu_c(const Geo &g, int *cu_c, cudaStream_t st);
template <typename T>
cudaError_t launch_score_topk_generic(const Geo &g, const T *q_idx, const float *w, const T *k_idx,
                                      int32_t *ids, float *selscore, float *dump, long long dump_row0,
                                      long long dump_rows, cudaStream_t st);
template <typename T>
cudaError_t launch_teacher_generic(const Geo &g, const T *q, const T *kv, const T *kv_c, const float *sink,
                                   const int32_t *ids, float *teacher, cudaStream_t st);
cudaError_t launch_kl(const Geo &g, const int32_t *ids, const float *selscore, const float *dense_scores,
                      const float *teacher, float *gbuf, float *row_loss, float *gd, int ncp, cudaStream_t st);
template <typename T>
cudaError_t launch_grad_generic(const Geo &g, const T *q_idx, const float *w, const T *k_idx,
                                const int32_t *ids, const float *gbuf, T *dq_idx, float *dw, float *dk_acc,
                                cudaStream_t st);
template <typename T>
cudaError_t launch_finalize(const Geo &g, const float *dk_acc, T *dk_idx, const float *row_loss, float *loss,
                            cudaStream_t st);

size_t score_topk_generic_smem(const Geo &g);
size_t teacher_generic_smem(const Geo &g, bool bf16);
size_t grad_generic_smem(const Geo &g);

}  // namespace csa
