// k_teacher_tc.cu -- the full-CSA teacher on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// For query row t and main-attention head h ("[Bug] DSV4 unfused CSA indexer loss ..." (Megatron-LM issue
// #5776): "Paper reference" equations for Z_h and t_j; sec. 3, the attention shares one denominator over the
// sliding window, the selected compressed keys and the sink; the proposal comment's factored form):
//   l_h = log(exp(a_h) + sum_{j in C} exp(c_hj) + sum_{r in W} exp(w_hr)),  c = sigma q.kv_c, w = sigma q.kv
//   T_j = sum_h exp(c_hj - l_h),   t_j = T_j / max(sum_{k in C} T_k, 1e-10)
//
// Mapping (bf16, H = 64 heads, D in {64, 128, 192}).  A work item is 2 consecutive query rows of one sequence.
// The MMA computes D[(row, h), key] = q[row, h] . key with M = 2 rows x 64 heads = 128 (A = the item's q rows,
// K-major, resident), N = 256 keys (B = a tile of kv_c or of the window's kv rows, K-major, TMA), K = D.  N = 256
// keeps the single issuing thread ahead of the tensor core: one MMA runs 128 cycles, about twice what the thread
// needs to issue it together with its share of the barrier traffic.  With
// (row, head) on TMEM lanes each epilogue thread owns one head of one row, so the per-head log-sum-exp is an
// in-register running sum over the key columns.  The keys are taken densely per tile (every visible
// compressed key, every window position) and masked by the row's selection and window.
//   pass 1: window tiles + compressed tiles -> per-(row,h) sum against a reference maximum, then l_h with the
//           sink (or with a given sink-and-window log-sum-exp, when there are no window tiles);
//   pass 2: compressed tiles again, read in the 16-lane TMEM shape -> exp(c - l_h) on selected keys, four heads
//           added per thread and the rest of the 64 heads of a row by a short reduce-scatter, into shared
//           per-key T rows; then the L1 normalisation and the write-out in the id slot order (helper warps).
// Roles: warp 0 TMA, warp 1 TMEM (two 256-column accumulators) + MMA issue, warps 2..17 epilogue (four warps
// per TMEM lane quadrant, each with two 32-column chunks of every tile), warps 18..19 per-item helpers.
// Waits are bounded as in the other tensor-core kernels.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

#include <cudaTypedefs.h>
#include <stdlib.h>

namespace csa {

static __device__ int g_teacher_error = 0;

cudaError_t teacher_tc_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_teacher_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_teacher_error, &zero, sizeof(int));
}

namespace teach {

using namespace ptx;

constexpr int H = 64, RP = 2, M = RP * H, NK = 256;
constexpr int QKB = M * 64 * 2;                 // 16 KB: one 64-wide K-block of the item's 128 (row, head) q rows
constexpr int KB = NK * 64 * 2;                 // 32 KB: one 64-wide K-block of a 256-key tile
constexpr int MAXKB = 3;                        // D <= 192
constexpr int QBUF = MAXKB * QKB;               // 48 KB: the item's q rows
constexpr int BSTG = 3;                         // key K-block stages
constexpr int NCMAX = 1024;
constexpr int THREADS = 640, EPI = 512;          // warps 2..17 epilogue, 18..19 per-item helpers
constexpr uint32_t TMEM_COLS = 512;             // two 256-column fp32 accumulators
constexpr uint32_t IDESC = idesc_bf16(128, NK, false, false);

constexpr int OFF_Q = 0;
constexpr int OFF_B = OFF_Q + 2 * QBUF;                     // 96 KB
constexpr int OFF_T = OFF_B + BSTG * KB;                    // 192 KB: 2 item parities x 2 rows x NCMAX fp32
constexpr int OFF_SEL = OFF_T + 2 * RP * NCMAX * 4;         // 208 KB: selection bit words, 2 x 2 rows x NCMAX bits
constexpr int OFF_PART = OFF_SEL + 2 * RP * NCMAX / 8;      // 2 item parities x 4 column quarters x 128 x (m, s)
constexpr int OFF_MISC = OFF_PART + 2 * 4 * M * 8;
constexpr int SMEM = OFF_MISC + 1024 + 1024;
static_assert(SMEM <= 232448, "teacher shared memory exceeds the per-block limit");

struct Args {
    Geo g;
    const float *sink;
    const int32_t *ids;
    float *teacher;
    const int *cu_g;      // THD: row-pair items per segment [nseg + 1]
    int total;            // SBHD/BSHD items
    int nkb;              // D / 64
};

struct Item {
    int b, n, s0;
    long long row0, row1;
    int v0, v1, vmax;
    int len_real;
    long long gid0, key_y;
    int p_lo, nw, nct;    // window start position, window tiles, compressed tiles
};

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
// bits lo..hi (inclusive) of a 32-bit word, after clamping to 0..31; 0 when the range is empty
__device__ __forceinline__ uint32_t range_bits(int lo, int hi)
{
    if (lo < 0) lo = 0;
    if (hi > 31) hi = 31;
    if (hi < lo) return 0u;
    const uint32_t upto = hi == 31 ? 0xffffffffu : ((1u << (hi + 1)) - 1u);
    return upto & ~((1u << lo) - 1u);
}

__device__ __forceinline__ int find_seg(const int *cu, int nseg, int x)
{
    int lo = 0, hi = nseg - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

__device__ __forceinline__ long long row_of(const Geo &g, int b, int s)
{
    if (g.layout == CSA_SBHD) return (long long)s * g.B + b;
    if (g.layout == CSA_BSHD) return (long long)b * g.S + s;
    return (long long)__ldg(g.cu_q + b) + s;
}

__device__ Item decode(const Args &a, int i, int total)
{
    const Geo &g = a.g;
    Item it;
    int len_phys;
    if (g.layout == CSA_THD) {
        const int ir = total - 1 - i;
        it.b = find_seg(a.cu_g, g.B, ir);
        it.s0 = (ir - __ldg(a.cu_g + it.b)) * RP;
        len_phys = __ldg(g.cu_q + it.b + 1) - __ldg(g.cu_q + it.b);
        it.len_real = __ldg(g.cu_real + it.b + 1) - __ldg(g.cu_real + it.b);
        it.gid0 = __ldg(g.cu_c + it.b);
    } else {
        const int groups = (g.S + RP - 1) / RP;
        it.b = i % g.B;
        it.s0 = (groups - 1 - i / g.B) * RP;
        len_phys = it.len_real = g.S;
        it.gid0 = (long long)it.b * g.nc;
    }
    it.key_y = it.gid0;
    int nc = it.len_real / g.ratio;
    if (nc > g.NC) nc = g.NC;
    if (g.layout == CSA_THD && it.gid0 + nc > g.key_rows) nc = it.gid0 < g.key_rows ? (int)(g.key_rows - it.gid0) : 0;
    it.n = it.s0 + 1 < len_phys ? 2 : 1;
    it.row0 = row_of(g, it.b, it.s0);
    it.row1 = it.n > 1 ? row_of(g, it.b, it.s0 + 1) : it.row0;
    auto vis = [&](int s) { int v = s < it.len_real ? (s + 1) / g.ratio : 0; return v < nc ? v : nc; };
    it.v0 = vis(it.s0);
    it.v1 = it.n > 1 ? vis(it.s0 + 1) : 0;
    it.vmax = it.v0 > it.v1 ? it.v0 : it.v1;
    const int s_last = it.s0 + it.n - 1;
    it.p_lo = it.s0 - g.window + 1;
    if (it.p_lo < 0) it.p_lo = 0;
    it.nw = (it.vmax > 0 && g.window > 0) ? (s_last - it.p_lo + 1 + NK - 1) / NK : 0;
    it.nct = (it.vmax + NK - 1) / NK;
    return it;
}

__device__ __forceinline__ int item_total(const Args &a)
{
    return a.g.layout == CSA_THD ? __ldg(a.cu_g + a.g.B) : a.total;
}

// tile tt of an item: window tiles, then compressed tiles (pass 1), then compressed tiles again (pass 2)
__device__ __forceinline__ int ntiles(const Item &it) { return it.nw + 2 * it.nct; }

// 20 warps: 5 on each of the SM's four schedulers, whose 16 K-register files then cap a thread at 96 registers
__global__ void __launch_bounds__(THREADS, 1)
teacher_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                  const __grid_constant__ CUtensorMap map_kvc, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sQ = smem + OFF_Q;
    unsigned char *sB = smem + OFF_B;
    float *sT = reinterpret_cast<float *>(smem + OFF_T);                // [2][RP][NCMAX]
    uint32_t *sMask = reinterpret_cast<uint32_t *>(smem + OFF_SEL);     // [2][RP][NCMAX / 32]
    float2 *sPart = reinterpret_cast<float2 *>(smem + OFF_PART);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_MISC);
    uint64_t *b_full = bars, *b_empty = bars + BSTG, *q_full = bars + 12, *q_empty = bars + 14;
    uint64_t *t_full = bars + 16, *t_empty = bars + 18, *mma_done = bars + 20;
    uint64_t *mask_full = bars + 22, *t_done = bars + 24;  // [item parity]: helpers -> epilogue, epilogue -> helpers
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC + 256);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 264);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    const bool sbhd = g.layout == CSA_SBHD;
    const int nkb = a.nkb;
    int *err = &g_teacher_error;

    if (threadIdx.x == 0) {
        for (int i = 0; i < BSTG; i++) { mbar_init(b_full + i, 1); mbar_init(b_empty + i, 1); }
        for (int i = 0; i < 2; i++) {
            mbar_init(q_full + i, 1);
            mbar_init(q_empty + i, 1);
            mbar_init(t_full + i, 1);
            mbar_init(t_empty + i, EPI / 32);
            mbar_init(mask_full + i, 2);
            mbar_init(t_done + i, EPI / 32);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = item_total(a);

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ TMA producer
            int hs = 0, ai = 0;
            int last_hs[BSTG];
            int last_ai[2] = {-1, -1};
            for (int i = 0; i < BSTG; i++) last_hs[i] = -1;
            for (int i = blockIdx.x; i < total; i += gridDim.x) {
                const Item it = decode(a, i, total);
                if (it.vmax == 0) continue;
                const int qb = ai & 1;
                wait_bar(q_empty + qb, ((ai >> 1) & 1) ^ 1, abort_flag, err, 41);
                mbar_expect_tx(q_full + qb, (uint32_t)(nkb * QKB));
                for (int r = 0; r < RP; r++)
                    for (int kb = 0; kb < nkb; kb++)
                        tma_load_3d(sQ + qb * QBUF + kb * QKB + r * (H * 128), &map_q, q_full + qb, kb * 64, 0,
                                    (int)(r == 0 ? it.row0 : it.row1));
                last_ai[qb] = ai;
                ai++;
                const int nt = ntiles(it);
                for (int tt = 0; tt < nt; tt++) {
                    const bool win = tt < it.nw;
                    const int t = win ? tt : (tt - it.nw) % (it.nct > 0 ? it.nct : 1);
                    for (int kb = 0; kb < nkb; kb++) {
                        const int st = hs % BSTG;
                        wait_bar(b_empty + st, ((hs / BSTG) & 1) ^ 1, abort_flag, err, 42);
                        mbar_expect_tx(b_full + st, KB);
                        unsigned char *dst = sB + st * KB;
                        if (win) {
                            const int p = it.p_lo + t * NK;
                            if (sbhd) tma_load_3d(dst, &map_kv, b_full + st, kb * 64, it.b, p);
                            else tma_load_2d(dst, &map_kv, b_full + st, kb * 64, (int)row_of(g, it.b, p));
                        } else {
                            if (sbhd) tma_load_3d(dst, &map_kvc, b_full + st, kb * 64, it.b, t * NK);
                            else tma_load_2d(dst, &map_kvc, b_full + st, kb * 64, (int)(it.key_y + t * NK));
                        }
                        last_hs[st] = hs;
                        hs++;
                    }
                }
            }
            for (int st = 0; st < BSTG; st++)
                if (last_hs[st] >= 0) drain_bar(b_full + st, (last_hs[st] / BSTG) & 1, err);
            for (int qb = 0; qb < 2; qb++)
                if (last_ai[qb] >= 0) drain_bar(q_full + qb, (last_ai[qb] >> 1) & 1, err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA issue (whole warp)
        // The warp runs the loop together (warp-uniform stage indices and descriptors); one elected lane issues
        // each MMA and commit.  Items are decoded lane-parallel (lane l: the CTA's item k + l) and the loop reads
        // the tile count of item k by a shuffle.  B-stage ring position (st, parity bph).  A barrier probe costs
        // a shared-memory round trip, so the barriers of a whole tile (its accumulator and its nkb B stages) are
        // probed together, once per 4 nkb MMAs; only those not yet complete are then waited on.
        int st = 0, ai = 0, tc = 0, k = 0, nt_lane = 0;
        uint32_t bph = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int il = i + lane * (int)gridDim.x;
                if (il < total) {
                    const Item itl = decode(a, il, total);
                    nt_lane = itl.vmax == 0 ? 0 : ntiles(itl);
                } else {
                    nt_lane = 0;
                }
            }
            const int nt = __shfl_sync(0xffffffffu, nt_lane, k & 31);
            if (nt == 0) continue;
            const int qb = ai & 1;
            wait_bar(q_full + qb, (ai >> 1) & 1, abort_flag, err, 43);
            fence_after();
            const unsigned char *pq = sQ + qb * QBUF;
            for (int tt = 0; tt < nt; tt++) {
                const int tb = tc & 1;
                int sk[MAXKB];
                uint32_t pk[MAXKB];
                bool rk[MAXKB];
                const uint32_t tpar = ((tc >> 1) & 1) ^ 1;
                const bool rt = mbar_test(t_empty + tb, tpar);
#pragma unroll
                for (int kb = 0; kb < MAXKB; kb++) {
                    sk[kb] = st;
                    pk[kb] = bph;
                    rk[kb] = kb < nkb ? mbar_test(b_full + st, bph) : true;
                    if (kb < nkb && ++st == BSTG) {
                        st = 0;
                        bph ^= 1u;
                    }
                }
                if (!rt) wait_bar(t_empty + tb, tpar, abort_flag, err, 44);
#pragma unroll
                for (int kb = 0; kb < MAXKB; kb++)
                    if (!rk[kb]) wait_bar(b_full + sk[kb], pk[kb], abort_flag, err, 45);
                fence_after();
                const uint32_t d = tmem + tb * NK;
#pragma unroll
                for (int kb = 0; kb < MAXKB; kb++) {
                    if (kb >= nkb) break;
                    const unsigned char *pa = pq + kb * QKB, *pb = sB + sk[kb] * KB;
#pragma unroll
                    for (int k4 = 0; k4 < 4; k4++)
                        mma_bf16_w(d, desc_kmajor(pa + k4 * 32), desc_kmajor(pb + k4 * 32), IDESC, (kb | k4) ? 1u : 0u);
                    mma_commit_w(b_empty + sk[kb]);
                }
                mma_commit_w(t_full + tb);
                tc++;
            }
            mma_commit_w(q_empty + qb);
            ai++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp < 18) {
        // ---------------------------------------------------------------- epilogue
        // 16 warps: four per TMEM lane quadrant (warp % 4), warp cq = (warp - 2) / 4 of a quadrant reads two
        // 32-column chunks of every tile (col_of below).  The selection masks and the zeroed T rows of an
        // item come from the helper warps (buffer ic & 1), which also normalise and write the T rows.
        const int e = warp - 2, quad = warp & 3, cq = e >> 2;
        const int rh = quad * 32 + lane;      // (row, head) of this thread's TMEM lane
        const int i_row = rh >> 6, h = rh & 63;
        const float s2 = g.scale * 1.4426950408889634f;  // logits in log2 units: exp(c) = 2^(x * sigma * log2 e)
        const bool s2_pos = s2 > 0.f;  // then max(x s2) = s2 max(x): the scale folds into one FFMA per element
        // chunk c (0, 1) of warp cq covers columns [32 cq + 128 c, +32): the four warps of a quadrant share the
        // first 128 columns of a tile, so a partly filled tile (the window's, a row's last) keeps them all busy
        auto col_of = [&](int c) { return cq * 32 + c * 128; };
        int tc = 0;
        int ic = 0;
        for (int it_i = blockIdx.x; it_i < total; it_i += gridDim.x, ic++) {
            const Item it = decode(a, it_i, total);
            const int vme = i_row == 0 ? it.v0 : it.v1;
            const int s_me = it.s0 + i_row;
            const int ib = ic & 1;
            float *sTb = sT + ib * RP * NCMAX;
            const uint32_t *sMaskb = sMask + ib * RP * (NCMAX / 32);
            wait_bar(mask_full + ib, (ic >> 1) & 1, abort_flag, err, 47);
            // running log2-domain max and sum of this thread's (row, head) over its key columns
            float m = -INFINITY, ssum = 0.f, ell = 0.f;
            float ell4[4] = {0.f, 0.f, 0.f, 0.f};  // l_h of heads g, g + 8, g + 16, g + 24 of the quadrant
            const int nt = ntiles(it);
            const bool row_ok = s_me < it.len_real;
            for (int tt = 0; tt < nt; tt++) {
                const int tb = tc & 1;
                wait_bar(t_full + tb, (tc >> 1) & 1, abort_flag, err, 46);
                fence_after();
                const bool win = tt < it.nw;
                const bool pass2 = tt >= it.nw + it.nct;
                const int t = win ? tt : (tt - it.nw) % it.nct;
                if (pass2 && tt == it.nw + it.nct) {
                    // l_h (log2 units) from the four column quarters, combined in a fixed order, and the sink
                    // (sPart alternates by item parity: a warp can reach the next item's combine before a slow
                    // one has read this one's)
                    float2 *pp = sPart + ib * 4 * M;
                    pp[cq * M + rh] = make_float2(m, ssum);
                    named_bar(1, EPI);
                    float2 p[4];
#pragma unroll
                    for (int k = 0; k < 4; k++) p[k] = pp[k * M + rh];
                    // the non-compressed term: the sink, or a given sink-and-window log-sum-exp of this row
                    const float ah = g.lse_nc != nullptr
                                         ? __ldg(g.lse_nc + (i_row == 0 ? it.row0 : it.row1) * H + h) * 1.4426950408889634f
                                         : (g.no_sink ? -INFINITY : __ldg(a.sink + h) * 1.4426950408889634f);
                    const float mm = fmaxf(fmaxf(fmaxf(p[0].x, p[1].x), fmaxf(p[2].x, p[3].x)), ah);
                    float S = 0.f;
                    if (mm != -INFINITY) {
#pragma unroll
                        for (int k = 0; k < 4; k++)
                            if (p[k].x != -INFINITY) S += p[k].y * ex2(p[k].x - mm);
                        if (ah != -INFINITY) S += ex2(ah - mm);
                    }
                    ell = mm + lg2(S);
#pragma unroll
                    for (int k4 = 0; k4 < 4; k4++) ell4[k4] = __shfl_sync(0xffffffffu, ell, (lane >> 2) + 8 * k4);
                }
                // mask words of this warp's two 32-column chunks; they depend only on the warp's row, so the
                // skip of an all-masked sub-chunk and the full-word fast paths below are warp-uniform
                uint32_t mw[2];
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    const int col0 = col_of(c);
                    if (win) {
                        const int pbase = it.p_lo + t * NK + col0;
                        mw[c] = row_ok ? range_bits(s_me - g.window + 1 - pbase, s_me - pbase) : 0u;
                    } else {
                        const int j0 = t * NK + col0;
                        mw[c] = j0 < NCMAX ? (sMaskb[i_row * (NCMAX / 32) + (j0 >> 5)] & range_bits(0, vme - 1 - j0)) : 0u;
                    }
                }
                if ((mw[0] | mw[1]) != 0u) {
                    if (!pass2) {
                        // running sum against a reference max, one 32-column chunk at a time: the first chunk
                        // with columns sets the reference; a later chunk is summed against it directly and only
                        // re-based on its own max when its sum leaves the safe range (a logit more than ~64
                        // log2 units above the reference), so the common chunk needs no max pass
#pragma unroll 1
                        for (int c = 0; c < 2; c++) {
                            if (mw[c] == 0u) continue;
                            float x[32];
                            tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(tb * NK + col_of(c)), x);
                            if (s2_pos) {
                                if (mw[c] != 0xffffffffu) {
#pragma unroll
                                    for (int q = 0; q < 32; q++) x[q] = (mw[c] >> q) & 1u ? x[q] : -INFINITY;
                                }
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; q++) x[q] = (mw[c] >> q) & 1u ? x[q] * s2 : -INFINITY;
                            }
                            const float sc = s2_pos ? s2 : 1.f;
                            auto chunk_max = [&]() -> float {  // finite: the chunk holds an unmasked column
                                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                                for (int q = 0; q < 32; q++) mx[q & 3] = fmaxf(mx[q & 3], x[q]);
                                return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
                            };
                            auto chunk_sum = [&]() -> float {
                                float2 sm[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // columns q % 4
#pragma unroll
                                for (int q2 = 0; q2 < 16; q2++) {
                                    const float2 arg = fma2(make_float2(x[2 * q2], x[2 * q2 + 1]), make_float2(sc, sc),
                                                            make_float2(-m, -m));
                                    sm[q2 & 1] = add2(sm[q2 & 1], make_float2(ex2(arg.x), ex2(arg.y)));
                                }
                                return (sm[0].x + sm[0].y) + (sm[1].x + sm[1].y);
                            };
                            if (m == -INFINITY) m = chunk_max();
                            float cs = chunk_sum();
                            if (!(cs <= 0x1p64f)) {
                                const float cm = chunk_max();
                                if (cm > m) {
                                    ssum *= ex2(m - cm);
                                    m = cm;
                                }
                                cs = chunk_sum();
                            }
                            ssum += cs;
                        }
                    } else {
                        // pass 2, read in the 16-lane shape: a thread holds heads g, g + 8, g + 16, g + 24
                        // (g = lane / 4) of columns 8 p + 2 u + e (u = lane % 4, p = 0..3, e = 0..1); it adds its
                        // four heads in registers, and the eight threads of a column set reduce-scatter over g,
                        // leaving thread (g, u) with the 32-head sum of column 8 (g / 2) + 2 u + g % 2
                        const int u4 = lane & 3, g8 = lane >> 2;
#pragma unroll 1
                        for (int c = 0; c < 2; c++) {
                            if (mw[c] == 0u) continue;
                            const uint32_t ca = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(tb * NK + col_of(c));
                            uint32_t ra[16], rb[16];
                            tmem_ld16x256_x4(ca, ra);              // heads g, g + 8
                            tmem_ld16x256_x4(ca + (16u << 16), rb);  // heads g + 16, g + 24
                            const bool full = mw[c] == 0xffffffffu;
                            float s8[8];
#pragma unroll
                            for (int p4 = 0; p4 < 4; p4++) {
                                const int col = 8 * p4 + 2 * u4;
                                const bool b0 = full || ((mw[c] >> col) & 1u), b1 = full || ((mw[c] >> (col + 1)) & 1u);
                                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                                for (int k4 = 0; k4 < 4; k4++) {
                                    const uint32_t *r = k4 < 2 ? ra : rb;
                                    const int o = 4 * p4 + 2 * (k4 & 1);
                                    const float2 arg = fma2(make_float2(__uint_as_float(r[o]), __uint_as_float(r[o + 1])),
                                                            make_float2(s2, s2), make_float2(-ell4[k4], -ell4[k4]));
                                    const float e0 = ex2(arg.x), e1 = ex2(arg.y);  // then the mask: no branch
                                    acc = add2(acc, make_float2(b0 ? e0 : 0.f, b1 ? e1 : 0.f));
                                }
                                s8[2 * p4] = acc.x;
                                s8[2 * p4 + 1] = acc.y;
                            }
#pragma unroll
                            for (int hv = 4; hv >= 1; hv >>= 1) {
                                const int off = hv * 4;  // the lane bit of g's bit log2(hv)
                                const bool up = (lane & off) != 0;
#pragma unroll
                                for (int q = 0; q < hv; q++) {
                                    const float send = up ? s8[q] : s8[q + hv];
                                    const float keep = up ? s8[q + hv] : s8[q];
                                    s8[q] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                                }
                            }
                            const int j = t * NK + col_of(c) + 8 * (g8 >> 1) + 2 * u4 + (g8 & 1);
                            if (j < NCMAX && s8[0] != 0.f) atomicAdd(sTb + i_row * NCMAX + j, s8[0]);
                        }
                    }
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(t_empty + tb);
                tc++;
            }
            // this warp's T contributions to buffer ib are in
            __syncwarp();
            if (lane == 0) mbar_arrive(t_done + ib);
        }
    } else {
        // ---------------------------------------------------------------- per-item helpers (warps 18, 19)
        // Warp 18 + r owns row r of every item.  For item ic (buffer ic & 1): zero its T row, build its selection
        // bit words, signal mask_full; then, once the epilogue has summed item ic - 1 into the other buffer
        // (t_done), L1-normalise that row and write it out in the id slot order.  Buffer reuse is ordered by the
        // warp's own program order (item ic - 2's write-out precedes item ic's set-up).
        const int r = warp - 18;
        auto writeout = [&](const Item &it, int icw) {
            const int ib = icw & 1;
            wait_bar(t_done + ib, (icw >> 1) & 1, abort_flag, err, 48);
            if (r >= it.n) return;
            const float *tr = sT + (ib * RP + r) * NCMAX;
            const int v = r == 0 ? it.v0 : it.v1;
            float part = 0.f;
            for (int j = lane; j < v; j += 32) part += tr[j];
            const float inv = 1.f / fmaxf(warp_sum(part), 1e-10f);
            const long long row = r == 0 ? it.row0 : it.row1;
            float *trow = a.teacher + row * g.TW;
            if (g.sparse) {
                for (int s = lane; s < g.TW; s += 32) {
                    const int32_t id = s < g.K ? __ldg(a.ids + row * g.K + s) : -1;
                    const long long j = (long long)id - it.gid0;
                    trow[s] = (id >= 0 && j >= 0 && j < v) ? tr[j] * inv : 0.f;
                }
            } else {
                for (int j = lane; j < g.TW; j += 32) trow[j] = j < v ? tr[j] * inv : 0.f;
            }
        };
        Item prev;
        int ic = 0;
        for (int it_i = blockIdx.x; it_i < total; it_i += gridDim.x, ic++) {
            const Item it = decode(a, it_i, total);
            const int ib = ic & 1;
            float4 *tz = reinterpret_cast<float4 *>(sT + (ib * RP + r) * NCMAX);
            for (int x = lane; x < NCMAX / 4; x += 32) tz[x] = make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t *mk = sMask + (ib * RP + r) * (NCMAX / 32);
            const int v = r == 0 ? it.v0 : it.v1;
            if (g.sparse) {
                mk[lane] = 0u;
                __syncwarp();
                if (r < it.n && v > 0) {
                    const long long row = r == 0 ? it.row0 : it.row1;
                    for (int s = lane; s < g.K; s += 32) {
                        const int32_t id = __ldg(a.ids + row * g.K + s);
                        const long long j = (long long)id - it.gid0;
                        if (id >= 0 && j >= 0 && j < v) atomicOr(mk + (j >> 5), 1u << (j & 31));
                    }
                }
            } else {
                mk[lane] = range_bits(0, v - 1 - lane * 32);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mask_full + ib);
            if (ic > 0) writeout(prev, ic - 1);
            prev = it;
        }
        if (ic > 0) writeout(prev, ic - 1);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

__global__ void build_items_kernel(Geo g, int *cu_g)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    cu_g[0] = 0;
    for (int b = 0; b < g.B; b++) {
        const int lp = __ldg(g.cu_q + b + 1) - __ldg(g.cu_q + b);
        acc += lp > 0 ? (lp + RP - 1) / RP : 0;
        cu_g[b + 1] = acc;
    }
}

}  // namespace teach

// ------------------------------------------------------------------ host side

bool tc_teacher_supported(const Geo &g, bool bf16)
{
    const char *f = getenv("CSA_FORCE_GENERIC");
    if (f != nullptr && f[0] == '1') return false;
    return bf16 && g.H == teach::H && g.D % 64 == 0 && g.D / 64 >= 1 && g.D / 64 <= teach::MAXKB && g.NC >= 1 &&
           g.NC <= teach::NCMAX && g.K >= 1 && g.rows > 0 && g.key_rows > 0 && g.TW <= 4096;
}

size_t tc_teacher_workspace_bytes(const Geo &g) { return sizeof(int) * (size_t)(g.layout == CSA_THD ? g.B + 1 : 1); }

cudaError_t launch_teacher_tc(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *kv,
                              const __nv_bfloat16 *kv_c, const float *sink, const int32_t *ids, float *teacher,
                              void *ws, cudaStream_t st)
{
    using namespace teach;
    CUtensorMap mq, mkv, mkc;
    // q as [rows][H][D] with a 64 x 64 x 1 box
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.D, (cuuint64_t)g.H, (cuuint64_t)g.rows};
        const cuuint64_t strides[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.H * g.D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)g.H, 1};
        if (!tc_encode_bf16(&mq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    if (g.window == 0) {  // no window tile is ever loaded: the kv map is never used
        if (g.layout == CSA_SBHD) {
            const cuuint64_t dkc[3] = {(cuuint64_t)g.D, (cuuint64_t)g.B, (cuuint64_t)g.nc};
            const cuuint64_t skc[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.B * g.D * 2};
            const cuuint32_t box[3] = {64, 1, (cuuint32_t)NK};
            if (!tc_encode_bf16(&mkc, kv_c, 3, dkc, skc, box)) return cudaErrorInvalidValue;
        } else {
            const cuuint64_t dkc[2] = {(cuuint64_t)g.D, (cuuint64_t)g.key_rows};
            const cuuint64_t s1[1] = {(cuuint64_t)g.D * 2};
            const cuuint32_t box[2] = {64, (cuuint32_t)NK};
            if (!tc_encode_bf16(&mkc, kv_c, 2, dkc, s1, box)) return cudaErrorInvalidValue;
        }
        mkv = mkc;
    } else if (g.layout == CSA_SBHD) {
        const cuuint64_t dkv[3] = {(cuuint64_t)g.D, (cuuint64_t)g.B, (cuuint64_t)g.S};
        const cuuint64_t skv[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.B * g.D * 2};
        const cuuint64_t dkc[3] = {(cuuint64_t)g.D, (cuuint64_t)g.B, (cuuint64_t)g.nc};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)NK};
        if (!tc_encode_bf16(&mkv, kv, 3, dkv, skv, box) || !tc_encode_bf16(&mkc, kv_c, 3, dkc, skv, box))
            return cudaErrorInvalidValue;
    } else {
        const cuuint64_t dkv[2] = {(cuuint64_t)g.D, (cuuint64_t)g.rows};
        const cuuint64_t dkc[2] = {(cuuint64_t)g.D, (cuuint64_t)g.key_rows};
        const cuuint64_t s1[1] = {(cuuint64_t)g.D * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)NK};
        if (!tc_encode_bf16(&mkv, kv, 2, dkv, s1, box) || !tc_encode_bf16(&mkc, kv_c, 2, dkc, s1, box))
            return cudaErrorInvalidValue;
    }
    Args a = {};  // every field set below; zero first so none is ever left unset
    a.g = g;
    a.sink = sink;
    a.ids = ids;
    a.teacher = teacher;
    a.cu_g = nullptr;
    a.total = 0;
    a.nkb = g.D / 64;
    int upper;
    if (g.layout == CSA_THD) {
        int *cu_g = static_cast<int *>(ws);
        build_items_kernel<<<1, 32, 0, st>>>(g, cu_g);
        note_launches(1);
        a.cu_g = cu_g;
        upper = (g.rows + RP - 1) / RP + g.B;
    } else {
        a.total = g.B * ((g.S + RP - 1) / RP);
        upper = a.total;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(teacher_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const int grid = upper < sms ? (upper > 0 ? upper : 1) : sms;
    teacher_tc_kernel<<<grid, THREADS, SMEM, st>>>(mq, mkv, mkc, a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
