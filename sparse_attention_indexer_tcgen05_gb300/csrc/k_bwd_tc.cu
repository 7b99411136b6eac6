// k_bwd_tc.cu -- the indexer backward on the 5th-generation tensor cores (tcgen05 + TMEM + TMA).
//
// Given g_ts = dloss/dI_ts (from the KL step, zero outside the support C), the gradients of
// I[t,s] = sum_j w[t,j] max(0, x_tjs), x_tjs = q_idx[t,j] . k_idx[s] are
//   dQ'[t,j] = sum_s g_ts 1[x_tjs > 0] k_idx[s]           dQ_idx[t,j] = w[t,j] dQ'[t,j]
//   dW[t,j]  = sum_s g_ts max(0, x_tjs) = q_idx[t,j] . dQ'[t,j]
//   dK[s]    = sum_t sum_j g_ts w[t,j] 1[x_tjs > 0] q_idx[t,j]
// ("[Bug] DSV4 unfused CSA indexer loss ..." (Megatron-LM issue #5776), the proposal comment: gradients only
// for the indexer Q, weights and K; "Megatron-LM PR #8539" item 1: the backward takes global top-k ids.)
//
// x is recomputed on the tensor cores over every visible key tile (dense in keys, masked by g), so both
// kernels stream contiguous k_idx / q_idx tiles by TMA; no per-element global atomics:
//   * row-owner kernel (dQ_idx, dW): a work item is 2 query rows (N = 128 (row, head) pairs).  Per key tile:
//     MMA1 X[key, (row,h)] = k . q^T (M 128 keys, K 128), the epilogue forms G'[key, (row,h)] =
//     g 1[x > 0] in bf16 as an MN-major operand, and MMA2 accumulates dQ'^T... stored as
//     D[(row,h), d] += sum_key G'[key,(row,h)] k[key, d] in TMEM over all tiles of the item.
//   * key-owner kernel (dK): a unit is one key tile and a chunk of up to 128 rows that see it.  Per row pair:
//     MMA1 as above, the epilogue forms G[key, (row,h)] = g w 1[x > 0] (K-major), and MMA3 accumulates
//     dK[key, d] += sum_(row,h) G q[(row,h), d] in TMEM; the unit flushes its 128 x 128 fp32 partial once.
// Roles: warp 0 TMA, warp 1 TMEM + MMA issue, warp 2 stages each item's g (and w) into shared memory ahead of
// use, warps 4..11 epilogue.  Waits are bounded as in the score kernel.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

#include <stdlib.h>

namespace csa {

static __device__ int g_bwd_error = 0;

cudaError_t bwd_tc_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_bwd_error, &zero, sizeof(int));
}

namespace bwd {

using namespace ptx;

constexpr int HI = 64, DI = 128, NKEY = 128;
constexpr int RP = 2;                          // query rows per item / row pair
constexpr int M_PAIRS = RP * 64;               // (row, head) pairs of an item
constexpr int NCMAX = 1024;                    // key axis the row-owner's dense g rows hold
constexpr int HALF = NKEY * 64 * 2;            // 16 KB: 128 rows x 64 bf16
constexpr int QBLK = 2 * HALF;                 // 32 KB: 2 rows x 64 heads x 128 d, two K-halves
constexpr int THREADS = 384;                   // key-owner kernel: 12 warps
constexpr int EPI = 256;                       //   its epilogue: warps 4..11
constexpr int R_THREADS = 640;                 // row-owner kernel: 20 warps
constexpr int R_EPI = 512;                     //   its epilogue: warps 4..19, four per TMEM lane quadrant
constexpr int CH = 128;                        // rows per key-owner unit
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_X = idesc_bf16(128, 128, false, false);   // X = k . q^T (key-owner), X^T = q . k^T
constexpr uint32_t IDESC_DQ = idesc_bf16(128, 128, false, true);   // dQ' += G'^T k  (A in TMEM, B MN-major)
constexpr uint32_t IDESC_DK = idesc_bf16(128, 128, false, true);   // dK += G q      (A in TMEM, B MN-major)

// row-owner shared memory
constexpr int R_ASTG = 8;                                     // k-tile halves: four tiles in flight
constexpr int R_XSTG = 3;                                     // X / G' TMEM slots
static_assert((2 * R_ASTG + 11 + 3 * R_XSTG) * 8 <= 512, "row-owner barriers overlap the TMEM slot");
constexpr int R_OFF_A = 0;
constexpr int R_OFF_B = R_OFF_A + R_ASTG * HALF;              // 128 KB: the q tiles of two items
constexpr int R_OFF_GD = R_OFF_B + 2 * QBLK;                  // 192 KB: 2 bufs x 2 rows x NCMAX fp32
constexpr int R_OFF_W = R_OFF_GD + 2 * RP * NCMAX * 4;        // 208 KB: 2 bufs x 2 rows x 64 fp32
constexpr int R_OFF_DW = R_OFF_W + 2 * RP * HI * 4;           // dW partials: 2 item parities x 4 d quarters x 128
constexpr int R_OFF_MISC = R_OFF_DW + 2 * 4 * M_PAIRS * 4;
constexpr int R_SMEM = R_OFF_MISC + 1024 + 1024;

// key-owner shared memory
constexpr int K_BSTG = 5, K_GSTG = 4;
constexpr int K_OFF_A = 0;                                     // the unit's key tile, 32 KB
constexpr int K_OFF_B = K_OFF_A + 2 * HALF;                    // 5 q blocks (G lives in TMEM)
constexpr int K_OFF_GT = K_OFF_B + K_BSTG * QBLK;              // g tiles: 4 x 2 rows x 128 fp32
constexpr int K_OFF_WT = K_OFF_GT + K_GSTG * RP * NKEY * 4;    // w rows: 4 x 2 rows x 64 fp32
constexpr int K_OFF_MISC = K_OFF_WT + K_GSTG * RP * HI * 4;
constexpr int K_SMEM = K_OFF_MISC + 1024 + 1024;
static_assert((2 + 2 * K_BSTG + 10 + 2 * K_GSTG + 1) * 8 <= 256, "key-owner barriers overlap the TMEM slot");

struct Args {
    Geo g;
    const float *w;
    const int32_t *ids;      // [rows, K]
    const float *gbuf;       // [rows, TW] dloss/dI in the teacher's slot layout
    const int32_t *toff;     // [rows, NT + 1] first slot of each key tile (sparse)
    int NT;                  // key tiles of the widest key axis
    __nv_bfloat16 *dq;
    float *dw;
    float *dk_acc;           // [key rows, DI] fp32, zeroed by the caller
    const int *cu_g;         // THD: row-pair items per segment [nseg+1]
    const int *cu_u;         // THD: key-owner units per segment [nseg+1]
    int total_items, total_units;     // SBHD/BSHD
    int units_per_seq;                // SBHD/BSHD
};

// ------------------------------------------------------------------ geometry

struct Seg {
    int b, len_phys, len_real, nc;
    long long gid0;          // global id of local key 0
    long long key_y;         // TMA row coordinate of local key 0 (2D maps)
};

__device__ __forceinline__ Seg seg_of(const Geo &g, int b)
{
    Seg s;
    s.b = b;
    if (g.layout == CSA_THD) {
        s.len_phys = __ldg(g.cu_q + b + 1) - __ldg(g.cu_q + b);
        s.len_real = __ldg(g.cu_real + b + 1) - __ldg(g.cu_real + b);
        s.gid0 = __ldg(g.cu_c + b);
    } else {
        s.len_phys = s.len_real = g.S;
        s.gid0 = (long long)b * g.nc;
    }
    s.key_y = s.gid0;
    int nc = s.len_real / g.ratio;
    if (nc > g.NC) nc = g.NC;
    if (g.layout == CSA_THD && s.gid0 + nc > g.key_rows) nc = s.gid0 < g.key_rows ? (int)(g.key_rows - s.gid0) : 0;
    s.nc = nc;
    return s;
}

__device__ __forceinline__ long long row_of(const Geo &g, int b, int s)
{
    if (g.layout == CSA_SBHD) return (long long)s * g.B + b;
    if (g.layout == CSA_BSHD) return (long long)b * g.S + s;
    return (long long)__ldg(g.cu_q + b) + s;
}

__device__ __forceinline__ int vis(const Geo &g, const Seg &sg, int s)
{
    if (s >= sg.len_real) return 0;
    int v = (s + 1) / g.ratio;
    return v < sg.nc ? v : sg.nc;
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

// A row-pair item of the row-owner kernel.
struct Pair {
    Seg sg;
    int n;                    // rows present (1..2)
    long long row0, row1;
    int v0, v1, vmax;
};

__device__ Pair decode_pair(const Args &a, int i)
{
    const Geo &g = a.g;
    Pair p;
    int b, s0;
    if (g.layout == CSA_THD) {
        const int total = __ldg(a.cu_g + g.B);
        const int ir = total - 1 - i;
        b = find_seg(a.cu_g, g.B, ir);
        s0 = (ir - __ldg(a.cu_g + b)) * RP;
    } else {
        const int groups = (g.S + RP - 1) / RP;
        b = i % g.B;
        s0 = (groups - 1 - i / g.B) * RP;
    }
    p.sg = seg_of(g, b);
    p.n = s0 + 1 < p.sg.len_phys ? 2 : 1;
    p.row0 = row_of(g, b, s0);
    p.row1 = p.n > 1 ? row_of(g, b, s0 + 1) : p.row0;
    p.v0 = vis(g, p.sg, s0);
    p.v1 = p.n > 1 ? vis(g, p.sg, s0 + 1) : 0;
    p.vmax = p.v0 > p.v1 ? p.v0 : p.v1;
    return p;
}

__device__ __forceinline__ int pair_total(const Args &a)
{
    return a.g.layout == CSA_THD ? __ldg(a.cu_g + a.g.B) : a.total_items;
}

// Key-owner units sit on an absolute grid of CH-row chunks; chunk c of a segment is paired with every key
// tile its rows can see, key tiles fastest, so the units that read the same q_idx rows run at the same
// time and share them through L2.
__host__ __device__ inline int chunk_tiles(int c, int len_real, int nc, int ratio)
{
    int last = (c + 1) * CH < len_real ? (c + 1) * CH : len_real;  // one past the chunk's last position
    int v = last / ratio;                                           // visible keys of its last row
    if (v > nc) v = nc;
    return (v + NKEY - 1) / NKEY;
}

__host__ __device__ inline int units_of_len(int len_real, int nc, int ratio)
{
    int u = 0;
    const int nch = (len_real + CH - 1) / CH;
    for (int c = 0; c < nch; c++) u += chunk_tiles(c, len_real, nc, ratio);
    return u;
}

struct Unit {
    Seg sg;
    int kt;
    int s_lo, s_hi;           // row positions [s_lo, s_hi)
    int npairs;
};

__device__ Unit decode_unit(const Args &a, int u)
{
    const Geo &g = a.g;
    Unit U;
    int b, lu;
    if (g.layout == CSA_THD) {
        b = find_seg(a.cu_u, g.B, u);
        lu = u - __ldg(a.cu_u + b);
    } else {
        b = u % g.B;
        lu = u / g.B;
    }
    U.sg = seg_of(g, b);
    U.kt = 0;
    U.s_lo = U.s_hi = 0;
    const int nch = (U.sg.len_real + CH - 1) / CH;
    for (int c = 0; c < nch; c++) {
        const int nt = chunk_tiles(c, U.sg.len_real, U.sg.nc, g.ratio);
        if (lu < nt) {
            U.kt = lu;
            U.s_lo = c * CH;
            U.s_hi = min(U.sg.len_real, U.s_lo + CH);
            break;
        }
        lu -= nt;
    }
    U.npairs = (U.s_hi - U.s_lo + 1) / RP;
    return U;
}

__device__ __forceinline__ int unit_total(const Args &a)
{
    return a.g.layout == CSA_THD ? __ldg(a.cu_u + a.g.B) : a.total_units;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// ------------------------------------------------------------------ row-owner kernel: dQ_idx, dW

__global__ void __launch_bounds__(R_THREADS, 1)
dq_dw_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem + R_OFF_A;
    unsigned char *sB = smem + R_OFF_B;
    float *sGD = reinterpret_cast<float *>(smem + R_OFF_GD);
    float *sW = reinterpret_cast<float *>(smem + R_OFF_W);
    float *sDW = reinterpret_cast<float *>(smem + R_OFF_DW);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + R_OFF_MISC);
    uint64_t *a_full = bars, *a_empty = bars + R_ASTG, *b_full = bars + 2 * R_ASTG, *b_empty = b_full + 2;
    uint64_t *x_full = b_full + 4, *x_empty = x_full + R_XSTG, *g_full = x_empty + R_XSTG;
    uint64_t *dq_full = g_full + R_XSTG, *dq_empty = dq_full + 1, *gd_full = dq_full + 2, *gd_empty = dq_full + 4;
    uint64_t *mma_done = dq_full + 6;                                  // 2 R_ASTG + 11 + 3 R_XSTG barriers
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + R_OFF_MISC + 512);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + R_OFF_MISC + 520);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    const bool sbhd = g.layout == CSA_SBHD;
    int *err = &g_bwd_error;

    if (threadIdx.x == 0) {
        for (int i = 0; i < R_ASTG; i++) { mbar_init(a_full + i, 1); mbar_init(a_empty + i, 1); }
        for (int i = 0; i < 2; i++) {
            mbar_init(b_full + i, 1);
            mbar_init(b_empty + i, R_EPI / 32);
            mbar_init(gd_full + i, 1);
            mbar_init(gd_empty + i, R_EPI / 32);
        }
        for (int i = 0; i < R_XSTG; i++) {
            mbar_init(x_full + i, 1);
            mbar_init(x_empty + i, 1);
            mbar_init(g_full + i, R_EPI / 32);
        }
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, R_EPI / 32);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: three slots of 128 columns, each holding one key tile's X^T (fp32) and then, in place, its G'^T as
    // the A operand of dQ' (bf16 pairs; epilogue warp qq writes its 16 pair columns over the first half of its
    // own 32 X columns, so key pairs of keys [16 s, 16 s + 16) sit at column 32 (s / 2) + 8 (s % 2)); dQ' (128).
    const uint32_t tX = tmem, tDQ = tmem + R_XSTG * 128;
    const int total = pair_total(a);

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ TMA producer
            // k tiles stream through the half-stage ring; an item's q tile is requested as soon as its buffer
            // is free: that buffer is probed before every k-half load of the previous item, and waited for at
            // the latest when the item starts.
            int hs = 0, ai = 0, qi = 0;
            int last_hs[R_ASTG];
            int last_q[2] = {-1, -1};
            for (int i = 0; i < R_ASTG; i++) last_hs[i] = -1;
            auto load_q = [&](const Pair &p) {
                const int bb = qi & 1;
                mbar_expect_tx(b_full + bb, QBLK);
                for (int r = 0; r < RP; r++)
                    for (int kh = 0; kh < 2; kh++)
                        tma_load_3d(sB + bb * QBLK + kh * HALF + r * (HI * 128), &map_q, b_full + bb, kh * 64, 0,
                                    (int)(r == 0 ? p.row0 : p.row1));
                last_q[bb] = qi;
                qi++;
            };
            // the next item with visible keys after item index i (or total)
            auto next_item = [&](int i, Pair &np) -> int {
                for (int j = i + gridDim.x; j < total; j += gridDim.x) {
                    np = decode_pair(a, j);
                    if (np.vmax > 0) return j;
                }
                return total;
            };
            Pair cur;
            int i = blockIdx.x;
            if (i < total) {
                cur = decode_pair(a, i);
                if (cur.vmax == 0) i = next_item(i, cur);
            }
            while (i < total) {
                Pair nxt;
                const int inext = next_item(i, nxt);
                if (qi == ai) {
                    wait_bar(b_empty + (qi & 1), ((qi >> 1) & 1) ^ 1, abort_flag, err, 1);
                    load_q(cur);
                }
                const int nt = (cur.vmax + NKEY - 1) / NKEY;
                for (int t = 0; t < nt; t++)
                    for (int kh = 0; kh < 2; kh++) {
                        if (qi == ai + 1 && inext < total && mbar_test(b_empty + (qi & 1), ((qi >> 1) & 1) ^ 1))
                            load_q(nxt);
                        const int st = hs % R_ASTG;
                        wait_bar(a_empty + st, ((hs / R_ASTG) & 1) ^ 1, abort_flag, err, 2);
                        mbar_expect_tx(a_full + st, HALF);
                        if (sbhd)
                            tma_load_3d(sA + st * HALF, &map_k, a_full + st, kh * 64, cur.sg.b, t * NKEY);
                        else
                            tma_load_2d(sA + st * HALF, &map_k, a_full + st, kh * 64, (int)(cur.sg.key_y + t * NKEY));
                        last_hs[st] = hs;
                        hs++;
                    }
                ai++;
                i = inext;
                cur = nxt;
            }
            for (int st = 0; st < R_ASTG; st++)
                if (last_hs[st] >= 0) drain_bar(a_full + st, (last_hs[st] / R_ASTG) & 1, err);
            for (int bb = 0; bb < 2; bb++)
                if (last_q[bb] >= 0) drain_bar(b_full + bb, (last_q[bb] >> 1) & 1, err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA issue (whole warp)
        // The warp runs the loop together so stage indices and descriptors stay warp-uniform; one elected lane
        // issues each MMA and commit.  Item decoding is lane-parallel: lane l decodes the CTA's item k + l, the
        // loop reads the tile count of item k by a shuffle.  A half-stage ring: tile t takes stages
        // (st, st + 1), parity aph (R_ASTG is even).  The next group's barriers are probed together and early
        // (mbar_test); a probe that comes back false falls back to the bounded waits.
        //   X^T[(row,h), key] = q . k^T   (A = the item's q tile, B = the k tile, both K-major)
        //   dQ'[(row,h), d]  += G'^T k    (A = G'^T from TMEM, B = the same k tile read MN-major)
        // The dQ' group of a tile is issued two tiles behind its X^T (three X / G' slots), so the epilogue's
        // X -> G' latency is covered by two X^T groups of tensor work.
        int st = 0, ai = 0, dqc = 0, k = 0, nt_lane = 0;
        int xb = 0, gb = 0;              // X slot of the next X^T group / of the next dQ' group
        uint32_t aph = 0, xph = 0, gph = 0;
        int sd = 0;                      // k-tile stage of the next dQ' group (dQ' groups follow the X order)
        bool x_ready = false;
        auto probe_x = [&]() -> bool {
            const bool r0 = mbar_test(x_empty + xb, xph ^ 1);
            const bool r1 = mbar_test(a_full + st, aph);
            const bool r2 = mbar_test(a_full + st + 1, aph);
            return r0 && r1 && r2;
        };
        auto mma2 = [&](bool first) {
            if (first) wait_bar(dq_empty, (dqc & 1) ^ 1, abort_flag, err, 3);
            wait_bar(g_full + gb, gph, abort_flag, err, 4);
            x_ready = probe_x();  // the next X group (this item's next tile or the next item's first)
            fence_after();
            const int sp = sd;
            sd = sd + 2 == R_ASTG ? 0 : sd + 2;
            const unsigned char *pk = sA + sp * HALF;
            const uint32_t tg = tX + gb * 128;
#pragma unroll
            for (int s = 0; s < 8; s++)
                mma_bf16_ts_w(tDQ, tg + (s >> 1) * 32 + (s & 1) * 8, desc_sw128(pk + s * 2048, HALF, 1024), IDESC_DQ,
                              (first && s == 0) ? 0u : 1u);
            mma_commit_w(x_empty + gb);
            mma_commit_w(a_empty + sp);
            mma_commit_w(a_empty + sp + 1);
            if (++gb == R_XSTG) {
                gb = 0;
                gph ^= 1u;
            }
        };
        for (int i = blockIdx.x; i < total; i += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int il = i + lane * (int)gridDim.x;
                nt_lane = il < total ? (decode_pair(a, il).vmax + NKEY - 1) / NKEY : 0;
            }
            const int nt = __shfl_sync(0xffffffffu, nt_lane, k & 31);
            if (nt == 0) continue;
            const int bb = ai & 1;
            wait_bar(b_full + bb, (ai >> 1) & 1, abort_flag, err, 5);
            fence_after();
            const unsigned char *pq = sB + bb * QBLK;
            for (int t = 0; t < nt; t++) {
                if (!x_ready) x_ready = probe_x();
                if (!x_ready) {
                    wait_bar(x_empty + xb, xph ^ 1, abort_flag, err, 6);
                    wait_bar(a_full + st, aph, abort_flag, err, 7);
                    wait_bar(a_full + st + 1, aph, abort_flag, err, 7);
                }
                x_ready = false;
                fence_after();
                const unsigned char *pk = sA + st * HALF;
#pragma unroll
                for (int kh = 0; kh < 2; kh++)
#pragma unroll
                    for (int k4 = 0; k4 < 4; k4++)
                        mma_bf16_w(tX + xb * 128, desc_kmajor(pq + kh * HALF + k4 * 32),
                                   desc_kmajor(pk + kh * HALF + k4 * 32), IDESC_X, (kh | k4) ? 1u : 0u);
                mma_commit_w(x_full + xb);
                if (++xb == R_XSTG) {
                    xb = 0;
                    xph ^= 1u;
                }
                st += 2;
                if (st == R_ASTG) {
                    st = 0;
                    aph ^= 1u;
                }
                if (t >= 2) mma2(t == 2);
            }
            for (int t = nt < 2 ? 0 : nt - 2; t < nt; t++) mma2(t == 0);
            mma_commit_w(dq_full);
            dqc++;
            ai++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------------- g / w stagers
        // Warp 2 prepares the even items (buffer 0), warp 3 the odd ones (buffer 1).  Every global load of a
        // row is issued before any is used, then scattered into the dense per-row g buffer of the item.
        const int me = warp - 2;
        int ic = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            if ((ic & 1) != me) continue;
            const Pair p = decode_pair(a, i);
            const int gb = ic & 1;
            wait_bar(gd_empty + gb, ((ic >> 1) & 1) ^ 1, abort_flag, err, 8);
            float *gd = sGD + gb * RP * NCMAX;
            for (int j4 = lane; j4 * 4 < p.vmax; j4 += 32) {
                reinterpret_cast<float4 *>(gd)[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(gd + NCMAX)[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            float wv[RP][2];
#pragma unroll
            for (int r = 0; r < RP; r++) {
                const long long row = r == 0 ? p.row0 : p.row1;
                wv[r][0] = (r < p.n) ? __ldg(a.w + row * HI + lane) : 0.f;
                wv[r][1] = (r < p.n) ? __ldg(a.w + row * HI + lane + 32) : 0.f;
            }
            __syncwarp();
            constexpr int CHUNK = 8;   // slots per lane per pass
            const int span = g.sparse ? g.K : p.vmax;
            for (int base = 0; base < span; base += 32 * CHUNK) {
                int32_t idv[RP][CHUNK];
                float gv[RP][CHUNK];
#pragma unroll
                for (int r = 0; r < RP; r++) {
                    const int v = r == 0 ? p.v0 : p.v1;
                    const long long row = r == 0 ? p.row0 : p.row1;
#pragma unroll
                    for (int c = 0; c < CHUNK; c++) {
                        const int s = base + c * 32 + lane;
                        const bool ok = v > 0 && s < (g.sparse ? g.K : v);
                        idv[r][c] = ok ? (g.sparse ? __ldg(a.ids + row * g.K + s) : s) : -1;
                        gv[r][c] = ok ? __ldg(a.gbuf + row * g.TW + s) : 0.f;
                    }
                }
#pragma unroll
                for (int r = 0; r < RP; r++) {
                    const int v = r == 0 ? p.v0 : p.v1;
#pragma unroll
                    for (int c = 0; c < CHUNK; c++) {
                        if (idv[r][c] < 0) continue;
                        const long long j = g.sparse ? (long long)idv[r][c] - p.sg.gid0 : idv[r][c];
                        if (j >= 0 && j < v) gd[r * NCMAX + j] = gv[r][c];
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < RP; r++) {
                sW[gb * RP * HI + r * HI + lane] = wv[r][0];
                sW[gb * RP * HI + r * HI + lane + 32] = wv[r][1];
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(gd_full + gb);
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue (16 warps)
        // Lane (quad*32 + lane) = (row, head).  Warp qq = (warp - 4) / 4 of a quadrant owns key columns
        // [32 qq, 32 qq + 32) of every tile and the d quarter [32 qq, 32 qq + 32) of the dQ' readout.
        const int quad = warp & 3, qq = (warp - 4) >> 2;
        const int rh = quad * 32 + lane;
        const int er = rh >> 6, h = rh & 63;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int xb = 0, dqc = 0, ai = 0, ic = 0;
        uint32_t xph = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            const Pair p = decode_pair(a, i);
            const int gb = ic & 1;
            wait_bar(gd_full + gb, (ic >> 1) & 1, abort_flag, err, 9);
            const float *gd = sGD + gb * RP * NCMAX + er * NCMAX;
            const int v_me = er == 0 ? p.v0 : p.v1;
            const int nt = (p.vmax + NKEY - 1) / NKEY;
            for (int t = 0; t < nt; t++) {
                wait_bar(x_full + xb, xph, abort_flag, err, 10);
                fence_after();
                const int j0 = t * NKEY + qq * 32;  // first key of this warp's columns
                uint32_t xr[32];
                const uint32_t tcol = tX + lane_off + (uint32_t)(xb * 128 + qq * 32);
                tmem_ld32_async(tcol, xr);
                // g of the row for these 32 keys (the same addresses across the warp: broadcast reads), fetched
                // while the TMEM load is in flight; keys at or beyond the row's visible count give 0
                float gk[32];
#pragma unroll
                for (int q4 = 0; q4 < 8; q4++) {
                    const int j = j0 + 4 * q4;
                    const float4 g4 = *reinterpret_cast<const float4 *>(gd + j);
                    gk[4 * q4] = j < v_me ? g4.x : 0.f;
                    gk[4 * q4 + 1] = j + 1 < v_me ? g4.y : 0.f;
                    gk[4 * q4 + 2] = j + 2 < v_me ? g4.z : 0.f;
                    gk[4 * q4 + 3] = j + 3 < v_me ? g4.w : 0.f;
                }
                tmem_wait_ld(xr);
                uint32_t pk[16];
#pragma unroll
                for (int q2 = 0; q2 < 16; q2++)
                    pk[q2] = pack_bf16(__uint_as_float(xr[2 * q2]) > 0.f ? gk[2 * q2] : 0.f,
                                       __uint_as_float(xr[2 * q2 + 1]) > 0.f ? gk[2 * q2 + 1] : 0.f);
                tmem_st16(tcol, pk);  // G' over this warp's own X columns (already read)
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(g_full + xb);
                if (++xb == R_XSTG) {
                    xb = 0;
                    xph ^= 1u;
                }
            }
            // ---- dQ' readout: this warp's 32 of the 128 d of its (row, head)
            const bool exists = er < p.n;
            const long long row = er == 0 ? p.row0 : p.row1;
            float pa[4] = {0.f, 0.f, 0.f, 0.f};
            if (nt > 0) {
                const int bb = ai & 1;
                wait_bar(dq_full, dqc & 1, abort_flag, err, 12);
                fence_after();
                uint32_t vr[32];
                tmem_ld32_async(tDQ + lane_off + (uint32_t)(qq * 32), vr);
                // q_idx[row, h, 32 qq .. +32] from the q tile (K-major, 128-B swizzle: K-half qq / 2, 16-B chunks
                // 4 (qq % 2) .. +4 of the row)
                const unsigned char *qb = sB + bb * QBLK + (qq >> 1) * HALF;
                uint4 qv[4];
#pragma unroll
                for (int c = 0; c < 4; c++) qv[c] = *reinterpret_cast<const uint4 *>(qb + sw128_off(rh, (qq & 1) * 4 + c));
                tmem_wait_ld(vr);
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(dq_empty);
                dqc++;
                const float wv = sW[gb * RP * HI + er * HI + h];
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const __nv_bfloat162 *q2 = reinterpret_cast<const __nv_bfloat162 *>(&qv[c]);
#pragma unroll
                    for (int u = 0; u < 4; u++) {
                        const float2 qf = __bfloat1622float2(q2[u]);
                        pa[(2 * u) & 3] = fmaf(qf.x, __uint_as_float(vr[c * 8 + 2 * u]), pa[(2 * u) & 3]);
                        pa[(2 * u + 1) & 3] = fmaf(qf.y, __uint_as_float(vr[c * 8 + 2 * u + 1]), pa[(2 * u + 1) & 3]);
                    }
                }
                if (exists) {
                    __nv_bfloat16 *out = a.dq + row * (HI * DI) + h * DI + qq * 32;
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        uint4 o;
                        o.x = pack_bf16(wv * __uint_as_float(vr[c * 8 + 0]), wv * __uint_as_float(vr[c * 8 + 1]));
                        o.y = pack_bf16(wv * __uint_as_float(vr[c * 8 + 2]), wv * __uint_as_float(vr[c * 8 + 3]));
                        o.z = pack_bf16(wv * __uint_as_float(vr[c * 8 + 4]), wv * __uint_as_float(vr[c * 8 + 5]));
                        o.w = pack_bf16(wv * __uint_as_float(vr[c * 8 + 6]), wv * __uint_as_float(vr[c * 8 + 7]));
                        *reinterpret_cast<uint4 *>(out + c * 8) = o;
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(b_empty + bb);  // q tile no longer read
                ai++;
            } else if (exists) {
                __nv_bfloat16 *out = a.dq + row * (HI * DI) + h * DI + qq * 32;
                for (int c = 0; c < 4; c++) *reinterpret_cast<uint4 *>(out + c * 8) = make_uint4(0, 0, 0, 0);
            }
            // dW = q . dQ' over the four d quarters, summed in a fixed order (sDW alternates by item parity, so
            // one barrier per item suffices)
            float *dwb = sDW + (ic & 1) * 4 * M_PAIRS;
            dwb[qq * M_PAIRS + rh] = (pa[0] + pa[1]) + (pa[2] + pa[3]);
            named_bar(1, R_EPI);
            if (qq == 0 && exists)
                a.dw[row * HI + h] = (dwb[rh] + dwb[M_PAIRS + rh]) + (dwb[2 * M_PAIRS + rh] + dwb[3 * M_PAIRS + rh]);
            __syncwarp();
            if (lane == 0) mbar_arrive(gd_empty + gb);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ key-owner kernel: dK

__global__ void __launch_bounds__(THREADS, 1)
dk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *sA = smem + K_OFF_A;
    unsigned char *sB = smem + K_OFF_B;
    float *sGT = reinterpret_cast<float *>(smem + K_OFF_GT);
    float *sWT = reinterpret_cast<float *>(smem + K_OFF_WT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + K_OFF_MISC);
    uint64_t *a_full = bars, *a_empty = bars + 1, *b_full = bars + 2, *b_empty = b_full + K_BSTG;
    uint64_t *x_full = b_empty + K_BSTG, *x_empty = x_full + 2, *gk_full = x_full + 4, *gk_empty = x_full + 6;
    uint64_t *dk_full = x_full + 8, *dk_empty = x_full + 9, *gt_full = x_full + 10, *gt_empty = gt_full + K_GSTG;
    uint64_t *mma_done = gt_empty + K_GSTG;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + K_OFF_MISC + 256);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + K_OFF_MISC + 264);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    const bool sbhd = g.layout == CSA_SBHD;
    int *err = &g_bwd_error;

    if (threadIdx.x == 0) {
        mbar_init(a_full, 1);
        mbar_init(a_empty, 1);
        for (int i = 0; i < K_BSTG; i++) { mbar_init(b_full + i, 1); mbar_init(b_empty + i, 1); }
        for (int i = 0; i < 2; i++) {
            mbar_init(x_full + i, 1);
            mbar_init(x_empty + i, 8);
            mbar_init(gk_full + i, 8);
            mbar_init(gk_empty + i, 1);
        }
        for (int i = 0; i < K_GSTG; i++) { mbar_init(gt_full + i, 1); mbar_init(gt_empty + i, 8); }
        mbar_init(dk_full, 1);
        mbar_init(dk_empty, 8);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: X (2 x 128 fp32 columns), dK (128), G as the A operand of dK (2 x 64 columns of bf16 pairs)
    const uint32_t tX = tmem, tDK = tmem + 256, tG = tmem + 384;
    const int total = unit_total(a);

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ TMA producer
            int uc = 0, qs = 0;
            int last_qs[K_BSTG];
            for (int x = 0; x < K_BSTG; x++) last_qs[x] = -1;
            int last_uc = -1;
            for (int u = blockIdx.x; u < total; u += gridDim.x) {
                const Unit U = decode_unit(a, u);
                if (U.npairs == 0) continue;
                wait_bar(a_empty, (uc & 1) ^ 1, abort_flag, err, 21);
                mbar_expect_tx(a_full, 2 * HALF);
                for (int kh = 0; kh < 2; kh++) {
                    if (sbhd)
                        tma_load_3d(sA + kh * HALF, &map_k, a_full, kh * 64, U.sg.b, U.kt * NKEY);
                    else
                        tma_load_2d(sA + kh * HALF, &map_k, a_full, kh * 64, (int)(U.sg.key_y + U.kt * NKEY));
                }
                last_uc = uc;
                uc++;
                for (int pi = 0; pi < U.npairs; pi++) {
                    const int bs = qs % K_BSTG;
                    wait_bar(b_empty + bs, ((qs / K_BSTG) & 1) ^ 1, abort_flag, err, 22);
                    mbar_expect_tx(b_full + bs, QBLK);
                    const int s0 = U.s_lo + pi * RP;
                    const long long r0 = row_of(g, U.sg.b, s0);
                    const long long r1 = s0 + 1 < U.s_hi ? row_of(g, U.sg.b, s0 + 1) : r0;
                    for (int r = 0; r < RP; r++)
                        for (int kh = 0; kh < 2; kh++)
                            tma_load_3d(sB + bs * QBLK + kh * HALF + r * (HI * 128), &map_q, b_full + bs, kh * 64, 0,
                                        (int)(r == 0 ? r0 : r1));
                    last_qs[bs] = qs;
                    qs++;
                }
            }
            if (last_uc >= 0) drain_bar(a_full, last_uc & 1, err);
            for (int bs = 0; bs < K_BSTG; bs++)
                if (last_qs[bs] >= 0) drain_bar(b_full + bs, (last_qs[bs] / K_BSTG) & 1, err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA issue (whole warp)
        // As in the row-owner kernel: warp-uniform loop, elected issue, lane-parallel unit decoding, early
        // probes of the next group's barriers.  q-block ring position (bs, parity bph).
        int uc = 0, bs = 0, xc = 0, gkc = 0, dkc = 0, k = 0, np_lane = 0;
        uint32_t bph = 0;
        bool x_ready = false, g_ready = false;
        auto probe_x = [&]() -> bool {
            const bool r0 = mbar_test(x_empty + (xc & 1), ((xc >> 1) & 1) ^ 1);
            const bool r1 = mbar_test(b_full + bs, bph);
            return r0 && r1;
        };
        auto mma3 = [&](int bp, bool first) {
            if (first) wait_bar(dk_empty, (dkc & 1) ^ 1, abort_flag, err, 23);
            const int gkb = gkc & 1;
            if (!g_ready) wait_bar(gk_full + gkb, (gkc >> 1) & 1, abort_flag, err, 24);
            x_ready = probe_x();
            fence_after();
            const unsigned char *pq = sB + bp * QBLK;
#pragma unroll
            for (int s = 0; s < 8; s++)
                mma_bf16_ts_w(tDK, tG + gkb * 64 + s * 8, desc_sw128(pq + s * 2048, HALF, 1024), IDESC_DK,
                              (first && s == 0) ? 0u : 1u);
            mma_commit_w(gk_empty + gkb);
            mma_commit_w(b_empty + bp);
            gkc++;
        };
        for (int u = blockIdx.x; u < total; u += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int ul = u + lane * (int)gridDim.x;
                np_lane = ul < total ? decode_unit(a, ul).npairs : 0;
            }
            const int npairs = __shfl_sync(0xffffffffu, np_lane, k & 31);
            if (npairs == 0) continue;
            wait_bar(a_full, uc & 1, abort_flag, err, 25);
            fence_after();
            int bs_prev = 0;
            for (int pi = 0; pi < npairs; pi++) {
                const int tb = xc & 1;
                if (!x_ready) x_ready = probe_x();
                if (!x_ready) {
                    wait_bar(x_empty + tb, ((xc >> 1) & 1) ^ 1, abort_flag, err, 26);
                    wait_bar(b_full + bs, bph, abort_flag, err, 27);
                }
                x_ready = false;
                g_ready = pi > 0 && mbar_test(gk_full + (gkc & 1), (gkc >> 1) & 1);
                fence_after();
                const unsigned char *pq = sB + bs * QBLK;
#pragma unroll
                for (int kh = 0; kh < 2; kh++)
#pragma unroll
                    for (int k4 = 0; k4 < 4; k4++)
                        mma_bf16_w(tX + tb * 128, desc_kmajor(sA + kh * HALF + k4 * 32), desc_kmajor(pq + kh * HALF + k4 * 32),
                                   IDESC_X, (kh | k4) ? 1u : 0u);
                mma_commit_w(x_full + tb);
                xc++;
                const int bs_cur = bs;
                if (++bs == K_BSTG) {
                    bs = 0;
                    bph ^= 1u;
                }
                if (pi > 0) mma3(bs_prev, pi == 1);
                bs_prev = bs_cur;
            }
            g_ready = false;
            mma3(bs_prev, npairs == 1);
            mma_commit_w(dk_full);
            mma_commit_w(a_empty);
            dkc++;
            uc++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------------- g / w stagers (per row pair)
        // Two warps take alternate row pairs; each issues all loads of a pair before using them.
        const int me = warp - 2;
        int pc = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u);
            const long long key_lo = U.sg.gid0 + (long long)U.kt * NKEY;
            for (int pi = 0; pi < U.npairs; pi++, pc++) {
                if ((pc & 1) != me) continue;
                const int gs = pc % K_GSTG;
                wait_bar(gt_empty + gs, ((pc / K_GSTG) & 1) ^ 1, abort_flag, err, 28);
                float *gt = sGT + gs * RP * NKEY;
                float *wt = sWT + gs * RP * HI;
                long long row[RP];
                bool ok[RP];
                int v[RP];
                int t0[RP], t1[RP];
                float wv[RP][2];
#pragma unroll
                for (int r = 0; r < RP; r++) {
                    const int s = U.s_lo + pi * RP + r;
                    ok[r] = s < U.s_hi;
                    row[r] = row_of(g, U.sg.b, ok[r] ? s : U.s_lo);
                    v[r] = ok[r] ? vis(g, U.sg, s) : 0;
                    wv[r][0] = ok[r] ? __ldg(a.w + row[r] * HI + lane) : 0.f;
                    wv[r][1] = ok[r] ? __ldg(a.w + row[r] * HI + lane + 32) : 0.f;
                    t0[r] = (ok[r] && g.sparse) ? __ldg(a.toff + row[r] * (a.NT + 1) + U.kt) : 0;
                    t1[r] = (ok[r] && g.sparse) ? __ldg(a.toff + row[r] * (a.NT + 1) + U.kt + 1) : 0;
                }
#pragma unroll
                for (int x = 0; x < RP * NKEY / 32; x++) gt[x * 32 + lane] = 0.f;
                int32_t idv[RP][4];
                float gv[RP][4];
#pragma unroll
                for (int r = 0; r < RP; r++)
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        if (g.sparse) {
                            const int sl = t0[r] + c * 32 + lane;
                            const bool in = ok[r] && sl < t1[r];
                            idv[r][c] = in ? __ldg(a.ids + row[r] * g.K + sl) : -1;
                            gv[r][c] = in ? __ldg(a.gbuf + row[r] * g.TW + sl) : 0.f;
                        } else {
                            const int j = U.kt * NKEY + c * 32 + lane;
                            const bool in = ok[r] && j < v[r];
                            idv[r][c] = in ? j : -1;
                            gv[r][c] = in ? __ldg(a.gbuf + row[r] * g.TW + j) : 0.f;
                        }
                    }
                __syncwarp();
#pragma unroll
                for (int r = 0; r < RP; r++) {
                    wt[r * HI + lane] = wv[r][0];
                    wt[r * HI + lane + 32] = wv[r][1];
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        if (idv[r][c] < 0) continue;
                        long long kk, j;
                        if (g.sparse) {
                            kk = (long long)idv[r][c] - key_lo;
                            j = kk + (long long)U.kt * NKEY;
                        } else {
                            j = idv[r][c];
                            kk = j - (long long)U.kt * NKEY;
                        }
                        if (kk >= 0 && kk < NKEY && j < v[r]) gt[r * NKEY + kk] = gv[r][c];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gt_full + gs);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        const int e = warp - 4, quad = warp & 3, half = e >> 2;
        const int k = quad * 32 + lane;
        int xc = 0, gkc = 0, dkc = 0, pc = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u);
            for (int pi = 0; pi < U.npairs; pi++, pc++) {
                const int gs = pc % K_GSTG;
                const int tb = xc & 1;
                wait_bar(gt_full + gs, (pc / K_GSTG) & 1, abort_flag, err, 29);
                wait_bar(x_full + tb, (xc >> 1) & 1, abort_flag, err, 30);
                fence_after();
                const float gk = sGT[gs * RP * NKEY + half * NKEY + k];
                const float *wr = sWT + gs * RP * HI + half * HI;
                uint32_t pk[32];
#pragma unroll
                for (int c = 0; c < 2; c++) {
                    float x[32];
                    tmem_ld32(tX + ((uint32_t)(quad * 32) << 16) + (uint32_t)(tb * 128 + half * 64 + c * 32), x);
#pragma unroll
                    for (int q2 = 0; q2 < 16; q2++) {
                        const int hh = c * 32 + 2 * q2;
                        pk[c * 16 + q2] = pack_bf16(x[2 * q2] > 0.f ? gk * wr[hh] : 0.f,
                                                    x[2 * q2 + 1] > 0.f ? gk * wr[hh + 1] : 0.f);
                    }
                }
                fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(x_empty + tb);
                    mbar_arrive(gt_empty + gs);
                }
                const int gkb = gkc & 1;
                wait_bar(gk_empty + gkb, ((gkc >> 1) & 1) ^ 1, abort_flag, err, 31);
                fence_after();
                // G[key, (row, h)] of this warp's row half: K = (row, h) pairs, columns 32 half .. +32 of buffer gkb
                tmem_st32(tG + ((uint32_t)(quad * 32) << 16) + (uint32_t)(gkb * 64 + half * 32), pk);
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gk_full + gkb);
                xc++;
                gkc++;
            }
            if (U.npairs == 0) continue;
            // ---- flush the unit's dK partial: lane = key, this warp's 64 of the 128 d
            wait_bar(dk_full, dkc & 1, abort_flag, err, 32);
            fence_after();
            float vv[64];
            {
                float x[32];
                tmem_ld32(tDK + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 64), x);
#pragma unroll
                for (int c = 0; c < 32; c++) vv[c] = x[c];
                tmem_ld32(tDK + ((uint32_t)(quad * 32) << 16) + (uint32_t)(half * 64 + 32), x);
#pragma unroll
                for (int c = 0; c < 32; c++) vv[32 + c] = x[c];
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dk_empty);
            dkc++;
            const int j = U.kt * NKEY + k;
            if (j < U.sg.nc) {
                const long long gid = U.sg.gid0 + j;
                const long long kr = g.layout == CSA_SBHD ? (gid % g.nc) * g.B + gid / g.nc : gid;
                float *dst = a.dk_acc + kr * DI + half * 64;
#pragma unroll
                for (int c = 0; c < 16; c++)
                    atomicAdd(reinterpret_cast<float4 *>(dst + 4 * c),
                              make_float4(vv[4 * c], vv[4 * c + 1], vv[4 * c + 2], vv[4 * c + 3]));
            }
        }
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// THD: row-pair items and key-owner units per segment
__global__ void build_bwd_offsets_kernel(Geo g, int *cu_g, int *cu_u)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int ag = 0, au = 0;
    cu_g[0] = 0;
    cu_u[0] = 0;
    for (int b = 0; b < g.B; b++) {
        const int lp = __ldg(g.cu_q + b + 1) - __ldg(g.cu_q + b);
        const int lr = __ldg(g.cu_real + b + 1) - __ldg(g.cu_real + b);
        ag += lp > 0 ? (lp + RP - 1) / RP : 0;
        const long long gid0 = __ldg(g.cu_c + b);
        int nc = lr > 0 ? lr / g.ratio : 0;
        if (nc > g.NC) nc = g.NC;
        if (gid0 + nc > g.key_rows) nc = gid0 < g.key_rows ? (int)(g.key_rows - gid0) : 0;
        au += lr > 0 ? units_of_len(lr, nc, g.ratio) : 0;
        cu_g[b + 1] = ag;
        cu_u[b + 1] = au;
    }
}

}  // namespace bwd

// ------------------------------------------------------------------ host side

bool tc_bwd_supported(const Geo &g, bool bf16)
{
    const char *f = getenv("CSA_FORCE_GENERIC");
    if (f != nullptr && f[0] == '1') return false;
    return bf16 && g.HI == bwd::HI && g.DI == bwd::DI && g.NC >= 1 && g.NC <= bwd::NCMAX && g.K >= 1 &&
           g.rows > 0 && g.key_rows > 0;
}

int tc_bwd_tiles(const Geo &g) { return (g.NC + bwd::NKEY - 1) / bwd::NKEY; }

size_t tc_bwd_workspace_bytes(const Geo &g)
{
    const size_t offs = sizeof(int) * 2 * (size_t)(g.layout == CSA_THD ? g.B + 1 : 1);
    const size_t toff = sizeof(int) * (size_t)g.rows * (size_t)(tc_bwd_tiles(g) + 1);
    return ((offs + 255) & ~(size_t)255) + toff;
}

cudaError_t launch_bwd_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                          const int32_t *ids, const float *gbuf, const int32_t *toff, __nv_bfloat16 *dq, float *dw,
                          float *dk_acc, void *ws, cudaStream_t st)
{
    using namespace bwd;
    CUtensorMap mq, mk;
    if (!tc_encode_q_map(&mq, q_idx, g) || !tc_encode_k_map(&mk, k_idx, g)) return cudaErrorInvalidValue;
    Args a;
    a.g = g;
    a.w = w;
    a.ids = ids;
    a.gbuf = gbuf;
    a.toff = toff;
    a.NT = tc_bwd_tiles(g);
    a.dq = dq;
    a.dw = dw;
    a.dk_acc = dk_acc;
    a.cu_g = a.cu_u = nullptr;
    a.total_items = a.total_units = a.units_per_seq = 0;
    int upper_items, upper_units;
    if (g.layout == CSA_THD) {
        int *cu_g = static_cast<int *>(ws);
        int *cu_u = cu_g + (g.B + 1);
        build_bwd_offsets_kernel<<<1, 32, 0, st>>>(g, cu_g, cu_u);
        note_launches(1);
        a.cu_g = cu_g;
        a.cu_u = cu_u;
        upper_items = (g.rows + RP - 1) / RP + g.B;
        upper_units = (g.rows + CH - 1) / CH * a.NT + g.B * a.NT;
    } else {
        a.total_items = g.B * ((g.S + RP - 1) / RP);
        a.units_per_seq = units_of_len(g.S, g.nc, g.ratio);
        a.total_units = g.B * a.units_per_seq;
        upper_items = a.total_items;
        upper_units = a.total_units;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dq_dw_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, R_SMEM);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, K_SMEM);
    if (e != cudaSuccess) return e;
    const int g1 = upper_items < sms ? (upper_items > 0 ? upper_items : 1) : sms;
    dq_dw_tc_kernel<<<g1, R_THREADS, R_SMEM, st>>>(mq, mk, a);
    note_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (upper_units > 0) {
        const int g2 = upper_units < sms ? upper_units : sms;
        dk_tc_kernel<<<g2, THREADS, K_SMEM, st>>>(mq, mk, a);
        note_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace csa
