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
// kernels stream contiguous tiles by TMA; no per-element global atomics.  On key axes up to 1024 keys g arrives
// by key (the KL step's gd rows, position-major), so a row pair's g over a key tile, its w rows, its q_idx rows
// and a k tile are one TMA copy each.  On longer key axes g stays in the KL step's slot layout ([rows][K], the
// row's ascending ids) and a builder warp assembles each row's 128-key g tile in shared memory: the row-owner's
// walks the row's slots with a cursor, the key-owner's reads the tile's slot range from a per-row table of tile
// offsets (tile_offsets_kernel), so no [rows][keys] array is ever written.
//   * row-owner kernel (dQ_idx, dW): a work item is 2 query rows (M = 128 (row, head) pairs).  Per key tile:
//     MMA1 X^T[(row,h), key] = q . k^T (N 128 keys, K 128) into one of three TMEM slots, the epilogue forms
//     G'^T = g 1[x > 0] in bf16 over its own X columns, and MMA2 accumulates dQ'[(row,h), d] += G'^T k
//     (A from TMEM, B = the k tile read MN-major) over all tiles of the item; the item's dQ' read-out is
//     deferred behind the next item's first two tiles.
//   * key-owner kernel (dK): a unit is one key tile and a chunk of up to 128 rows that see it.  Per row pair:
//     MMA1 X[key, (row,h)] = k . q^T, the epilogue forms G = g w 1[x > 0] in bf16 over its own X columns, and
//     MMA3 accumulates dK[key, d] += G q (A from TMEM, B = the q block read MN-major); the unit flushes its
//     128 x 128 fp32 partial once.  It is launched as a programmatic dependent of the row-owner kernel.
// Roles (both kernels, 20 warps): warp 0 TMA, warp 1 TMEM + the X MMAs, warp 2 the dQ'/dK MMAs, warp 3 the g-tile
// builder on long key axes (idle otherwise), warps 4..19 epilogue.  Waits are bounded as in the score kernel.
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
constexpr int NCMAX = 1024;                    // key axis the row-owner's dense g rows hold (longer: g tiles built)
constexpr int GR = 8;                          // long key axis: row-owner g tiles in flight (2 rows x 128 keys each)
constexpr int HALF = NKEY * 64 * 2;            // 16 KB: 128 rows x 64 bf16
constexpr int QBLK = 2 * HALF;                 // 32 KB: 2 rows x 64 heads x 128 d, two K-halves
constexpr int THREADS = 640;                   // key-owner kernel: 20 warps
constexpr int EPI = 512;                       //   its epilogue: warps 4..19
constexpr int R_THREADS = 640;                 // row-owner kernel: 20 warps
constexpr int R_EPI = 512;                     //   its epilogue: warps 4..19, four per TMEM lane quadrant
constexpr int CH = 128;                        // rows per key-owner unit
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t IDESC_X = idesc_bf16(128, 128, false, false);   // X = k . q^T (key-owner), X^T = q . k^T
constexpr uint32_t IDESC_DQ = idesc_bf16(128, 128, false, true);   // dQ' += G'^T k  (A in TMEM, B MN-major)
constexpr uint32_t IDESC_DK = idesc_bf16(128, 128, false, true);   // dK += G q      (A in TMEM, B MN-major)

// row-owner shared memory
constexpr int R_ASTG = 4;                                     // k tiles in flight
constexpr int R_XSTG = 3;                                     // X / G' TMEM slots
static_assert((2 * R_ASTG + 19 + 3 * R_XSTG + 2 * GR) * 8 <= 512, "row-owner barriers overlap the TMEM slot");
constexpr int KTILE = 2 * HALF;                               // 32 KB: 128 keys x 128 d, two K-halves
constexpr int R_OFF_A = 0;
constexpr int R_OFF_B = R_OFF_A + R_ASTG * KTILE;             // 128 KB: the q tiles of two items
constexpr int R_OFF_GD = R_OFF_B + 2 * QBLK;                  // 192 KB: 2 bufs x key tiles x 2 rows x 128 fp32
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
constexpr int K_OFF_RNG = K_OFF_WT + K_GSTG * RP * HI * 4;      // long key axis: a unit's slot ranges, CH x 2 int
constexpr int K_OFF_MISC = K_OFF_RNG + CH * 2 * 4;
constexpr int K_SMEM = K_OFF_MISC + 1024 + 1024;
constexpr int K_XSTG = 3;                                      // X / G TMEM slots
static_assert((2 + 2 * K_BSTG + 3 * K_XSTG + 2 + 2 * K_GSTG + 1) * 8 <= 256, "key-owner barriers overlap the TMEM slot");

struct Args {
    Geo g;
    __nv_bfloat16 *dq;
    float *dw;
    float *dk_acc;           // [key rows, DI] fp32, zeroed by the caller
    const int *cu_g;         // THD: row-pair items per segment [nseg+1]
    const int *cu_u;         // THD: key-owner units per segment [nseg+1]
    int total_items, total_units;     // SBHD/BSHD
    int units_per_seq;                // SBHD/BSHD
    // long key axis: g by slot [rows][K], the ids, and per row the first slot of each key tile [rows][NT + 1]
    bool lng;
    const float *gslot;
    const int32_t *ids;
    const int *toff;
    const unsigned long long *sgn;   // signs of x by slot [rows][K], from the gathered row-owner
    int NT;
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
    int s0;                   // position of the first row
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
    p.s0 = s0;
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

// A role visits its units in ascending order, so the walk over a segment's row chunks resumes where the previous
// unit's walk stopped (a cursor per thread); it restarts from chunk 0 when the segment changes or the index goes
// back.  (Walking from chunk 0 for every unit cost each warp ~340 iterations of two integer divisions per unit on
// a 512-chunk sequence.)
struct UnitCursor {
    int b = -1, c = 0, base = 0;  // segment, current chunk, units of the chunks before it
};

__device__ Unit decode_unit(const Args &a, int u, UnitCursor &cur)
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
    if (b != cur.b || lu < cur.base) {
        cur.b = b;
        cur.c = 0;
        cur.base = 0;
    }
    const int nch = (U.sg.len_real + CH - 1) / CH;
    while (cur.c < nch) {
        const int nt = chunk_tiles(cur.c, U.sg.len_real, U.sg.nc, g.ratio);
        if (lu - cur.base < nt) {
            U.kt = lu - cur.base;
            U.s_lo = cur.c * CH;
            U.s_hi = min(U.sg.len_real, U.s_lo + CH);
            break;
        }
        cur.base += nt;
        cur.c++;
    }
    U.npairs = (U.s_hi - U.s_lo + 1) / RP;
    return U;
}

// The slot ranges [lo, hi) of key tile U.kt in the unit's rows, from the tile-offset rows, into sRng[r][2] (clamped to
// [0, K]); every load of the warp is issued before any is used (at most CH = 128 rows: four per lane).
__device__ __forceinline__ void load_ranges(const Args &a, const Unit &U, int nrow, int *sRng, int lane)
{
    static_assert(CH == 128, "four rows per lane");
    const int K = a.g.K;
    int lo[4], hi[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int r = lane + 32 * i;
        lo[i] = hi[i] = 0;
        if (r < nrow) {
            const int *o = a.toff + row_of(a.g, U.sg.b, U.s_lo + r) * (long long)(a.NT + 1);
            lo[i] = __ldg(o + U.kt);
            hi[i] = __ldg(o + U.kt + 1);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const int r = lane + 32 * i;
        if (r < nrow) {
            const int l = lo[i] < 0 ? 0 : (lo[i] > K ? K : lo[i]);
            sRng[2 * r] = l;
            sRng[2 * r + 1] = hi[i] < l ? l : (hi[i] > K ? K : hi[i]);
        }
    }
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

// TMA coordinates of a row pair (positions s0, s0 + 1 of segment b): (y, z) in the pair maps of q_idx and w
// ([.., rows, 1] for BSHD / THD, [.., B, S] for SBHD), and the pair's first row in the position-major g rows.
struct PairAt {
    int y, z, prow;
};
__device__ __forceinline__ PairAt pair_at(const Geo &g, int b, int s0, long long row0)
{
    PairAt q;
    if (g.layout == CSA_SBHD) {
        q.y = b;
        q.z = s0;
        q.prow = b * g.S + s0;
    } else {
        q.y = (int)row0;
        q.z = 0;
        q.prow = (int)row0;
    }
    return q;
}

// ------------------------------------------------------------------ row-owner kernel: dQ_idx, dW

__global__ void __launch_bounds__(R_THREADS, 1)
dq_dw_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
                const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_w, Args a)
{
    // the key-owner kernel reads nothing this one writes: let it take each SM this kernel leaves
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sA = smem + R_OFF_A;
    unsigned char *sB = smem + R_OFF_B;
    float *sGD = reinterpret_cast<float *>(smem + R_OFF_GD);
    float *sW = reinterpret_cast<float *>(smem + R_OFF_W);
    float *sDW = reinterpret_cast<float *>(smem + R_OFF_DW);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + R_OFF_MISC);
    uint64_t *a_full = bars, *a_empty = bars + R_ASTG, *b_full = bars + 2 * R_ASTG, *b_empty = b_full + 2;
    uint64_t *x_full = b_full + 4, *x_empty = x_full + R_XSTG, *g_full = x_empty + R_XSTG;
    uint64_t *dq_full = g_full + R_XSTG, *dq_empty = dq_full + 1, *gd_full = dq_full + 2, *gd_empty = dq_full + 4;
    uint64_t *mma_done = dq_full + 6;                                  // 2 R_ASTG + 19 + 3 R_XSTG barriers
    uint64_t *dw_bar = dq_full + 7;                                    // [item parity][quadrant]: dW partials
    uint64_t *gr_full = dq_full + 15, *gr_empty = gr_full + GR;        // long key axis: built g tiles
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
        mbar_init(mma_done, 2);
        for (int i = 0; i < 8; i++) mbar_init(dw_bar + i, 4);
        for (int i = 0; i < GR; i++) {
            mbar_init(gr_full + i, 1);
            mbar_init(gr_empty + i, R_EPI / 32);
        }
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
            // k tiles stream through a four-tile ring (one copy per tile); an item's q tile (one copy for both
            // rows) is requested as soon as its buffer is free: that buffer is probed before every k-tile load
            // of the previous item, and waited for at the latest when the item starts.
            int hs = 0, ai = 0, qi = 0;
            int last_hs[R_ASTG];
            int last_q[2] = {-1, -1};
            for (int i = 0; i < R_ASTG; i++) last_hs[i] = -1;
            // the item's g rows over its visible key tiles (one copy of both rows per tile) and its w rows, into
            // buffer ai & 1
            // (long key axis: the w rows only; the builder warp assembles the g tiles)
            auto load_gw = [&](const Pair &p, const PairAt &at) {
                const int gb = ai & 1;
                wait_bar(gd_empty + gb, ((ai >> 1) & 1) ^ 1, abort_flag, err, 8);
                const int nt = a.lng ? 0 : (p.vmax + NKEY - 1) / NKEY;
                mbar_expect_tx(gd_full + gb, (uint32_t)(nt * RP * NKEY * 4 + RP * HI * 4));
                for (int kt = 0; kt < nt; kt++)
                    tma_load_2d(sGD + gb * RP * NCMAX + kt * RP * NKEY, &map_g, gd_full + gb, kt * NKEY, at.prow);
                tma_load_3d(sW + gb * RP * HI, &map_w, gd_full + gb, 0, at.y, at.z);
            };
            auto load_q = [&](const PairAt &at) {
                const int bb = qi & 1;
                mbar_expect_tx(b_full + bb, QBLK);
                tma_load_5d(sB + bb * QBLK, &map_q, b_full + bb, 0, 0, at.y, at.z, 0);
                last_q[bb] = qi;
                qi++;
            };
            auto at_of = [&](const Pair &p) { return pair_at(g, p.sg.b, p.s0, p.row0); };
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
                const PairAt at = at_of(cur);
                if (qi == ai) {
                    wait_bar(b_empty + (qi & 1), ((qi >> 1) & 1) ^ 1, abort_flag, err, 1);
                    load_q(at);
                }
                load_gw(cur, at);
                const int nt = (cur.vmax + NKEY - 1) / NKEY;
                for (int t = 0; t < nt; t++) {
                    if (qi == ai + 1 && inext < total && mbar_test(b_empty + (qi & 1), ((qi >> 1) & 1) ^ 1))
                        load_q(at_of(nxt));
                    const int st = hs % R_ASTG;
                    wait_bar(a_empty + st, ((hs / R_ASTG) & 1) ^ 1, abort_flag, err, 2);
                    mbar_expect_tx(a_full + st, KTILE);
                    if (sbhd)
                        tma_load_4d(sA + st * KTILE, &map_k, a_full + st, 0, cur.sg.b, t * NKEY, 0);
                    else
                        tma_load_3d(sA + st * KTILE, &map_k, a_full + st, 0, (int)(cur.sg.key_y + t * NKEY), 0);
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
            for (int gb = 0; gb < 2 && gb < ai; gb++) {
                const int last = ai - 1 - ((ai - 1 - gb) & 1);  // the last item that used buffer gb
                drain_bar(gd_full + gb, (last >> 1) & 1, err);
            }
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------- MMA issue (two warps, whole warp each)
        // Warp 1 issues the X^T groups, warp 2 the dQ' groups; each commits its own groups, so neither waits on
        // the other's issue overhead.  Each warp runs its loop together (stage indices and descriptors stay
        // warp-uniform; one elected lane issues); item decoding is lane-parallel: lane l decodes the CTA's item
        // k + l, the loop reads the tile count of item k by a shuffle.  k-tile stage st, parity aph; X / G' slot
        // xb, parity xph.
        //   X^T[(row,h), key] = q . k^T   (A = the item's q tile, B = the k tile, both K-major)
        //   dQ'[(row,h), d]  += G'^T k    (A = G'^T from TMEM, B = the same k tile read MN-major)
        const bool xw = warp == 1;
        int st = 0, ai = 0, k = 0, nt_lane = 0, xb = 0;
        uint32_t aph = 0, xph = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int il = i + lane * (int)gridDim.x;
                nt_lane = il < total ? (decode_pair(a, il).vmax + NKEY - 1) / NKEY : 0;
            }
            const int nt = __shfl_sync(0xffffffffu, nt_lane, k & 31);
            if (nt == 0) continue;
            const int bb = ai & 1;
            if (xw) {
                wait_bar(b_full + bb, (ai >> 1) & 1, abort_flag, err, 5);
                fence_after();
            }
            const unsigned char *pq = sB + bb * QBLK;
            for (int t = 0; t < nt; t++) {
                const unsigned char *pk = sA + st * KTILE;
                if (xw) {
                    const bool r0 = mbar_test(x_empty + xb, xph ^ 1);
                    const bool r1 = mbar_test(a_full + st, aph);
                    if (!(r0 && r1)) {
                        wait_bar(x_empty + xb, xph ^ 1, abort_flag, err, 6);
                        wait_bar(a_full + st, aph, abort_flag, err, 7);
                    }
                    fence_after();
#pragma unroll
                    for (int kh = 0; kh < 2; kh++)
#pragma unroll
                        for (int k4 = 0; k4 < 4; k4++)
                            mma_bf16_w(tX + xb * 128, desc_kmajor(pq + kh * HALF + k4 * 32),
                                       desc_kmajor(pk + kh * HALF + k4 * 32), IDESC_X, (kh | k4) ? 1u : 0u);
                    mma_commit_w(x_full + xb);
                } else {
                    if (t == 0) wait_bar(dq_empty, (ai & 1) ^ 1, abort_flag, err, 3);
                    wait_bar(g_full + xb, xph, abort_flag, err, 4);
                    fence_after();
                    const uint32_t tg = tX + xb * 128;
#pragma unroll
                    for (int s = 0; s < 8; s++)
                        mma_bf16_ts_w(tDQ, tg + (s >> 1) * 32 + (s & 1) * 8, desc_sw128(pk + s * 2048, HALF, 1024),
                                      IDESC_DQ, (t == 0 && s == 0) ? 0u : 1u);
                    mma_commit_w(x_empty + xb);
                    mma_commit_w(a_empty + st);
                }
                if (++xb == R_XSTG) {
                    xb = 0;
                    xph ^= 1u;
                }
                if (++st == R_ASTG) {
                    st = 0;
                    aph ^= 1u;
                }
            }
            if (!xw) mma_commit_w(dq_full);
            ai++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp == 3 && a.lng) {
        // ---------------------------------------------------------------- g-tile builder (long key axis)
        // Half-warp r builds row r of the item: for each key tile, in order, 128 floats of g by key (zero off the
        // row's selection) from the row's slots, whose ids ascend.  It walks the slots with a cursor over chunks of
        // 16 (chunk A being placed, chunk B loaded ahead); a chunk advances once all its keys lie below the tile's
        // end.  Keys outside the tile or the row's visible range are never placed.
        const int half = lane >> 4, hl = lane & 15;
        const unsigned hmask = 0xffffu << (16 * half);
        const int K = g.K;
        float *sG = sGD;  // [GR][RP][NKEY]
        int tcnt = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Pair p = decode_pair(a, i);
            const int nt = (p.vmax + NKEY - 1) / NKEY;
            if (nt == 0) continue;
            const bool present = half < p.n;
            const long long row = half == 0 ? p.row0 : p.row1;
            const int v_me = half == 0 ? p.v0 : p.v1;
            const int32_t *rid = a.ids + row * K;
            const float *rg = a.gslot + row * K;
            auto load = [&](int sl, int &j, float &gv) {  // key (INT_MAX when unusable) and g of slot sl
                j = 0x7fffffff;
                gv = 0.f;
                if (present && sl < K) {
                    const int32_t id = __ldg(rid + sl);
                    const long long jj = (long long)id - p.sg.gid0;
                    if (id >= 0 && jj >= 0 && jj < v_me) {
                        j = (int)jj;
                        gv = __ldg(rg + sl);
                    }
                }
            };
            int cur = 0, ja, jb;
            float ga, gb_;
            load(hl, ja, ga);
            load(16 + hl, jb, gb_);
            for (int t = 0; t < nt; t++, tcnt++) {
                const int slot = tcnt % GR;
                wait_bar(gr_empty + slot, ((tcnt / GR) & 1) ^ 1, abort_flag, err, 14);
                float *dst = sG + slot * RP * NKEY + half * NKEY;
                reinterpret_cast<float4 *>(dst)[2 * hl] = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(dst)[2 * hl + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                __syncwarp();
                const int t0 = t * NKEY, t1 = t0 + NKEY;
                while (true) {
                    if (ja >= t0 && ja < t1) dst[ja - t0] = ga;
                    const unsigned below = __ballot_sync(0xffffffffu, ja < t1);
                    const bool adv = present && (below & hmask) == hmask;
                    if (!__any_sync(0xffffffffu, adv)) break;
                    if (adv) {
                        ja = jb;
                        ga = gb_;
                        cur += 16;
                        load(cur + 16 + hl, jb, gb_);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gr_full + slot);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue (16 warps)
        // Lane (quad*32 + lane) = (row, head).  Warp qq = (warp - 4) / 4 of a quadrant owns key columns
        // [32 qq, 32 qq + 32) of every tile and the d quarter [32 qq, 32 qq + 32) of the dQ' readout.
        const int quad = warp & 3, qq = (warp - 4) >> 2;
        const int rh = quad * 32 + lane;
        const int er = rh >> 6, h = rh & 63;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        // An item's dQ' read-out is deferred until the next item's first LAG tiles have been converted, so the
        // drain of its last dQ' group overlaps useful work (LAG <= R_XSTG: those tiles' X slots were freed by
        // the previous item's dQ' groups, whose accumulator is the one being read out).
        constexpr int LAG = 2;
        static_assert(LAG <= R_XSTG, "deferred read-out would wait on its own X slots");
        struct Pend {
            long long row;
            int gb, ic;       // g / w / q buffer of the item, item index (dW buffer parity)
            bool tiles, exists, valid;
        };
        int xb = 0, dqc = 0, ai = 0, ic = 0, gcnt = 0;
        uint32_t xph = 0;
        // ---- one key tile: X^T -> G'^T over the warp's own columns
        auto tile = [&](const float *gd, int v_me, int t) {
            wait_bar(x_full + xb, xph, abort_flag, err, 10);
            fence_after();
            const int j0 = t * NKEY + qq * 32;  // first key of this warp's columns
            const float *gt = gd + t * RP * NKEY + qq * 32;
            const int gslot = gcnt % GR;
            if (a.lng) {  // the builder's tile (rows x 128 keys) of this key tile
                wait_bar(gr_full + gslot, (gcnt / GR) & 1, abort_flag, err, 15);
                gt = sGD + gslot * RP * NKEY + er * NKEY + qq * 32;
            }
            uint32_t xr[32];
            const uint32_t tcol = tX + lane_off + (uint32_t)(xb * 128 + qq * 32);
            tmem_ld32_async(tcol, xr);
            // g of the row for these 32 keys (the same addresses across the warp: broadcast reads), fetched
            // while the TMEM load is in flight; keys at or beyond the row's visible count give 0
            float gk[32];
#pragma unroll
            for (int q4 = 0; q4 < 8; q4++) {
                const float4 g4 = *reinterpret_cast<const float4 *>(gt + 4 * q4);
                gk[4 * q4] = g4.x;
                gk[4 * q4 + 1] = g4.y;
                gk[4 * q4 + 2] = g4.z;
                gk[4 * q4 + 3] = g4.w;
            }
            if (a.lng) {
                __syncwarp();
                if (lane == 0) mbar_arrive(gr_empty + gslot);
                gcnt++;
            }
            if (j0 + 32 > v_me) {  // warp-uniform: the row's last visible tile
#pragma unroll
                for (int q = 0; q < 32; q++) gk[q] = j0 + q < v_me ? gk[q] : 0.f;
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
        };
        // ---- an item's end: dQ' read-out (this warp's 32 of the 128 d of its (row, head)), dW, buffer release
        auto finish = [&](const Pend &P) {
            float pa[4] = {0.f, 0.f, 0.f, 0.f};
            if (P.tiles) {
                const int bb = P.gb;
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
                const float wv = sW[P.gb * RP * HI + er * HI + h];
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
                if (P.exists) {
                    __nv_bfloat16 *out = a.dq + P.row * (HI * DI) + h * DI + qq * 32;
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
            } else if (P.exists) {
                __nv_bfloat16 *out = a.dq + P.row * (HI * DI) + h * DI + qq * 32;
                for (int c = 0; c < 4; c++) *reinterpret_cast<uint4 *>(out + c * 8) = make_uint4(0, 0, 0, 0);
            }
            // dW = q . dQ' over the four d quarters, summed in a fixed order (sDW alternates by item parity; the
            // four warps of a quadrant meet on an mbarrier and the d-quarter-0 warp adds and writes)
            float *dwb = sDW + (P.ic & 1) * 4 * M_PAIRS;
            dwb[qq * M_PAIRS + rh] = (pa[0] + pa[1]) + (pa[2] + pa[3]);
            __syncwarp();
            uint64_t *dwq = dw_bar + (P.ic & 1) * 4 + quad;
            if (lane == 0) mbar_arrive(dwq);
            if (qq == 0) {
                wait_bar(dwq, (P.ic >> 1) & 1, abort_flag, err, 13);
                if (P.exists)
                    a.dw[P.row * HI + h] = (dwb[rh] + dwb[M_PAIRS + rh]) + (dwb[2 * M_PAIRS + rh] + dwb[3 * M_PAIRS + rh]);
            }
            __syncwarp();
            if (P.tiles && lane == 0) mbar_arrive(gd_empty + P.gb);
        };
        Pend pend;
        pend.valid = false;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            const Pair p = decode_pair(a, i);
            const int nt = (p.vmax + NKEY - 1) / NKEY;
            Pend cur;
            cur.row = er == 0 ? p.row0 : p.row1;
            cur.exists = er < p.n;
            cur.ic = ic;
            cur.tiles = nt > 0;
            cur.gb = ai & 1;  // g / w buffer of the items with visible keys (as the producer counts them)
            cur.valid = true;
            if (nt == 0) {
                if (pend.valid) finish(pend);
                pend.valid = false;
                finish(cur);
                continue;
            }
            wait_bar(gd_full + cur.gb, (ai >> 1) & 1, abort_flag, err, 9);
            const float *gd = sGD + cur.gb * RP * NCMAX + er * NKEY;  // [key tile][row][128]
            const int v_me = er == 0 ? p.v0 : p.v1;
            for (int t = 0; t < nt; t++) {
                tile(gd, v_me, t);
                if (t == LAG - 1 && pend.valid) {
                    finish(pend);
                    pend.valid = false;
                }
            }
            if (pend.valid) finish(pend);
            pend = cur;
            ai++;
        }
        if (pend.valid) finish(pend);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ key-owner kernel: dK

__global__ void __launch_bounds__(THREADS, 1)
dk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k,
             const __grid_constant__ CUtensorMap map_g, const __grid_constant__ CUtensorMap map_w, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sA = smem + K_OFF_A;
    unsigned char *sB = smem + K_OFF_B;
    float *sGT = reinterpret_cast<float *>(smem + K_OFF_GT);
    float *sWT = reinterpret_cast<float *>(smem + K_OFF_WT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + K_OFF_MISC);
    uint64_t *a_full = bars, *a_empty = bars + 1, *b_full = bars + 2, *b_empty = b_full + K_BSTG;
    uint64_t *x_full = b_empty + K_BSTG, *x_empty = x_full + K_XSTG, *gk_full = x_empty + K_XSTG;
    uint64_t *dk_full = gk_full + K_XSTG, *dk_empty = dk_full + 1, *gt_full = dk_full + 2, *gt_empty = gt_full + K_GSTG;
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
        for (int i = 0; i < K_XSTG; i++) {
            mbar_init(x_full + i, 1);
            mbar_init(x_empty + i, 1);
            mbar_init(gk_full + i, EPI / 32);
        }
        // long key axis: a g/w slot is full once the w copy has landed and the builder has written the g tile
        for (int i = 0; i < K_GSTG; i++) { mbar_init(gt_full + i, a.lng ? 2 : 1); mbar_init(gt_empty + i, EPI / 32); }
        mbar_init(dk_full, 1);
        mbar_init(dk_empty, EPI / 32);
        mbar_init(mma_done, 2);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: three slots of 128 columns, each holding one row pair's X (fp32) and then, in place, its G as the A
    // operand of dK (bf16 pairs; the epilogue warp of X columns [32 c, 32 c + 32) writes its 16 pair columns over
    // the first half of them, so the pairs of K indices [16 s, 16 s + 16) sit at column 32 (s / 2) + 8 (s % 2));
    // dK (128).
    const uint32_t tX = tmem, tDK = tmem + K_XSTG * 128;
    const int total = unit_total(a);

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ TMA producer
            int uc = 0, qs = 0;
            int last_qs[K_BSTG];
            for (int x = 0; x < K_BSTG; x++) last_qs[x] = -1;
            int last_uc = -1;
            UnitCursor cur;
            for (int u = blockIdx.x; u < total; u += gridDim.x) {
                const Unit U = decode_unit(a, u, cur);
                if (U.npairs == 0) continue;
                wait_bar(a_empty, (uc & 1) ^ 1, abort_flag, err, 21);
                mbar_expect_tx(a_full, KTILE);
                if (sbhd)
                    tma_load_4d(sA, &map_k, a_full, 0, U.sg.b, U.kt * NKEY, 0);
                else
                    tma_load_3d(sA, &map_k, a_full, 0, (int)(U.sg.key_y + U.kt * NKEY), 0);
                last_uc = uc;
                uc++;
                for (int pi = 0; pi < U.npairs; pi++) {
                    const int bs = qs % K_BSTG;
                    wait_bar(b_empty + bs, ((qs / K_BSTG) & 1) ^ 1, abort_flag, err, 22);
                    mbar_expect_tx(b_full + bs, QBLK);
                    // one copy each: the pair's q rows, its g over this key tile, its w rows (a second row past the
                    // chunk's end is read but never used)
                    const int s0 = U.s_lo + pi * RP;
                    const PairAt at = pair_at(g, U.sg.b, s0, row_of(g, U.sg.b, s0));
                    tma_load_5d(sB + bs * QBLK, &map_q, b_full + bs, 0, 0, at.y, at.z, 0);
                    last_qs[bs] = qs;
                    const int gs = qs % K_GSTG;
                    wait_bar(gt_empty + gs, ((qs / K_GSTG) & 1) ^ 1, abort_flag, err, 28);
                    mbar_expect_tx(gt_full + gs, (uint32_t)(RP * ((a.lng ? 0 : NKEY) + HI) * 4));
                    if (!a.lng) tma_load_2d(sGT + gs * RP * NKEY, &map_g, gt_full + gs, U.kt * NKEY, at.prow);
                    tma_load_3d(sWT + gs * RP * HI, &map_w, gt_full + gs, 0, at.y, at.z);
                    qs++;
                }
            }
            if (last_uc >= 0) drain_bar(a_full, last_uc & 1, err);
            for (int q = qs - K_GSTG < 0 ? 0 : qs - K_GSTG; q < qs; q++) drain_bar(gt_full + q % K_GSTG, (q / K_GSTG) & 1, err);
            for (int bs = 0; bs < K_BSTG; bs++)
                if (last_qs[bs] >= 0) drain_bar(b_full + bs, (last_qs[bs] / K_BSTG) & 1, err);
        }
    } else if (warp == 1 || warp == 2) {
        // ------------------------------------------------------------- MMA issue (two warps, whole warp each)
        // Warp 1 issues the X groups, warp 2 the dK groups; each commits its own groups, so neither waits on
        // the other's issue overhead.  Each warp runs its loop together (stage indices and descriptors stay
        // warp-uniform; one elected lane issues); unit decoding is lane-parallel: lane l decodes the CTA's unit
        // k + l, the loop reads the pair count of unit k by a shuffle.
        //   X[key, (row,h)]  = k . q^T    (A = the unit's key tile, B = the q block, both K-major)
        //   dK[key, d]      += G q        (A = G from TMEM, B = the same q block read MN-major)
        const bool xw = warp == 1;
        int uc = 0, bs = 0, k = 0, np_lane = 0, xb = 0;
        uint32_t bph = 0, xph = 0;
        UnitCursor lcur;  // lane l decodes units u + l * gridDim.x, ascending across refills
        for (int u = blockIdx.x; u < total; u += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int ul = u + lane * (int)gridDim.x;
                np_lane = ul < total ? decode_unit(a, ul, lcur).npairs : 0;
            }
            const int npairs = __shfl_sync(0xffffffffu, np_lane, k & 31);
            if (npairs == 0) continue;
            if (xw) {
                wait_bar(a_full, uc & 1, abort_flag, err, 25);
                fence_after();
            }
            for (int pi = 0; pi < npairs; pi++) {
                const unsigned char *pq = sB + bs * QBLK;
                if (xw) {
                    const bool r0 = mbar_test(x_empty + xb, xph ^ 1);
                    const bool r1 = mbar_test(b_full + bs, bph);
                    if (!(r0 && r1)) {
                        wait_bar(x_empty + xb, xph ^ 1, abort_flag, err, 26);
                        wait_bar(b_full + bs, bph, abort_flag, err, 27);
                    }
                    fence_after();
#pragma unroll
                    for (int kh = 0; kh < 2; kh++)
#pragma unroll
                        for (int k4 = 0; k4 < 4; k4++)
                            mma_bf16_w(tX + xb * 128, desc_kmajor(sA + kh * HALF + k4 * 32),
                                       desc_kmajor(pq + kh * HALF + k4 * 32), IDESC_X, (kh | k4) ? 1u : 0u);
                    mma_commit_w(x_full + xb);
                    if (pi == npairs - 1) mma_commit_w(a_empty);  // the key tile is read by the X groups only
                } else {
                    if (pi == 0) wait_bar(dk_empty, (uc & 1) ^ 1, abort_flag, err, 23);
                    wait_bar(gk_full + xb, xph, abort_flag, err, 24);
                    fence_after();
                    const uint32_t tg = tX + xb * 128;
#pragma unroll
                    for (int s = 0; s < 8; s++)
                        mma_bf16_ts_w(tDK, tg + (s >> 1) * 32 + (s & 1) * 8, desc_sw128(pq + s * 2048, HALF, 1024),
                                      IDESC_DK, (pi == 0 && s == 0) ? 0u : 1u);
                    mma_commit_w(x_empty + xb);
                    mma_commit_w(b_empty + bs);
                }
                if (++xb == K_XSTG) {
                    xb = 0;
                    xph ^= 1u;
                }
                if (++bs == K_BSTG) {
                    bs = 0;
                    bph ^= 1u;
                }
            }
            if (!xw) mma_commit_w(dk_full);
            uc++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp == 3 && a.lng) {
        // ---------------------------------------------------------------- g-tile builder (long key axis)
        // Per unit: the slot range [lo, hi) of the unit's key tile in each of its rows, from the tile-offset rows;
        // then per row pair, into the pair's g/w slot: half-warp r zeroes row r's 128 keys and places the g of its
        // slots lo .. hi - 1 (keys outside the tile are never placed).
        const int half = lane >> 4, hl = lane & 15;
        const int K = g.K;
        int *sRng = reinterpret_cast<int *>(smem + K_OFF_RNG);  // [CH][2]
        int pc = 0;
        UnitCursor cur;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u, cur);
            if (U.npairs == 0) continue;
            const int nrow = U.s_hi - U.s_lo;
            __syncwarp();
            load_ranges(a, U, nrow, sRng, lane);
            __syncwarp();
            const long long k0 = U.sg.gid0 + (long long)U.kt * NKEY;
            for (int pi = 0; pi < U.npairs; pi++, pc++) {
                const int gs = pc % K_GSTG;
                wait_bar(gt_empty + gs, ((pc / K_GSTG) & 1) ^ 1, abort_flag, err, 33);
                float *dst = sGT + gs * RP * NKEY + half * NKEY;
                reinterpret_cast<float4 *>(dst)[2 * hl] = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(dst)[2 * hl + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                __syncwarp();
                const int r = pi * RP + half;
                if (r < nrow) {
                    const long long row = row_of(g, U.sg.b, U.s_lo + r);
                    const int32_t *rid = a.ids + row * K;
                    const float *rg = a.gslot + row * K;
                    const int hi = sRng[2 * r + 1];
                    for (int sl = sRng[2 * r] + hl; sl < hi; sl += 16) {
                        const long long j = (long long)__ldg(rid + sl) - k0;
                        if (j >= 0 && j < NKEY) dst[j] = __ldg(rg + sl);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gt_full + gs);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue (16 warps)
        // Lane = key (quad * 32 + lane).  Warp sub = (warp - 4) / 4 of a quadrant owns X columns [32 sub, 32 sub +
        // 32): the heads [32 (sub % 2), +32) of row `half` = sub / 2 of the pair, and d quarter sub of the flush.
        const int quad = warp & 3, sub = (warp - 4) >> 2, half = sub >> 1, hq = sub & 1;
        const int k = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int xb = 0, dkc = 0, pc = 0;
        uint32_t xph = 0;
        UnitCursor cur;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u, cur);
            for (int pi = 0; pi < U.npairs; pi++, pc++) {
                const int gs = pc % K_GSTG;
                const uint32_t gph = (pc / K_GSTG) & 1;
                // this warp's row of the pair (absent past the chunk's end: its g, w were not loaded) and the
                // keys of the tile visible to it
                const int srow = U.s_lo + pi * RP + half;
                const bool row_ok = srow < U.s_hi;  // warp-uniform
                const int vrow = row_ok ? vis(g, U.sg, srow) : 0;
                const bool r0 = mbar_test(gt_full + gs, gph);
                const bool r1 = mbar_test(x_full + xb, xph);
                if (!(r0 && r1)) {
                    wait_bar(gt_full + gs, gph, abort_flag, err, 29);
                    wait_bar(x_full + xb, xph, abort_flag, err, 30);
                }
                fence_after();
                const uint32_t tcol = tX + lane_off + (uint32_t)(xb * 128 + sub * 32);
                uint32_t pk[16];
                if (row_ok) {
                    uint32_t xr[32];
                    tmem_ld32_async(tcol, xr);
                    const float gk = U.kt * NKEY + k < vrow ? sGT[gs * RP * NKEY + half * NKEY + k] : 0.f;
                    const float4 *wr4 = reinterpret_cast<const float4 *>(sWT + gs * RP * HI + half * HI + hq * 32);
                    float gw[32];
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        const float4 w4 = wr4[c];
                        const float2 lo = mul2(make_float2(gk, gk), make_float2(w4.x, w4.y));
                        const float2 hi = mul2(make_float2(gk, gk), make_float2(w4.z, w4.w));
                        gw[4 * c] = lo.x;
                        gw[4 * c + 1] = lo.y;
                        gw[4 * c + 2] = hi.x;
                        gw[4 * c + 3] = hi.y;
                    }
                    tmem_wait_ld(xr);
#pragma unroll
                    for (int q2 = 0; q2 < 16; q2++)
                        pk[q2] = pack_bf16(__uint_as_float(xr[2 * q2]) > 0.f ? gw[2 * q2] : 0.f,
                                           __uint_as_float(xr[2 * q2 + 1]) > 0.f ? gw[2 * q2 + 1] : 0.f);
                } else {
#pragma unroll
                    for (int c = 0; c < 16; c++) pk[c] = 0u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gt_empty + gs);
                // G[key, (row, h)] of these heads over this warp's own (already read) X columns
                tmem_st16(tcol, pk);
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gk_full + xb);
                if (++xb == K_XSTG) {
                    xb = 0;
                    xph ^= 1u;
                }
            }
            if (U.npairs == 0) continue;
            // ---- flush the unit's dK partial: lane = key, this warp's d quarter
            wait_bar(dk_full, dkc & 1, abort_flag, err, 32);
            fence_after();
            uint32_t vv[32];
            tmem_ld32_async(tDK + lane_off + (uint32_t)(sub * 32), vv);
            tmem_wait_ld(vv);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dk_empty);
            dkc++;
            const int j = U.kt * NKEY + k;
            if (j < U.sg.nc) {
                const long long gid = U.sg.gid0 + j;
                const long long kr = g.layout == CSA_SBHD ? (gid % g.nc) * g.B + gid / g.nc : gid;
                float *dst = a.dk_acc + kr * DI + sub * 32;
#pragma unroll
                for (int c = 0; c < 8; c++)
                    atomicAdd(reinterpret_cast<float4 *>(dst + 4 * c),
                              make_float4(__uint_as_float(vv[4 * c]), __uint_as_float(vv[4 * c + 1]),
                                          __uint_as_float(vv[4 * c + 2]), __uint_as_float(vv[4 * c + 3])));
            }
        }
    }

    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ key-owner kernel from sign bits: dK, long key axes

// On long key axes the gathered row-owner kernel has computed x for every selected (row, key) and stored its signs by
// slot (sgn[row][slot], bit h: x_tjh > 0).  This kernel takes the same units as dk_tc_kernel (a key tile and a chunk
// of up to 128 rows that see it) but forms, per row pair,
//   G[key, (row, h)] = g_ts w_tj 1[x_tjs > 0]          (zero off the row's selection)
// straight from g, w and the signs -- no X MMA and no k tile -- and MMA3 accumulates dK[key, d] += G q
// (A = G from TMEM, B = the pair's q block read MN-major).  Two builder warps (alternate pairs) place each row's g
// and signs for the tile's selected keys into shared memory from the slot range [lo, hi) of the per-row tile-offset
// table; the epilogue expands them into G in TMEM.
// Roles: warp 0 TMA (q blocks, w rows), warp 1 TMEM + MMA issue, warps 2..3 builders, warps 4..19 epilogue.
constexpr int S_QSTG = 6;                                        // q blocks in flight
constexpr int S_GSTG = 4;                                        // g / sign / w slots
constexpr int S_XSTG = 3;                                        // G slots in TMEM, 64 columns each
constexpr int S_OFF_B = 0;                                       // q blocks: 6 x 32 KB
constexpr int S_OFF_GT = S_OFF_B + S_QSTG * QBLK;                // g: slots x 2 rows x 128 fp32
constexpr int S_OFF_BT = S_OFF_GT + S_GSTG * RP * NKEY * 4;      // signs: slots x 2 rows x 128 u64
constexpr int S_OFF_WT = S_OFF_BT + S_GSTG * RP * NKEY * 8;      // w rows: slots x 2 rows x 64 fp32
constexpr int S_OFF_RNG = S_OFF_WT + S_GSTG * RP * HI * 4;       // per builder: a unit's slot ranges, CH x 2 int
constexpr int S_OFF_MISC = S_OFF_RNG + 2 * CH * 2 * 4;
constexpr int S_SMEM = S_OFF_MISC + 1024 + 1024;
static_assert(S_SMEM <= 232448, "sign-bit key-owner shared memory exceeds the per-block limit");
static_assert((2 * S_QSTG + 2 * S_GSTG + 2 * S_XSTG + 3) * 8 <= 256, "sign-bit key-owner barriers overlap the TMEM slot");

__global__ void __launch_bounds__(THREADS, 1)
dk_sign_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_w, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sB = smem + S_OFF_B;
    float *sGT = reinterpret_cast<float *>(smem + S_OFF_GT);
    unsigned long long *sBT = reinterpret_cast<unsigned long long *>(smem + S_OFF_BT);
    float *sWT = reinterpret_cast<float *>(smem + S_OFF_WT);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S_OFF_MISC);
    uint64_t *b_full = bars, *b_empty = bars + S_QSTG, *gt_full = bars + 2 * S_QSTG, *gt_empty = gt_full + S_GSTG;
    uint64_t *gk_full = gt_empty + S_GSTG, *x_empty = gk_full + S_XSTG;
    uint64_t *dk_full = x_empty + S_XSTG, *dk_empty = dk_full + 1, *mma_done = dk_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + S_OFF_MISC + 256);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + S_OFF_MISC + 264);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    int *err = &g_bwd_error;

    if (threadIdx.x == 0) {
        for (int i = 0; i < S_QSTG; i++) { mbar_init(b_full + i, 1); mbar_init(b_empty + i, 1); }
        // a g/sign/w slot is full once its w copy has landed and a builder has placed g and the signs
        for (int i = 0; i < S_GSTG; i++) { mbar_init(gt_full + i, 2); mbar_init(gt_empty + i, EPI / 32); }
        for (int i = 0; i < S_XSTG; i++) { mbar_init(gk_full + i, EPI / 32); mbar_init(x_empty + i, 1); }
        mbar_init(dk_full, 1);
        mbar_init(dk_empty, EPI / 32);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    // TMEM: three G slots of 64 columns (bf16 pairs: K index (row, h) = 64 row + h at column (64 row + h) / 2), and
    // dK (128 columns) at 256
    const uint32_t tG = tmem, tDK = tmem + 256;
    const int total = unit_total(a);

    if (warp == 0) {
        if (lane == 0) {  // ------------------------------------------------ TMA producer
            int qs = 0, pc = 0;
            UnitCursor cur;
            for (int u = blockIdx.x; u < total; u += gridDim.x) {
                const Unit U = decode_unit(a, u, cur);
                for (int pi = 0; pi < U.npairs; pi++) {
                    // the pair's q rows and w rows, one copy each (a second row past the chunk's end is read, never used)
                    const int s0 = U.s_lo + pi * RP;
                    const PairAt at = pair_at(g, U.sg.b, s0, row_of(g, U.sg.b, s0));
                    const int bs = qs % S_QSTG;
                    wait_bar(b_empty + bs, ((qs / S_QSTG) & 1) ^ 1, abort_flag, err, 34);
                    mbar_expect_tx(b_full + bs, QBLK);
                    tma_load_5d(sB + bs * QBLK, &map_q, b_full + bs, 0, 0, at.y, at.z, 0);
                    qs++;
                    const int gs = pc % S_GSTG;
                    wait_bar(gt_empty + gs, ((pc / S_GSTG) & 1) ^ 1, abort_flag, err, 35);
                    mbar_expect_tx(gt_full + gs, (uint32_t)(RP * HI * 4));
                    tma_load_3d(sWT + gs * RP * HI, &map_w, gt_full + gs, 0, at.y, at.z);
                    pc++;
                }
            }
            for (int q = qs - S_QSTG < 0 ? 0 : qs - S_QSTG; q < qs; q++) drain_bar(b_full + q % S_QSTG, (q / S_QSTG) & 1, err);
            for (int q = pc - S_GSTG < 0 ? 0 : pc - S_GSTG; q < pc; q++) drain_bar(gt_full + q % S_GSTG, (q / S_GSTG) & 1, err);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------------------- MMA issue (whole warp)
        //   dK[key, d] += G q   (A = G from TMEM, K index (row, h); B = the pair's q block read MN-major)
        // After each pair's MMAs the next pair's q block and G slot are probed in one shared-memory round trip,
        // which overlaps the MMAs just queued; the warp waits only when either was not yet complete.  (The next
        // pair's barriers cannot be two phases behind: their previous uses have been consumed.)
        int qs = 0, xc = 0, uc = 0;
        bool rdy = false;  // the next pair's q block and G slot are known complete
        UnitCursor cur;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u, cur);
            if (U.npairs == 0) continue;
            for (int pi = 0; pi < U.npairs; pi++) {
                const int bs = qs % S_QSTG, xb = xc % S_XSTG;
                if (pi == 0) wait_bar(dk_empty, (uc & 1) ^ 1, abort_flag, err, 36);
                if (!rdy) {
                    wait_bar(b_full + bs, (qs / S_QSTG) & 1, abort_flag, err, 37);
                    wait_bar(gk_full + xb, (xc / S_XSTG) & 1, abort_flag, err, 38);
                }
                fence_after();
                // eight MMAs of K = 16 (A: G columns 8 s of the slot; B: the q block, 2 KB further per MMA) in two
                // groups of four under one elect each, then the commits
                const uint64_t bq = desc_sw128(sB + bs * QBLK, HALF, 1024);
                mma4_ts_w(tDK, tG + (uint32_t)(xb * 64), 8, 16, bq, 2048 >> 4, IDESC_DK, pi == 0 ? 0u : 1u, 0u);
                mma4_ts_w(tDK, tG + (uint32_t)(xb * 64 + 32), 8, 16, bq + (4 * 2048 >> 4), 2048 >> 4, IDESC_DK, 1u,
                          su32(x_empty + xb));
                mma_commit_w(b_empty + bs);
                qs++;
                xc++;
                rdy = mbar_test2(b_full + qs % S_QSTG, (qs / S_QSTG) & 1, gk_full + xc % S_XSTG, (xc / S_XSTG) & 1) == 3u;
            }
            mma_commit_w(dk_full);
            uc++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp == 2 || warp == 3) {
        // ---------------------------------------------------------------- builders (pairs alternate between them)
        // Per unit: the slot range [lo, hi) of its key tile in each of its rows.  Per row pair of this builder, into
        // the pair's slot: half-warp r zeroes row r's 128 keys and places g and the signs of its slots lo .. hi - 1,
        // all loaded at once (at most 128 per row and tile: eight per lane); keys outside the tile are never placed.
        const int bw = warp - 2;
        const int half = lane >> 4, hl = lane & 15;
        const int K = g.K;
        int *sRng = reinterpret_cast<int *>(smem + S_OFF_RNG) + bw * CH * 2;
        int pc = 0;
        UnitCursor cur;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u, cur);
            if (U.npairs == 0) continue;
            const int nrow = U.s_hi - U.s_lo;
            __syncwarp();
            load_ranges(a, U, nrow, sRng, lane);
            __syncwarp();
            const long long k0 = U.sg.gid0 + (long long)U.kt * NKEY;
            for (int pi = 0; pi < U.npairs; pi++, pc++) {
                if ((pc & 1) != bw) continue;
                const int gs = pc % S_GSTG;
                const int r = pi * RP + half;
                // the pair's entries, loaded before the slot is waited for
                int32_t id[8];
                float gv[8];
                unsigned long long bv[8];
                int lo = 0, hi = 0;
                long long row = 0;
                if (r < nrow) {
                    row = row_of(g, U.sg.b, U.s_lo + r);
                    lo = sRng[2 * r];
                    hi = sRng[2 * r + 1];
                }
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const int sl = lo + hl + 16 * e;
                    id[e] = -1;
                    gv[e] = 0.f;
                    bv[e] = 0ull;
                    if (sl < hi) {
                        id[e] = __ldg(a.ids + row * K + sl);
                        gv[e] = __ldg(a.gslot + row * K + sl);
                        bv[e] = __ldg(a.sgn + row * K + sl);
                    }
                }
                wait_bar(gt_empty + gs, ((pc / S_GSTG) & 1) ^ 1, abort_flag, err, 39);
                float *dg = sGT + (gs * RP + half) * NKEY;
                unsigned long long *db = sBT + (gs * RP + half) * NKEY;
                reinterpret_cast<float4 *>(dg)[2 * hl] = make_float4(0.f, 0.f, 0.f, 0.f);
                reinterpret_cast<float4 *>(dg)[2 * hl + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int e = 0; e < 4; e++) reinterpret_cast<ulonglong2 *>(db)[4 * hl + e] = make_ulonglong2(0ull, 0ull);
                __syncwarp();
#pragma unroll
                for (int e = 0; e < 8; e++) {
                    const long long j = (long long)id[e] - k0;
                    if (id[e] >= 0 && j >= 0 && j < NKEY) {
                        dg[j] = gv[e];
                        db[j] = bv[e];
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gt_full + gs);
            }
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue (16 warps)
        // Lane = key (quad * 32 + lane).  Warp sub = (warp - 4) / 4 of a quadrant forms G for heads [32 (sub % 2), +32)
        // of row `half` = sub / 2 of the pair (16 pair columns at 32 half + 16 (sub % 2) of the G slot) and flushes d
        // quarter sub of the unit's dK.
        const int quad = warp & 3, sub = (warp - 4) >> 2, half = sub >> 1, hq = sub & 1;
        const int k = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int xc = 0, dkc = 0, pc = 0;
        UnitCursor cur;
        for (int u = blockIdx.x; u < total; u += gridDim.x) {
            const Unit U = decode_unit(a, u, cur);
            for (int pi = 0; pi < U.npairs; pi++, pc++, xc++) {
                const int gs = pc % S_GSTG, xb = xc % S_XSTG;
                const bool row_ok = U.s_lo + pi * RP + half < U.s_hi;  // warp-uniform
                wait_bar(gt_full + gs, (pc / S_GSTG) & 1, abort_flag, err, 40);
                wait_bar(x_empty + xb, ((xc / S_XSTG) & 1) ^ 1, abort_flag, err, 41);
                fence_after();
                uint32_t pk[16];
                if (row_ok) {
                    const float gk = sGT[(gs * RP + half) * NKEY + k];
                    const uint32_t bits = (uint32_t)(sBT[(gs * RP + half) * NKEY + k] >> (32 * hq));
                    const float4 *wr4 = reinterpret_cast<const float4 *>(sWT + gs * RP * HI + half * HI + hq * 32);
#pragma unroll
                    for (int c = 0; c < 8; c++) {
                        const float4 w4 = wr4[c];
                        const float2 lo = mul2(make_float2(gk, gk), make_float2(w4.x, w4.y));
                        const float2 hi = mul2(make_float2(gk, gk), make_float2(w4.z, w4.w));
                        pk[2 * c] = pack_bf16((bits >> (4 * c)) & 1u ? lo.x : 0.f, (bits >> (4 * c + 1)) & 1u ? lo.y : 0.f);
                        pk[2 * c + 1] = pack_bf16((bits >> (4 * c + 2)) & 1u ? hi.x : 0.f, (bits >> (4 * c + 3)) & 1u ? hi.y : 0.f);
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; c++) pk[c] = 0u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(gt_empty + gs);
                tmem_st16(tG + lane_off + (uint32_t)(xb * 64 + half * 32 + hq * 16), pk);
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(gk_full + xb);
            }
            if (U.npairs == 0) continue;
            // ---- flush the unit's dK partial: lane = key, this warp's d quarter
            wait_bar(dk_full, dkc & 1, abort_flag, err, 42);
            fence_after();
            uint32_t vv[32];
            tmem_ld32_async(tDK + lane_off + (uint32_t)(sub * 32), vv);
            tmem_wait_ld(vv);
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dk_empty);
            dkc++;
            const int j = U.kt * NKEY + k;
            if (j < U.sg.nc) {
                const long long gid = U.sg.gid0 + j;
                const long long kr = g.layout == CSA_SBHD ? (gid % g.nc) * g.B + gid / g.nc : gid;
                float *dst = a.dk_acc + kr * DI + sub * 32;
#pragma unroll
                for (int c = 0; c < 8; c++)
                    atomicAdd(reinterpret_cast<float4 *>(dst + 4 * c),
                              make_float4(__uint_as_float(vv[4 * c]), __uint_as_float(vv[4 * c + 1]),
                                          __uint_as_float(vv[4 * c + 2]), __uint_as_float(vv[4 * c + 3])));
            }
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

// Long key axis: toff[r][b] = the first slot of row r whose key (id minus the row's first key) lies at or above
// 128 b, b = 0 .. NT (the slots hold ascending valid ids, then -1 pads; a pad or an invalid id counts as past the
// last tile, and a virtual slot K closes the remaining boundaries).  One warp per row.
__global__ void tile_offsets_kernel(Geo g, const int32_t *__restrict__ ids, int *__restrict__ toff, int NT)
{
    const int lane = threadIdx.x & 31;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long r = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < g.rows; r += nwarps) {
        const Row R = decode_row(g, r);
        const long long gid0 = key_gid(g, R, 0);
        int *o = toff + r * (long long)(NT + 1);
        const int32_t *rid = ids + r * (long long)g.K;
        int prev = -1;  // tile of the slot before this chunk
        for (int s0 = 0; s0 <= g.K; s0 += 32) {
            const int sl = s0 + lane;
            int ts = NT;
            if (sl < g.K) {
                const int32_t id = __ldg(rid + sl);
                const long long j = (long long)id - gid0;
                if (id >= 0 && j >= 0 && j < R.v) ts = (int)(j >> 7) < NT ? (int)(j >> 7) : NT;
            }
            int tp = __shfl_up_sync(0xffffffffu, ts, 1);
            if (lane == 0) tp = prev;
            if (sl <= g.K)
                for (int b = tp + 1; b <= ts; b++) o[b] = sl;
            prev = __shfl_sync(0xffffffffu, ts, 31);
        }
    }
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
    // long key axes take the sparse loss (g by slot, assembled from the ascending ids)
    return bf16 && g.HI == bwd::HI && g.DI == bwd::DI && g.NC >= 1 && (g.NC <= bwd::NCMAX || g.sparse) &&
           g.K >= 1 && g.rows > 0 && g.key_rows > 0;
}

bool tc_bwd_long(const Geo &g) { return g.NC > bwd::NCMAX; }

int tc_bwd_tiles(const Geo &g) { return (g.NC + bwd::NKEY - 1) / bwd::NKEY; }

int tc_bwd_ncp(const Geo &g) { return tc_bwd_tiles(g) * bwd::NKEY; }

static size_t bwd_offsets_bytes(const Geo &g)
{
    const size_t offs = sizeof(int) * 2 * (size_t)(g.layout == CSA_THD ? g.B + 1 : 1);
    return (offs + 255) & ~(size_t)255;
}

// long key axis: the tile-offset rows, then the signs of x by slot
static size_t toff_bytes(const Geo &g)
{
    return ((sizeof(int) * (size_t)g.rows * (size_t)(tc_bwd_tiles(g) + 1)) + 255) & ~(size_t)255;
}

size_t tc_bwd_workspace_bytes(const Geo &g)
{
    if (tc_bwd_long(g))
        return bwd_offsets_bytes(g) + toff_bytes(g) + sizeof(unsigned long long) * (size_t)g.rows * (size_t)g.K;
    return bwd_offsets_bytes(g) + sizeof(float) * (size_t)g.rows * (size_t)tc_bwd_ncp(g);
}

float *tc_bwd_gd(const Geo &g, void *ws)
{
    return reinterpret_cast<float *>(static_cast<char *>(ws) + bwd_offsets_bytes(g));
}

cudaError_t launch_bwd_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                          __nv_bfloat16 *dq, float *dw, float *dk_acc, void *ws, const int32_t *ids,
                          const float *gslot, cudaStream_t st)
{
    using namespace bwd;
    const bool lng = tc_bwd_long(g);
    // Pair maps: a row pair of q_idx (both K-halves: [half][row][head][64 d] in shared memory) and of w in one
    // copy; a k tile (both K-halves: [half][key][64 d]) in one copy; g rows by position, two rows x 128 keys.
    const bool sb = g.layout == CSA_SBHD;
    const cuuint64_t rowb = (cuuint64_t)HI * DI * 2;
    const cuuint64_t y_n = sb ? (cuuint64_t)g.B : (cuuint64_t)g.rows, z_n = sb ? (cuuint64_t)g.S : 1;
    const cuuint64_t z_str = sb ? (cuuint64_t)g.B * rowb : (cuuint64_t)g.rows * rowb;
    const cuuint32_t by = sb ? 1 : 2, bz = sb ? 2 : 1;
    const cuuint64_t qd[5] = {64, (cuuint64_t)HI, y_n, z_n, 2};
    const cuuint64_t qs[4] = {(cuuint64_t)DI * 2, rowb, z_str, 128};
    const cuuint32_t qb[5] = {64, (cuuint32_t)HI, by, bz, 2};
    const cuuint64_t wd[3] = {(cuuint64_t)HI, y_n, z_n};
    const cuuint64_t ws_[2] = {(cuuint64_t)HI * 4, sb ? (cuuint64_t)g.B * HI * 4 : (cuuint64_t)g.rows * HI * 4};
    const cuuint32_t wb[3] = {(cuuint32_t)HI, by, bz};
    const cuuint64_t gdim[2] = {(cuuint64_t)tc_bwd_ncp(g), (cuuint64_t)g.rows};
    const cuuint64_t gstr[1] = {(cuuint64_t)tc_bwd_ncp(g) * 4};
    const cuuint32_t gbox[2] = {NKEY, RP};
    CUtensorMap mq, mk, mg, mw;
    bool ok = tc_encode_bf16(&mq, q_idx, 5, qd, qs, qb) && tc_encode_f32(&mw, w, 3, wd, ws_, wb);
    if (lng) mg = mw;  // no by-key g rows: the map is never used
    else ok = ok && tc_encode_f32(&mg, tc_bwd_gd(g, ws), 2, gdim, gstr, gbox);
    if (sb) {
        const cuuint64_t kd[4] = {64, (cuuint64_t)g.B, (cuuint64_t)g.nc, 2};
        const cuuint64_t ks[3] = {(cuuint64_t)DI * 2, (cuuint64_t)g.B * DI * 2, 128};
        const cuuint32_t kb[4] = {64, 1, NKEY, 2};
        ok = ok && tc_encode_bf16(&mk, k_idx, 4, kd, ks, kb);
    } else {
        const cuuint64_t kd[3] = {64, (cuuint64_t)g.key_rows, 2};
        const cuuint64_t ks[2] = {(cuuint64_t)DI * 2, 128};
        const cuuint32_t kb[3] = {64, NKEY, 2};
        ok = ok && tc_encode_bf16(&mk, k_idx, 3, kd, ks, kb);
    }
    if (!ok) return cudaErrorInvalidValue;
    const int NT = tc_bwd_tiles(g);
    Args a = {};  // every field set below; zero first so none is ever left unset
    a.g = g;
    a.dq = dq;
    a.dw = dw;
    a.dk_acc = dk_acc;
    a.cu_g = a.cu_u = nullptr;
    a.total_items = a.total_units = a.units_per_seq = 0;
    a.lng = lng;
    a.gslot = gslot;
    a.ids = ids;
    a.NT = NT;
    a.toff = lng ? reinterpret_cast<const int *>(tc_bwd_gd(g, ws)) : nullptr;
    unsigned long long *sgn =
        lng ? reinterpret_cast<unsigned long long *>(reinterpret_cast<char *>(tc_bwd_gd(g, ws)) + toff_bytes(g)) : nullptr;
    a.sgn = sgn;
    int upper_items, upper_units;
    if (g.layout == CSA_THD) {
        int *cu_g = static_cast<int *>(ws);
        int *cu_u = cu_g + (g.B + 1);
        build_bwd_offsets_kernel<<<1, 32, 0, st>>>(g, cu_g, cu_u);
        note_launches(1);
        a.cu_g = cu_g;
        a.cu_u = cu_u;
        upper_items = (g.rows + RP - 1) / RP + g.B;
        upper_units = (g.rows + CH - 1) / CH * NT + g.B * NT;
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
    if (lng) {
        const long long blocks = ((long long)g.rows + 7) / 8;
        tile_offsets_kernel<<<(int)(blocks < sms * 16 ? blocks : sms * 16), 256, 0, st>>>(
            g, ids, const_cast<int *>(a.toff), NT);
        note_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (lng) {
        // long key axis: the row-owner over each row's selected keys only
        e = launch_dq_dw_gather_tc(g, q_idx, w, k_idx, ids, gslot, dq, dw, sgn, st);
    } else {
        const int g1 = upper_items < sms ? (upper_items > 0 ? upper_items : 1) : sms;
        dq_dw_tc_kernel<<<g1, R_THREADS, R_SMEM, st>>>(mq, mk, mg, mw, a);
        note_launches(1);
        e = cudaGetLastError();
    }
    if (e != cudaSuccess) return e;
    if (lng && upper_units > 0) {
        // long key axis: dK from the signs the row-owner has just written (stream order, no overlap)
        e = cudaFuncSetAttribute(dk_sign_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, S_SMEM);
        if (e != cudaSuccess) return e;
        const int g2 = upper_units < sms ? upper_units : sms;
        dk_sign_tc_kernel<<<g2, THREADS, S_SMEM, st>>>(mq, mw, a);
        note_launches(1);
        return cudaGetLastError();
    }
    if (upper_units > 0) {
        // launched as a programmatic dependent of the row-owner kernel (which it does not depend on), so its
        // CTAs start on the SMs the row-owner's last items leave idle
        const int g2 = upper_units < sms ? upper_units : sms;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(g2);
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = K_SMEM;
        cfg.stream = st;
        cudaLaunchAttribute at[1];
        at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        at[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = at;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, dk_tc_kernel, mq, mk, mg, mw, a);
        if (e != cudaSuccess) return e;
        note_launches(1);
    }
    return cudaGetLastError();
}

}  // namespace csa
