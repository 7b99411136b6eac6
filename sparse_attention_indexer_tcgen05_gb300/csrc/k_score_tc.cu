// k_score_tc.cu -- indexer score GEMM on the 5th-generation tensor cores (tcgen05 + TMEM + TMA), fused
// with the ReLU.w head reduction, the compressed causal mask and an exact per-row top-k in shared memory.
//
// What it computes ("[Bug] DSV4 unfused CSA indexer loss uses a compressed-only teacher ..." (Megatron-LM
// issue #5776), sec. 1 excerpt: mask where(arange(n_c) >= positions // ratio, -inf, 0) and
// min(index_topk, n_compressed); sec. 3 excerpt: invalid slots -1; "Megatron-LM PR #8539" item 1: global ids):
//   I[t,s] = sum_j w[t,j] * max(0, q_idx[t,j] . k_idx[s]) for the keys s < i_t / r, then the K largest per row
//   (ties to the lower key), written as ascending global ids with their fp32 scores.
//
// Shape taken: bf16 values, H_I = 64 indexer heads, D_I = 128.  Key axes up to 1024 keep an item's score rows
// whole in shared memory (score_topk_tc_kernel); longer ones (up to 65535 keys, K <= 3840) stream the score
// tiles into per-row candidate buffers (score_topk_long_tc_kernel, below).  Other shapes and fp32 values take
// the CUDA-core kernels.
//
// Mapping.  A work item is 4 consecutive query positions of one sequence (or THD segment).  The MMA computes
// D[key, (row, head)] = k_idx[key] . q_idx[row, head] with M = 128 keys (A = a k_idx tile, K-major, streamed
// by TMA), N = 4 rows x 64 heads = 256 (B = the item's q_idx rows, K-major, resident), K = 128 (8 MMAs of
// K = 16).  With keys on TMEM lanes and (row, head) on columns, each epilogue thread owns one key and reduces
// the 64 heads of a row in registers: no cross-thread reduction.  TMEM holds two 256-column accumulators
// (double buffer), so the epilogue of one key tile overlaps the MMAs of the next.
//
// Roles (one CTA per SM, persistent, static round-robin over items ordered heaviest first):
//   warp 0      TMA producer: B (q_idx rows, 64 KB, 2 buffers) and A (k_idx K-halves, 16 KB, 3 stages)
//   warp 1      TMEM allocation and the tcgen05.mma issue (warp-wide loop, one elected lane issues)
//   warps 2..9  epilogue (TMEM -> registers -> ReLU.w reduction -> shared score rows, two item buffers)
//   warps 10..17 top-k, one warp per row, two sets taking alternate items (three score buffers), while the
//               epilogue runs the following items:
//               the exact k-th largest score by a bitwise search on order-preserving keys held in
//               registers, then the selection written by a stable ballot compaction.
//   (long key axis: warps 10..13, one per row, follow the epilogue tile by tile through a six-tile ring; each
//    keeps the row's current best candidates, cuts them back to about the top K with a radix walk when the
//    buffer fills, and to exactly the top K at the row's end.)
//
// Every mbarrier wait is bounded: on expiry the kernel records an error code (read back by
// csa_check_device_status), stops waiting (so every role still runs its loops to the end with uniform
// control flow), drains its own TMA copies and MMAs with timer-bounded waits, frees TMEM and returns.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <stdlib.h>

namespace csa {

static __device__ int g_tc_error = 0;

cudaError_t tc_read_clear_error(int *flag)
{
    int f1 = 0, f2 = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&f1, g_tc_error, sizeof(int));
    if (e != cudaSuccess) return e;
    if (f1 != 0) {
        int zero = 0;
        e = cudaMemcpyToSymbol(g_tc_error, &zero, sizeof(int));
        if (e != cudaSuccess) return e;
    }
    e = bwd_tc_read_clear_error(&f2);
    if (e != cudaSuccess) return e;
    int f3 = 0, f4 = 0, f5 = 0;
    e = teacher_tc_read_clear_error(&f3);
    if (e != cudaSuccess) return e;
    e = teacher_h128_read_clear_error(&f4);
    if (e != cudaSuccess) return e;
    e = bwd_gather_read_clear_error(&f5);
    // the first kernel's code, as 100 x kernel + site (1 score, 2 backward, 3 64-head teacher, 4 128-head
    // teacher, 5 gathered row-owner); site 99 is a drain that ran out
    *flag = f1 != 0 ? 100 + f1 : (f2 != 0 ? 200 + f2 : (f3 != 0 ? 300 + f3 : (f4 != 0 ? 400 + f4 : (f5 != 0 ? 500 + f5 : 0))));
    return e;
}

namespace tcs {

using namespace ptx;

constexpr int ROWS = 4;                       // query rows per work item
constexpr int HI = 64, DI = 128;              // indexer heads / dim taken by this kernel
constexpr int NKEY = 128;                     // keys per tile (MMA M)
constexpr int NCOL = ROWS * HI;               // MMA N = 256
constexpr int NCMAX = 1024;                   // longest key axis whose score rows are held whole in shared memory
constexpr int A_HALF = NKEY * 64 * 2;         // 16 KB: one 64-wide K-half of a key tile
constexpr int A_STAGES = 3;
constexpr int B_HALF = NCOL * 64 * 2;         // 32 KB
constexpr int B_BUF = 2 * B_HALF;             // 64 KB
constexpr int EPI = 256;
constexpr int SEL_WARP0 = 10;
constexpr int TMEM_COLS = 512;

// Two instantiations of one kernel body:
//   short key axis (<= NCMAX keys): an item's score rows are kept whole in shared memory (three item buffers)
//     and each row is selected by one warp once the item is done; two sets of four selection warps take
//     alternate items; the q_idx rows of two items are resident (double buffer).
//   long key axis: the score rows stream through a ring of key tiles; the selection warp of each row keeps a
//     candidate buffer of at most CAP (key, index) entries in ascending key order and admits a new key only
//     when it lies strictly above the row's current threshold, a value with at least K buffered keys at or above
//     it (a later key loses a tie, so no key at or below it can reach the top K).  Whenever the next tile might
//     not fit, the buffer is cut back to the keys at or above a radix bin edge with between K and K + 256 keys
//     above it (that edge becomes the threshold); at the row's end it is cut to exactly the top K, ties to the
//     lower key.  One set of four selection warps; one q_idx buffer.
template <bool LONG> struct SC;
template <> struct SC<false> {
    static constexpr int THREADS = 576;       // warps 0 TMA, 1 MMA, 2..9 epilogue, 10..17 selection
    static constexpr int NB = 2;              // q_idx item buffers
    static constexpr int NSC = 3;             // item score buffers
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + A_STAGES * A_HALF;        // 48 KB
    static constexpr int OFF_SC = OFF_B + NB * B_BUF;              // 176 KB
    static constexpr int OFF_W = OFF_SC + NSC * ROWS * NCMAX * 4;  // score rows of three items
    static constexpr int OFF_MISC = OFF_W + ROWS * HI * 4;
    static constexpr int SMEM_ALLOC = OFF_MISC + 1024 + 1024;      // slack to align the base to 1024 B
};
template <> struct SC<true> {
    static constexpr int THREADS = 448;       // warps 0 TMA, 1 MMA, 2..9 epilogue, 10..13 selection
    static constexpr int NB = 1;
    static constexpr int NRING = 6;           // score tiles in flight between epilogue and selection (2 KB each)
    static constexpr int CAP = 4096;          // candidate entries per row
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + A_STAGES * A_HALF;        // 48 KB
    static constexpr int OFF_RING = OFF_B + NB * B_BUF;            // 112 KB
    static constexpr int OFF_W = OFF_RING + NRING * ROWS * NKEY * 4;
    static constexpr int OFF_CK = OFF_W + ROWS * HI * 4;           // candidate keys [ROWS][CAP] u32
    static constexpr int OFF_CI = OFF_CK + ROWS * CAP * 4;         // candidate indices [ROWS][CAP] u16
    static constexpr int OFF_HIST = OFF_CI + ROWS * CAP * 2;       // radix histograms [ROWS][256] u32
    static constexpr int OFF_MISC = OFF_HIST + ROWS * 256 * 4;
    static constexpr int SMEM_ALLOC = OFF_MISC + 1024 + 1024;
};
static_assert(SC<false>::SMEM_ALLOC <= 232448, "score kernel exceeds the 227 KB of shared memory a CTA may use");
static_assert(SC<true>::SMEM_ALLOC <= 232448, "long score kernel exceeds the 227 KB of shared memory a CTA may use");
// the epilogue -> selection barriers: X_BARS full and X_BARS empty ones after the 17 pipeline barriers, all below
// the TMEM slot at byte 256 of the barrier area
constexpr int X_BARS = 6;
static_assert(SC<true>::NRING <= X_BARS && SC<false>::NSC <= X_BARS && (17 + 2 * X_BARS) * 8 <= 256,
              "score kernel barriers overlap the TMEM slot");
// largest K the long kernel takes: an in-loop cut leaves room for two more tiles (at most K + slack entries, slack =
// min(256, CAP - 2 NKEY - K) >= 0, or a sampled pivot's at most n - 2 NKEY)
constexpr int LONG_KMAX = SC<true>::CAP - 2 * NKEY;
constexpr int LONG_NCMAX = 65535;             // candidate indices are 16-bit

constexpr uint32_t IDESC = idesc_bf16(NKEY, NCOL, false, false);  // A, B both K-major

struct Args {
    Geo g;
    const float *w;
    int32_t *ids;
    float *selscore;
    float *dump;
    long long dump_row0, dump_rows;
    const int *cu_g;     // THD: work-item offsets per segment [nseg+1]
    int total;           // SBHD/BSHD: number of work items (THD: read from cu_g[nseg])
};

// ------------------------------------------------------------------ work items

struct Item {
    int b, n;                 // segment / sequence, rows present (1..4)
    long long row[ROWS];      // memory rows
    int v[ROWS];              // visible keys per row
    int vmax;
    long long gid0;           // global id of local key 0
    long long key_y;          // TMA row coordinate of local key 0 (2D maps)
};

__device__ __forceinline__ int item_total(const Args &a)
{
    return a.g.layout == CSA_THD ? __ldg(a.cu_g + a.g.B) : a.total;
}

__device__ Item decode_item(const Args &a, int i, int total)
{
    const Geo &g = a.g;
    Item it;
    int s0, len_phys, len_real;
    long long c_base = 0;
    if (g.layout == CSA_THD) {
        const int ir = total - 1 - i;  // later segments first
        int lo = 0, hi = g.B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (__ldg(a.cu_g + mid) <= ir) lo = mid; else hi = mid - 1;
        }
        it.b = lo;
        s0 = (ir - __ldg(a.cu_g + lo)) * ROWS;
        len_phys = __ldg(g.cu_q + lo + 1) - __ldg(g.cu_q + lo);
        len_real = __ldg(g.cu_real + lo + 1) - __ldg(g.cu_real + lo);
        c_base = __ldg(g.cu_c + lo);
        it.gid0 = c_base;
        it.key_y = c_base;
    } else {
        const int groups = (g.S + ROWS - 1) / ROWS;
        it.b = i % g.B;
        s0 = (groups - 1 - i / g.B) * ROWS;  // latest positions (most keys) first
        len_phys = len_real = g.S;
        it.gid0 = (long long)it.b * g.nc;
        it.key_y = it.gid0;
    }
    it.n = 0;
    it.vmax = 0;
    for (int k = 0; k < ROWS; k++) {
        const int s = s0 + k;
        it.v[k] = 0;
        it.row[k] = -1;
        if (s >= len_phys) continue;
        it.n = k + 1;
        if (g.layout == CSA_SBHD) it.row[k] = (long long)s * g.B + it.b;
        else if (g.layout == CSA_BSHD) it.row[k] = (long long)it.b * g.S + s;
        else it.row[k] = (long long)__ldg(g.cu_q + it.b) + s;
        int v = s < len_real ? (s + 1) / g.ratio : 0;
        if (v > g.NC) v = g.NC;
        if (g.layout == CSA_THD && c_base + v > g.key_rows) v = c_base < g.key_rows ? (int)(g.key_rows - c_base) : 0;
        it.v[k] = v;
        it.vmax = v > it.vmax ? v : it.vmax;
    }
    return it;
}

// memory row of row k (0..3) of item i, or -1 when the item has no such row
__device__ long long item_row(const Args &a, int i, int total, int k)
{
    const Geo &g = a.g;
    int b, s0, len_phys;
    if (g.layout == CSA_THD) {
        const int ir = total - 1 - i;
        int lo = 0, hi = g.B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (__ldg(a.cu_g + mid) <= ir) lo = mid; else hi = mid - 1;
        }
        b = lo;
        s0 = (ir - __ldg(a.cu_g + lo)) * ROWS;
        len_phys = __ldg(g.cu_q + lo + 1) - __ldg(g.cu_q + lo);
    } else {
        const int groups = (g.S + ROWS - 1) / ROWS;
        b = i % g.B;
        s0 = (groups - 1 - i / g.B) * ROWS;
        len_phys = g.S;
    }
    const int s = s0 + k;
    if (s >= len_phys) return -1;
    if (g.layout == CSA_SBHD) return (long long)s * g.B + b;
    if (g.layout == CSA_BSHD) return (long long)b * g.S + s;
    return (long long)__ldg(g.cu_q + b) + s;
}

// ------------------------------------------------------------------ top-k of one row (a warp pair)

// inverse of score_key (the key of -0.0 is that of +0.0, so -0.0 comes back as +0.0: the same value)
__device__ __forceinline__ float key_score(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// One warp selects one row: the min(K, v) largest of the row's v scores, ties to the lower key, written in
// ascending key order.  Lane l holds the keys of slots j = 32 e + l (e = 0..31): conflict-free shared-memory
// reads, and key order is (e, lane), so a stable compaction takes one ballot per e.  The row's scores are
// read once into registers; `release` (an mbarrier, arrived by lane 0) is signalled as soon as the shared
// rows may be overwritten.
__device__ void select_row(const Args &a, const Item &it, int k, const float *sc, uint64_t *release)
{
    const Geo &g = a.g;
    const int lane = threadIdx.x & 31;
    const int v = it.v[k];
    const int K = g.K;
    const int kk = v < K ? v : K;
    const long long r = it.row[k];
    int32_t *orow = a.ids + r * K;
    float *srow = a.selscore + r * K;
    constexpr int PER = NCMAX / 32;
    uint32_t key[PER];
#pragma unroll
    for (int e = 0; e < PER; e++) {
        const int j = 32 * e + lane;
        key[e] = j < v ? score_key(sc[j]) : 0u;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(release);
    if (kk == v) {
        // every visible key is selected: ascending order as is
#pragma unroll
        for (int e = 0; e < PER; e++) {
            const int j = 32 * e + lane;
            if (j < v) {
                orow[j] = (int32_t)(it.gid0 + j);
                srow[j] = key_score(key[e]);
            }
        }
    } else {
        // the k-th largest key: the largest T with #(key >= T) >= kk, built bit by bit (keys of absent slots
        // are 0, below every present score's key); four independent partial counts per round.  The search
        // stops early once exactly kk keys lie at or above the candidate: that set is the top kk whatever the
        // remaining bits, and no tie is cut at T.
        uint32_t T = 0u;
        for (int bit = 31; bit >= 0; bit--) {
            const uint32_t cand = T | (1u << bit);
            unsigned c4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
            for (int e = 0; e < PER; e++) c4[e & 3] += key[e] >= cand ? 1u : 0u;
            const int c = (int)__reduce_add_sync(0xffffffffu, (c4[0] + c4[1]) + (c4[2] + c4[3]));
            if (c >= kk) {
                T = cand;
                if (c == kk) break;
            }
        }
        unsigned gt4[4] = {0u, 0u, 0u, 0u}, eq4[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int e = 0; e < PER; e++) {
            gt4[e & 3] += key[e] > T ? 1u : 0u;
            eq4[e & 3] += (key[e] == T && key[e] != 0u) ? 1u : 0u;
        }
        const int need_eq = kk - (int)__reduce_add_sync(0xffffffffu, (gt4[0] + gt4[1]) + (gt4[2] + gt4[3]));
        const int eq_tot = (int)__reduce_add_sync(0xffffffffu, (eq4[0] + eq4[1]) + (eq4[2] + eq4[3]));
        const unsigned lt_mask = (1u << lane) - 1u;
        int base = 0;
        if (eq_tot == need_eq) {
            // no tie is cut: every key >= T is selected
#pragma unroll
            for (int e = 0; e < PER; e++) {
                const bool sel = key[e] >= T && key[e] != 0u;
                const unsigned msel = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    const int pos = base + __popc(msel & lt_mask);
                    orow[pos] = (int32_t)(it.gid0 + 32 * e + lane);
                    srow[pos] = key_score(key[e]);
                }
                base += __popc(msel);
            }
        } else {
            int eq_base = 0;
#pragma unroll
            for (int e = 0; e < PER; e++) {
                const bool is_eq = key[e] == T && key[e] != 0u;
                const unsigned meq = __ballot_sync(0xffffffffu, is_eq);
                const bool sel = key[e] > T || (is_eq && eq_base + __popc(meq & lt_mask) < need_eq);
                eq_base += __popc(meq);
                const unsigned msel = __ballot_sync(0xffffffffu, sel);
                if (sel) {
                    const int pos = base + __popc(msel & lt_mask);
                    orow[pos] = (int32_t)(it.gid0 + 32 * e + lane);
                    srow[pos] = key_score(key[e]);
                }
                base += __popc(msel);
            }
        }
    }
    for (int s2 = kk + lane; s2 < K; s2 += 32) {
        orow[s2] = -1;
        srow[s2] = -INFINITY;
    }
}

// ------------------------------------------------------------------ long key axis: candidate buffers

// A cut point of the n keys ck[0..n), all in [lo, hi] (K <= n), one warp, by a radix walk in digits of up to
// 8 bits with a 256-bin histogram per pass.  The walk starts at the highest bit in which lo and hi differ (the
// bits above it are the same in every key, so no pass is spent on them).
//   slack < 0: returns the K-th largest key T; `need_eq` receives how many entries equal to T belong to the top K
//              (the rest of the top K lies strictly above T), or n when every entry equal to T does.
//   slack >= 0: may stop early, at the first digit whose bin holding the K-th largest key has a lower edge L with
//              at most K + slack keys at or above it; returns L (at least K keys lie at or above it), with
//              `need_eq` = n (every key equal to L is kept).  Reaching the last digit gives the exact answer.
// Once the bin holding the K-th largest key has at most 256 keys, they are collected into the histogram's space and
// the rest of the exact answer is found bit by bit in registers.
__device__ uint32_t kth_search(const uint32_t *ck, int n, int K, uint32_t lo, uint32_t hi, int slack, uint32_t *hist,
                               int &need_eq)
{
    const int lane = threadIdx.x & 31;
    if (lo == hi) {  // every key is the same: the first K of them
        need_eq = K < n ? K : n;
        return lo;
    }
    int hb = 31 - __clz(lo ^ hi);                 // top bit of the current digit
    uint32_t prefix = hi & ~((2u << hb) - 1u);    // the bits above it (2u << 31 wraps to 0: no common bits)
    int need = K;  // rank of the wanted entry among those matching the prefix, counted from the top
#pragma unroll 1
    while (true) {
        const int lb = hb >= 7 ? hb - 7 : 0;      // digit bits lb .. hb
        const uint32_t wmask = (2u << (hb - lb)) - 1u;
        const uint32_t pmask = ~((2u << hb) - 1u);
#pragma unroll
        for (int q = 0; q < 8; q++) hist[32 * q + lane] = 0u;
        __syncwarp();
        for (int e0 = 0; e0 < n; e0 += 256) {  // eight loads in flight per lane
            uint32_t kk[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int e = e0 + 32 * u + lane;
                kk[u] = e < n ? ck[e] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; u++)
                if (e0 + 32 * u + lane < n && (kk[u] & pmask) == prefix) atomicAdd(hist + ((kk[u] >> lb) & wmask), 1u);
        }
        __syncwarp();
        // lane l owns bins 255 - 8 l .. 248 - 8 l (descending); an inclusive scan over lanes counts the entries
        // in bins at or above each lane's lowest bin
        uint32_t c[8], tot = 0u;
#pragma unroll
        for (int q = 0; q < 8; q++) {
            c[q] = hist[255 - 8 * lane - q];
            tot += c[q];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t before = incl - tot;
        const bool mine = before < (uint32_t)need && (uint32_t)need <= incl;
        const unsigned who = __ballot_sync(0xffffffffu, mine);
        int bin = 0;
        uint32_t above = 0u, cnt = 0u;
        if (mine) {
            uint32_t acc = before;
#pragma unroll
            for (int q = 0; q < 8; q++) {
                if (bin == 0 && acc + c[q] >= (uint32_t)need) {
                    bin = 256 + 255 - 8 * lane - q;  // +256: found
                    cnt = c[q];
                }
                if (bin == 0) acc += c[q];
            }
            above = acc;
            bin -= 256;
        }
        const int src = __ffs(who) - 1;
        bin = __shfl_sync(0xffffffffu, bin, src);
        above = __shfl_sync(0xffffffffu, above, src);
        cnt = __shfl_sync(0xffffffffu, cnt, src);
        prefix |= (uint32_t)bin << lb;
        need -= (int)above;
        __syncwarp();
        if (lb == 0) {
            need_eq = need == (int)cnt ? n : need;  // cnt entries equal the whole key
            return prefix;
        }
        // keys at or above the bin's lower edge: K - need + cnt
        if (slack >= 0 && (int)cnt - need <= slack) {
            need_eq = n;
            return prefix;
        }
        if (cnt <= 256u) {
            // few keys in the bin: collect them (into the histogram's space) and find the need-th largest bit by bit,
            // eight per lane in registers, instead of a histogram pass per remaining digit
            const uint32_t cmask = ~((1u << lb) - 1u);
            int base = 0;
            for (int e0 = 0; e0 < n; e0 += 128) {  // four chunks per step: the loads and ballots overlap
                uint32_t k[4];
                unsigned mk[4];
#pragma unroll
                for (int u = 0; u < 4; u++) k[u] = e0 + 32 * u + lane < n ? ck[e0 + 32 * u + lane] : 0u;
#pragma unroll
                for (int u = 0; u < 4; u++) mk[u] = __ballot_sync(0xffffffffu, e0 + 32 * u + lane < n && (k[u] & cmask) == prefix);
#pragma unroll
                for (int u = 0; u < 4; u++) {
                    if ((mk[u] >> lane) & 1u) hist[base + __popc(mk[u] & ((1u << lane) - 1u))] = k[u];
                    base += __popc(mk[u]);
                }
            }
            __syncwarp();
            uint32_t key[8];
#pragma unroll
            for (int q = 0; q < 8; q++) key[q] = 32 * q + lane < (int)cnt ? hist[32 * q + lane] : 0u;
            uint32_t t = prefix;  // every collected key is at or above it
#pragma unroll 1
            for (int bit = lb - 1; bit >= 0; bit--) {
                const uint32_t cc = t | (1u << bit);
                unsigned c2 = 0u;
#pragma unroll
                for (int q = 0; q < 8; q++) c2 += key[q] >= cc ? 1u : 0u;
                if ((int)__reduce_add_sync(0xffffffffu, c2) >= need) t = cc;
            }
            unsigned gt = 0u, eq = 0u;
#pragma unroll
            for (int q = 0; q < 8; q++) {
                gt += key[q] > t ? 1u : 0u;
                eq += 32 * q + lane < (int)cnt && key[q] == t ? 1u : 0u;
            }
            need_eq = need - (int)__reduce_add_sync(0xffffffffu, gt);
            if (need_eq == (int)__reduce_add_sync(0xffffffffu, eq)) need_eq = n;  // every entry equal to t is kept
            __syncwarp();  // the list is read before the next cut zeroes the histogram
            return t;
        }
        hb = lb - 1;
    }
}

// A slack cut point by sampling (slack >= 0): a key L of the buffer with between K and K + slack keys at or above
// it, or false.  The pivot is the sampled key whose rank among 128 keys spread over the buffer matches the window's
// middle (found bit by bit in registers, from the highest bit in which lo and hi differ); one counting pass over
// the buffer checks it (compares and a warp sum, no atomics), and a miss moves the sample rank by the miss scaled
// to the sample, three tries at most.  The caller falls back to the radix walk.
__device__ __forceinline__ bool sample_cut(const uint32_t *ck, int n, int K, int slack, uint32_t lo, uint32_t hi,
                                           uint32_t &L)
{
    const int lane = threadIdx.x & 31;
    uint32_t sk[4];
#pragma unroll
    for (int q = 0; q < 4; q++) sk[q] = ck[(int)(((long long)(32 * q + lane) * n) >> 7)];
    const int target = K + slack / 2;
    int r = (int)(((long long)target * 128 + n / 2) / n);  // the target's rank among the samples, from the top
    const int hb = lo == hi ? -1 : 31 - __clz(lo ^ hi);
    const uint32_t prefix = hb < 0 ? lo : (hi & ~((2u << hb) - 1u));
#pragma unroll 1
    for (int attempt = 0; attempt < 3; attempt++) {
        r = r < 1 ? 1 : (r > 128 ? 128 : r);
        // P: the r-th largest sample (the largest value with at least r samples at or above it)
        uint32_t P = prefix;
#pragma unroll 1
        for (int bit = hb; bit >= 0; bit--) {
            const uint32_t cand = P | (1u << bit);
            unsigned c = 0u;
#pragma unroll
            for (int q = 0; q < 4; q++) c += sk[q] >= cand ? 1u : 0u;
            if ((int)__reduce_add_sync(0xffffffffu, c) >= r) P = cand;
        }
        unsigned cnt = 0u;
        for (int e0 = 0; e0 < n; e0 += 256) {  // eight loads in flight per lane
            uint32_t kk[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int e = e0 + 32 * u + lane;
                kk[u] = e < n ? ck[e] : 0u;
            }
#pragma unroll
            for (int u = 0; u < 8; u++) cnt += (e0 + 32 * u + lane < n && kk[u] >= P) ? 1u : 0u;
        }
        const int C = (int)__reduce_add_sync(0xffffffffu, cnt);
        if (C >= K && C <= K + slack) {
            L = P;
            return true;
        }
        int step = (int)(((long long)(target - C) * 128) / n);
        if (step == 0) step = C < K ? 1 : -1;
        r += step;
    }
    return false;
}

// Cuts the candidate buffer (ascending key index, keys in [lo, hi]) back to the entries at or above a cut point
// (exactly the top K, ties to the lower index, when slack < 0, found by kth_search; otherwise every key at or above
// a point L with at least K of them: a sampled pivot with at most K + 512 of them, and never more than n - 2 NKEY,
// else kth_search's bin edge with at most K + slack), keeping the ascending order (stable in-place compaction).
// Returns the new count; `thr` receives T (or L): a later key can enter the top K only above it.
__device__ int cut_candidates(uint32_t *ck, uint16_t *ci, int n, int K, uint32_t lo, uint32_t hi, int slack,
                              uint32_t *hist, uint32_t &thr)
{
    const int lane = threadIdx.x & 31;
    int need_eq = n;
    uint32_t T = 0u;
    // the sampled pivot may keep up to 512 keys past K (fewer when two more tiles would not fit after the cut):
    // a wider window than the radix walk's costs a few more cuts but misses less often
    const int wide = n - 2 * NKEY - K < 512 ? n - 2 * NKEY - K : 512;
    if (!(slack >= 0 && sample_cut(ck, n, K, wide > slack ? wide : slack, lo, hi, T)))
        T = kth_search(ck, n, K, lo, hi, slack, hist, need_eq);
    const unsigned lt = (1u << lane) - 1u;
    int base = 0, eq_seen = 0;
    if (need_eq >= n) {
        // every key at or above T is kept (a slack cut's bin edge, or a cut that splits no tie): no tie count, and
        // eight chunks per step (the loop is bound by its shared-memory latency, not by its instructions).  A step
        // writes only at or below its own entries, all read before the step's barrier.
        for (int c0 = 0; c0 < n; c0 += 256) {
            uint32_t k[8];
            uint16_t ix[8];
            unsigned mk[8];
#pragma unroll
            for (int u = 0; u < 8; u++) {
                const int e = c0 + 32 * u + lane;
                k[u] = e < n ? ck[e] : 0u;
                ix[u] = e < n ? ci[e] : (uint16_t)0;
            }
#pragma unroll
            for (int u = 0; u < 8; u++) mk[u] = __ballot_sync(0xffffffffu, c0 + 32 * u + lane < n && k[u] >= T);
            __syncwarp();  // every lane has read its entries before any is overwritten
#pragma unroll
            for (int u = 0; u < 8; u++) {
                if ((mk[u] >> lane) & 1u) {
                    const int pos = base + __popc(mk[u] & lt);
                    ck[pos] = k[u];
                    ci[pos] = ix[u];
                }
                base += __popc(mk[u]);
            }
        }
        __syncwarp();
        thr = T;
        return base;
    }
    // four 32-entry chunks per step, loaded and decided before any is written (one warp has little else to
    // overlap its shared-memory latency with); writes land at or below the step's own entries
    for (int c0 = 0; c0 < n; c0 += 128) {
        uint32_t k[4];
        uint16_t ix[4];
        unsigned meq[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const int e = c0 + 32 * u + lane;
            k[u] = e < n ? ck[e] : 0u;
            ix[u] = e < n ? ci[e] : (uint16_t)0;
        }
#pragma unroll
        for (int u = 0; u < 4; u++) meq[u] = __ballot_sync(0xffffffffu, c0 + 32 * u + lane < n && k[u] == T);
        bool keep[4];
        unsigned mk[4];
#pragma unroll
        for (int u = 0; u < 4; u++) {
            const bool in = c0 + 32 * u + lane < n;
            const bool eq = ((meq[u] >> lane) & 1u) != 0u;
            keep[u] = in && (k[u] > T || (eq && eq_seen + __popc(meq[u] & lt) < need_eq));
            eq_seen += __popc(meq[u]);
            mk[u] = __ballot_sync(0xffffffffu, keep[u]);
        }
        __syncwarp();  // every lane has read its entries before any is overwritten
#pragma unroll
        for (int u = 0; u < 4; u++) {
            if (keep[u]) {
                const int pos = base + __popc(mk[u] & lt);
                ck[pos] = k[u];
                ci[pos] = ix[u];
            }
            base += __popc(mk[u]);
        }
        __syncwarp();
    }
    thr = T;
    return base;
}

// ------------------------------------------------------------------ the kernel

template <bool LONG>
__device__ __forceinline__ void score_body(const CUtensorMap *map_q, const CUtensorMap *map_k, const Args &a)
{
    using C = SC<LONG>;
    constexpr int NB = C::NB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sA = smem + C::OFF_A;
    unsigned char *sB = smem + C::OFF_B;
    float *sW = reinterpret_cast<float *>(smem + C::OFF_W);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + C::OFF_MISC);
    uint64_t *a_full = bars, *a_empty = bars + 4, *b_full = bars + 8, *b_empty = bars + 10;
    uint64_t *t_full = bars + 12, *t_empty = bars + 14, *mma_done = bars + 16;
    // short axis: score rows of an item, epilogue -> selection (sc_full / sc_empty, NSC each);
    // long axis: score tiles (ring_full / ring_empty, NRING each)
    uint64_t *x_full = bars + 17, *x_empty = bars + 17 + X_BARS;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC + 256);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 264);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    const bool sbhd = g.layout == CSA_SBHD;

    if (threadIdx.x == 0) {
        for (int i = 0; i < A_STAGES; i++) { mbar_init(a_full + i, 1); mbar_init(a_empty + i, 1); }
        for (int i = 0; i < 2; i++) {
            mbar_init(b_full + i, 1);
            mbar_init(b_empty + i, 1);
            mbar_init(t_full + i, 1);
            mbar_init(t_empty + i, 8);
        }
        if constexpr (LONG) {
            for (int i = 0; i < C::NRING; i++) {
                mbar_init(x_full + i, EPI / 32);
                mbar_init(x_empty + i, ROWS);
            }
        } else {
            for (int i = 0; i < C::NSC; i++) {
                mbar_init(x_full + i, EPI / 32);
                mbar_init(x_empty + i, ROWS);
            }
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(tmem_slot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = item_total(a);

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            // With two q_idx buffers an item's rows are requested as soon as their buffer is free: that buffer is
            // probed before every k-half load of the previous item, and waited for at the latest when the item
            // starts.  With one buffer they are requested when the previous item's MMAs have read it.
            int hs = 0, ai = 0, qi = 0;
            int last_hs[A_STAGES];
            for (int x = 0; x < A_STAGES; x++) last_hs[x] = -1;
            int last_qi[2] = {-1, -1};
            auto load_q = [&](const Item &it) {
                const int bb = qi % NB;
                mbar_expect_tx(b_full + bb, B_BUF);
                for (int k = 0; k < ROWS; k++) {
                    const long long row = k < it.n ? it.row[k] : it.row[0];
                    for (int kh = 0; kh < 2; kh++)
                        tma_load_3d(sB + bb * B_BUF + kh * B_HALF + k * (HI * 128), map_q, b_full + bb, kh * 64, 0,
                                    (int)row);
                }
                last_qi[bb] = qi;
                qi++;
            };
            // the next item with visible keys after item index i (or total)
            auto next_item = [&](int i, Item &nx) -> int {
                for (int j = i + gridDim.x; j < total; j += gridDim.x) {
                    nx = decode_item(a, j, total);
                    if (nx.vmax > 0) return j;
                }
                return total;
            };
            Item cur;
            int i = blockIdx.x;
            if (i < total) {
                cur = decode_item(a, i, total);
                if (cur.vmax == 0) i = next_item(i, cur);
            }
            while (i < total) {
                Item nxt;
                const int inext = next_item(i, nxt);
                if (qi == ai) {
                    wait_bar(b_empty + qi % NB, ((qi / NB) & 1) ^ 1, abort_flag, &g_tc_error, 1);
                    load_q(cur);
                }
                const int nt = (cur.vmax + NKEY - 1) / NKEY;
                for (int t = 0; t < nt; t++)
                    for (int kh = 0; kh < 2; kh++) {
                        if (NB > 1 && qi == ai + 1 && inext < total &&
                            mbar_test(b_empty + qi % NB, ((qi / NB) & 1) ^ 1))
                            load_q(nxt);
                        const int st = hs % A_STAGES;
                        wait_bar(a_empty + st, ((hs / A_STAGES) & 1) ^ 1, abort_flag, &g_tc_error, 2);
                        mbar_expect_tx(a_full + st, A_HALF);
                        if (sbhd)
                            tma_load_3d(sA + st * A_HALF, map_k, a_full + st, kh * 64, cur.b, t * NKEY);
                        else
                            tma_load_2d(sA + st * A_HALF, map_k, a_full + st, kh * 64, (int)(cur.key_y + t * NKEY));
                        last_hs[st] = hs;
                        hs++;
                    }
                ai++;
                i = inext;
                cur = nxt;
            }
            // our own copies must land before the CTA exits
            for (int st = 0; st < A_STAGES; st++)
                if (last_hs[st] >= 0) drain_bar(a_full + st, (last_hs[st] / A_STAGES) & 1, &g_tc_error);
            for (int bb = 0; bb < NB; bb++)
                if (last_qi[bb] >= 0) drain_bar(b_full + bb, (last_qi[bb] / NB) & 1, &g_tc_error);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issue (whole warp)
        // The warp runs the loop together (warp-uniform stage indices and descriptors); one elected lane issues
        // each MMA and commit.  Items are decoded lane-parallel (lane l: the CTA's item k + l), the loop reads
        // the tile count of item k by a shuffle.  A-stage ring position (st, parity aph).  After each K-half's
        // MMAs the next stage's full barrier and the next accumulator's empty barrier are probed in one
        // shared-memory round trip, which overlaps the MMAs just queued (a probe placed before them would leave
        // the tensor pipe idle for its latency); a probe that comes back false falls back to the bounded wait.
        int st = 0, ai = 0, tc = 0, k = 0, nt_lane = 0;
        uint32_t aph = 0;
        bool a_ready = false, t_ready = false;
        for (int i = blockIdx.x; i < total; i += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int il = i + lane * (int)gridDim.x;
                nt_lane = il < total ? (decode_item(a, il, total).vmax + NKEY - 1) / NKEY : 0;
            }
            const int nt = __shfl_sync(0xffffffffu, nt_lane, k & 31);
            if (nt == 0) continue;
            const int bb = ai % NB;
            wait_bar(b_full + bb, (ai / NB) & 1, abort_flag, &g_tc_error, 3);
            fence_after();
            const unsigned char *pb0 = sB + bb * B_BUF;
            for (int t = 0; t < nt; t++) {
                const int tb = tc & 1;
                if (!t_ready) wait_bar(t_empty + tb, ((tc >> 1) & 1) ^ 1, abort_flag, &g_tc_error, 4);
                fence_after();
                const uint32_t d = tmem + (uint32_t)(tb * NCOL);
#pragma unroll
                for (int kh = 0; kh < 2; kh++) {
                    if (!a_ready) wait_bar(a_full + st, aph, abort_flag, &g_tc_error, 5);
                    const int st1 = st + 1 == A_STAGES ? 0 : st + 1;
                    const uint32_t ph1 = st1 == 0 ? aph ^ 1u : aph;
                    fence_after();
                    const unsigned char *pa = sA + st * A_HALF;
                    const unsigned char *pb = pb0 + kh * B_HALF;
                    // four MMAs of K = 16 under one elect, then the stage's commit
                    mma4_ss_w(d, desc_kmajor(pa), 2, desc_kmajor(pb), 2, IDESC, kh != 0 ? 1u : 0u, su32(a_empty + st));
                    // probe the next stage (and, after the tile's last K-half, the next accumulator) now that the
                    // MMAs are queued: the round trip overlaps them
                    const uint32_t m = mbar_test2(a_full + st1, ph1, t_empty + (tb ^ 1), (((tc + 1) >> 1) & 1) ^ 1);
                    a_ready = (m & 1u) != 0u;
                    if (kh == 1) t_ready = (m & 2u) != 0u;
                    st = st1;
                    aph = ph1;
                }
                mma_commit_w(t_full + tb);
                tc++;
            }
            mma_commit_w(b_empty + bb);
            ai++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, &g_tc_error);
    } else if (warp < SEL_WARP0) {
        // ---------------------------------------------------------- epilogue (warps 2..9)
        const int e = warp - 2;           // 0..7
        const int quad = warp & 3;        // TMEM lane quadrant this warp may access
        const int half = e >> 2;          // rows {2 half, 2 half + 1}
        const int et = threadIdx.x - 64;  // 0..255
        int tc = 0, ic = 0;
        // w of this thread's (row, head) for the next item, loaded one item ahead
        auto w_of = [&](int i) -> float {
            if (i >= total) return 0.f;
            const long long row = item_row(a, i, total, et >> 6);
            return row >= 0 ? __ldg(a.w + row * HI + (et & 63)) : 0.f;
        };
        float w_next = w_of(blockIdx.x);
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            const Item it = decode_item(a, i, total);
            named_bar(1, EPI);  // every epilogue warp has finished the previous item's tiles (sW)
            sW[et] = w_next;
            w_next = w_of(i + gridDim.x);
            named_bar(1, EPI);
            float *scb = nullptr;
            int sb = 0;
            if constexpr (!LONG) {
                // this item's score rows go to buffer ic % NSC, free once the selection warps have read item ic - NSC
                sb = ic % C::NSC;
                const int su = ic / C::NSC;
                scb = reinterpret_cast<float *>(smem + C::OFF_SC) + sb * ROWS * NCMAX;
                wait_bar(x_empty + sb, (su & 1) ^ 1, abort_flag, &g_tc_error, 7);
            }
            const int nt = (it.vmax + NKEY - 1) / NKEY;
            for (int t = 0; t < nt; t++) {
                const int tb = tc & 1;
                wait_bar(t_full + tb, (tc >> 1) & 1, abort_flag, &g_tc_error, 6);
                fence_after();
                const int j = t * NKEY + quad * 32 + lane;
                float accs[2];
#pragma unroll
                for (int rr = 0; rr < 2; rr++) {
                    const int k = half * 2 + rr;
                    // independent partial sums over heads h % 4, two per paired FMA
                    float2 ac[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        float x[32];
                        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(tb * NCOL + k * HI + c * 32), x);
                        const float2 *wk = reinterpret_cast<const float2 *>(sW + k * HI + c * 32);
#pragma unroll
                        for (int h2 = 0; h2 < 16; h2++)
                            ac[h2 & 1] = fma2(wk[h2], make_float2(fmaxf(x[2 * h2], 0.f), fmaxf(x[2 * h2 + 1], 0.f)), ac[h2 & 1]);
                    }
                    accs[rr] = (ac[0].x + ac[0].y) + (ac[1].x + ac[1].y);  // heads (0 + 1) + (2 + 3) mod 4
                    if constexpr (!LONG) {
                        if (k < it.n && j < it.v[k]) scb[k * NCMAX + j] = accs[rr];
                    }
                }
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(t_empty + tb);
                if constexpr (LONG) {
                    // the tile's scores of rows 2 half, 2 half + 1 into ring slot tc % NRING (keys past a row's
                    // visible count are written too; the selection masks them)
                    const int slot = tc % C::NRING;
                    wait_bar(x_empty + slot, ((tc / C::NRING) & 1) ^ 1, abort_flag, &g_tc_error, 7);
                    float *ring = reinterpret_cast<float *>(smem + C::OFF_RING) + slot * ROWS * NKEY;
                    ring[(half * 2) * NKEY + quad * 32 + lane] = accs[0];
                    ring[(half * 2 + 1) * NKEY + quad * 32 + lane] = accs[1];
                    __syncwarp();
                    if (lane == 0) mbar_arrive(x_full + slot);
                }
                tc++;
            }
            if constexpr (!LONG) {
                // hand the item's score rows to the selection warps
                __syncwarp();
                if (lane == 0) mbar_arrive(x_full + sb);
            }
        }
    } else if constexpr (!LONG) {
        // ---------------------------------------------------------- selection (warps 10..17: two sets of four,
        // alternate items, one row per warp)
        const int k = (warp - SEL_WARP0) & 3, set = (warp - SEL_WARP0) >> 2;
        float *sSC = reinterpret_cast<float *>(smem + C::OFF_SC);
        int ic = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            if ((ic & 1) != set) continue;
            const Item it = decode_item(a, i, total);
            const int sb = ic % C::NSC, su = ic / C::NSC;
            wait_bar(x_full + sb, su & 1, abort_flag, &g_tc_error, 8);
            const float *sc = sSC + sb * ROWS * NCMAX + k * NCMAX;
            if (k < it.n) {
                const long long r = it.row[k];
                if (a.dump != nullptr && r >= a.dump_row0 && r < a.dump_row0 + a.dump_rows) {
                    float *out = a.dump + (r - a.dump_row0) * (long long)g.NC;
                    for (int jj = lane; jj < g.NC; jj += 32) out[jj] = jj < it.v[k] ? sc[jj] : -INFINITY;
                }
            }
            if (k < it.n && a.ids != nullptr) {
                select_row(a, it, k, sc, x_empty + sb);
            } else {
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty + sb);
            }
        }
    } else {
        // ---------------------------------------------------------- selection, long key axis (warps 10..13, one
        // row each): consume the score tiles of every item in order; keep the row's candidates in shared memory
        const int k = warp - SEL_WARP0;
        uint32_t *ck = reinterpret_cast<uint32_t *>(smem + C::OFF_CK) + k * C::CAP;
        uint16_t *ci = reinterpret_cast<uint16_t *>(smem + C::OFF_CI) + k * C::CAP;
        uint32_t *hist = reinterpret_cast<uint32_t *>(smem + C::OFF_HIST) + k * 256;
        const float *ringb = reinterpret_cast<const float *>(smem + C::OFF_RING);
        const int K = g.K;
        // an in-loop cut may keep up to cut_slack entries past the top K (the exact cut comes at the row's end);
        // it must still leave room for two tiles, so the slack shrinks for K near the largest K taken
        const int cut_slack = C::CAP - 2 * NKEY - K < 256 ? C::CAP - 2 * NKEY - K : 256;
        const unsigned lt = (1u << lane) - 1u;
        int tc = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Item it = decode_item(a, i, total);
            const int nt = (it.vmax + NKEY - 1) / NKEY;
            const bool present = k < it.n;
            const int v = present ? it.v[k] : 0;
            const long long r = present ? it.row[k] : -1;
            float *dump_row = (present && a.dump != nullptr && r >= a.dump_row0 && r < a.dump_row0 + a.dump_rows)
                                  ? a.dump + (r - a.dump_row0) * (long long)g.NC
                                  : nullptr;
            const bool select = present && a.ids != nullptr;
            int n = 0;
            uint32_t thr = 0u;  // a key enters only above this (0: every score, before the first cut)
            uint32_t klo = 0xffffffffu, khi = 0u;  // bounds of this lane's buffered keys (after a cut: [thr, max])
            auto cut = [&](int slack) {
                const uint32_t lo = __reduce_min_sync(0xffffffffu, klo), hi = __reduce_max_sync(0xffffffffu, khi);
                n = cut_candidates(ck, ci, n, K, lo, hi, slack, hist, thr);
                klo = thr;
                khi = hi;
            };
            for (int t = 0; t < nt; t++, tc++) {
                const int slot = tc % C::NRING;
                wait_bar(x_full + slot, (tc / C::NRING) & 1, abort_flag, &g_tc_error, 8);
                float s[4];
#pragma unroll
                for (int c = 0; c < 4; c++) s[c] = ringb[(slot * ROWS + k) * NKEY + 32 * c + lane];
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty + slot);
                if (dump_row != nullptr) {
#pragma unroll
                    for (int c = 0; c < 4; c++) {
                        const int j = t * NKEY + 32 * c + lane;
                        if (j < g.NC) dump_row[j] = j < v ? s[c] : -INFINITY;
                    }
                }
                if (!select) continue;
                if (n + NKEY > C::CAP) cut(cut_slack);
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    const int j = t * NKEY + 32 * c + lane;
                    const uint32_t key = score_key(s[c]);
                    const bool in = j < v && key > thr;
                    const unsigned m = __ballot_sync(0xffffffffu, in);
                    if (in) {
                        const int pos = n + __popc(m & lt);
                        ck[pos] = key;
                        ci[pos] = (uint16_t)j;
                        klo = min(klo, key);
                        khi = max(khi, key);
                    }
                    n += __popc(m);
                }
                __syncwarp();
            }
            if (dump_row != nullptr)
                for (int j = nt * NKEY + lane; j < g.NC; j += 32) dump_row[j] = -INFINITY;
            if (!select) continue;
            if (n > K) cut(-1);
            __syncwarp();
            int32_t *orow = a.ids + r * K;
            float *srow = a.selscore + r * K;
            for (int s2 = lane; s2 < n; s2 += 32) {
                orow[s2] = (int32_t)(it.gid0 + ci[s2]);
                srow[s2] = key_score(ck[s2]);
            }
            for (int s2 = n + lane; s2 < K; s2 += 32) {
                orow[s2] = -1;
                srow[s2] = -INFINITY;
            }
            __syncwarp();
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
}

__global__ void __launch_bounds__(SC<false>::THREADS, 1)
score_topk_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k, Args a)
{
    score_body<false>(&map_q, &map_k, a);
}

__global__ void __launch_bounds__(SC<true>::THREADS, 1)
score_topk_long_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_k, Args a)
{
    score_body<true>(&map_q, &map_k, a);
}

// THD: work-item offsets per segment, cu_g[b+1] = cu_g[b] + ceil(physical length / 4)
__global__ void build_cu_g_kernel(const int *cu_q, int nseg, int *cu_g)
{
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    int acc = 0;
    cu_g[0] = 0;
    for (int b = 0; b < nseg; b++) {
        int len = cu_q[b + 1] - cu_q[b];
        acc += len > 0 ? (len + ROWS - 1) / ROWS : 0;
        cu_g[b + 1] = acc;
    }
}

}  // namespace tcs

// ------------------------------------------------------------------ host side

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool tc_encode_bf16(CUtensorMap *m, const void *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                    const cuuint32_t *box)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_encode_f32(CUtensorMap *m, const float *base, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                   const cuuint32_t *box)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<float *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_score_supported(const Geo &g, bool bf16)
{
    const char *f = getenv("CSA_FORCE_GENERIC");
    if (f != nullptr && f[0] == '1') return false;
    if (!(bf16 && g.HI == tcs::HI && g.DI == tcs::DI && g.NC >= 1 && g.K >= 1 && g.rows > 0 && g.key_rows > 0))
        return false;
    // short key axis: whole score rows in shared memory; long: streamed tiles and candidate buffers
    return g.NC <= tcs::NCMAX || (g.NC <= tcs::LONG_NCMAX && g.K <= tcs::LONG_KMAX);
}

size_t tc_workspace_bytes(const Geo &g) { return sizeof(int) * (size_t)(g.layout == CSA_THD ? g.B + 1 : 1); }

bool tc_encode_q_map(CUtensorMap *m, const void *q_idx, const Geo &g)
{
    const cuuint64_t dims[3] = {(cuuint64_t)g.DI, (cuuint64_t)g.HI, (cuuint64_t)g.rows};
    const cuuint64_t strides[2] = {(cuuint64_t)g.DI * 2, (cuuint64_t)g.HI * g.DI * 2};
    const cuuint32_t box[3] = {64, (cuuint32_t)g.HI, 1};
    return tc_encode_bf16(m, q_idx, 3, dims, strides, box);
}

bool tc_encode_k_map(CUtensorMap *m, const void *k_idx, const Geo &g)
{
    if (g.layout == CSA_SBHD) {
        const cuuint64_t dims[3] = {(cuuint64_t)g.DI, (cuuint64_t)g.B, (cuuint64_t)g.nc};
        const cuuint64_t strides[2] = {(cuuint64_t)g.DI * 2, (cuuint64_t)g.B * g.DI * 2};
        const cuuint32_t box[3] = {64, 1, 128};
        return tc_encode_bf16(m, k_idx, 3, dims, strides, box);
    }
    const cuuint64_t dims[2] = {(cuuint64_t)g.DI, (cuuint64_t)g.key_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)g.DI * 2};
    const cuuint32_t box[2] = {64, 128};
    return tc_encode_bf16(m, k_idx, 2, dims, strides, box);
}

static cudaError_t launch_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                             int32_t *ids, float *selscore, float *dump, long long row0, long long nrows, void *ws,
                             cudaStream_t st)
{
    using namespace tcs;
    CUtensorMap mq, mk;
    if (!tc_encode_q_map(&mq, q_idx, g) || !tc_encode_k_map(&mk, k_idx, g)) return cudaErrorInvalidValue;
    Args a = {};  // every field set below; zero first so none is ever left unset
    a.g = g;
    a.w = w;
    a.ids = ids;
    a.selscore = selscore;
    a.dump = dump;
    a.dump_row0 = row0;
    a.dump_rows = nrows;
    a.cu_g = nullptr;
    a.total = 0;
    int upper;
    if (g.layout == CSA_THD) {
        int *cu_g = static_cast<int *>(ws);
        build_cu_g_kernel<<<1, 32, 0, st>>>(g.cu_q, g.B, cu_g);
        note_launches(1);
        a.cu_g = cu_g;
        upper = (g.rows + ROWS - 1) / ROWS + g.B;
    } else {
        a.total = g.B * ((g.S + ROWS - 1) / ROWS);
        upper = a.total;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int grid = upper < sms ? (upper > 0 ? upper : 1) : sms;
    if (g.NC <= NCMAX) {
        e = cudaFuncSetAttribute(score_topk_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SC<false>::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        score_topk_tc_kernel<<<grid, SC<false>::THREADS, SC<false>::SMEM_ALLOC, st>>>(mq, mk, a);
    } else {
        e = cudaFuncSetAttribute(score_topk_long_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SC<true>::SMEM_ALLOC);
        if (e != cudaSuccess) return e;
        score_topk_long_tc_kernel<<<grid, SC<true>::THREADS, SC<true>::SMEM_ALLOC, st>>>(mq, mk, a);
    }
    note_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_score_topk_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w,
                                 const __nv_bfloat16 *k_idx, int32_t *ids, float *selscore, void *ws,
                                 cudaStream_t st)
{
    return launch_tc(g, q_idx, w, k_idx, ids, selscore, nullptr, 0, 0, ws, st);
}

cudaError_t launch_score_dump_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w,
                                 const __nv_bfloat16 *k_idx, float *dump, long long row0, long long nrows, void *ws,
                                 cudaStream_t st)
{
    return launch_tc(g, q_idx, w, k_idx, nullptr, nullptr, dump, row0, nrows, ws, st);
}

}  // namespace csa
