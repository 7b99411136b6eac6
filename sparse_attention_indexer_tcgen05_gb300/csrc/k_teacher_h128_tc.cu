// k_teacher_h128_tc.cu -- the full-CSA teacher for 128 main-attention heads on the 5th-generation tensor cores
// (tcgen05 + TMEM), with the selected compressed keys gathered from L2.
//
// For query row t and head h ("[Bug] DSV4 unfused CSA indexer loss ..." (Megatron-LM issue #5776): "Paper
// reference" equations for Z_h and t_j; sec. 3, one denominator over the sliding window, the selected compressed
// keys and the sink; the proposal comment's factored form):
//   l_h = log(exp(a_h) + sum_{j in C} exp(c_hj) + sum_{r in W} exp(w_hr)),  c = sigma q.kv_c, w = sigma q.kv
//   T_j = sum_h exp(c_hj - l_h),   t_j = T_j / max(sum_{k in C} T_k, 1e-10)
//
// Mapping (bf16, H = 128, D = 64 .. 512 in steps of 64).  A work item is one query row: its 128 heads fill the
// MMA's M = 128 lanes.  The row's q is the A operand and lives in TMEM (D / 2 columns, at most 256), so shared
// memory holds only key tiles: D[h, key] = q[h] . key with N = 128 keys per tile (two 128-column fp32
// accumulators next to q), K = D in 64-wide K-blocks, one 16 KB shared-memory stage per K-block.
//   * one ring of twelve 16 KB stages carries, in order, each row's q, its window tiles and its compressed
//     tiles (both passes), filled by one group of four producer warps: with the dense loss every stage is a TMA
//     tile load; with the sparse loss every stage (the selected compressed keys, and with them the row's q and
//     window rows) is copied by all four warps with 16-byte cp.async copies, each written to its place in the
//     128-byte-swizzled K-major tile.  (TMA's gather4 moves 512 bytes per instruction and measured about a
//     tenth of the tile-load rate from L2, too slow for 2048 keys of 1 KB per row.)
//   pass 1: window tiles + compressed tiles -> per-head running sum against a reference maximum, then l_h with
//           the sink (or a given sink-and-window log-sum-exp);
//   pass 2: compressed tiles again -> exp(c - l_h) summed over the 128 heads into shared per-slot T;
//   the helper warp then L1-normalises the row and writes it out; inside the backward (sparse loss) it takes the
//   row's KL step from the normalised row instead (loss and g from the selected scores), so the teacher rows
//   never go to memory and no separate KL launch runs.
// Between rows the epilogue warps copy the next row's q from its ring stages into TMEM once the current row's
// last MMAs have completed (the accumulators are double-buffered, the q columns are not).
// Roles: warp 1 TMEM + MMA issue, warps 2..9 epilogue (two per TMEM lane quadrant), warp 10 per-row helper,
// warps 11..14 producers (warp 0 has no role).  Waits are bounded as in the other tensor-core kernels.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

#include <stdlib.h>

namespace csa {

static __device__ int g_teacher_h128_error = 0;

cudaError_t teacher_h128_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_teacher_h128_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_teacher_h128_error, &zero, sizeof(int));
}

namespace tw {

using namespace ptx;

constexpr int H = 128, NK = 128;
constexpr int MAXKB = 8;                        // D <= 512
constexpr int STG = NK * 64 * 2;                // 16 KB: one K-block of a 128-key tile (or of the row's q)
constexpr int NSTG = 12;                        // ring stages
constexpr int TWMAX = 2048;                     // teacher row width held in shared memory
constexpr int THREADS = 480;                    // 15 warps
constexpr int EPI = 256;                        // warps 2..9
constexpr int EPI_WARP0 = 2, HELPER_WARP = 10, PROD_WARP0 = 11, NPROD = 128;
constexpr int GRP = 4;                          // gathered stages committed and handed over together
constexpr uint32_t TMEM_COLS = 512;             // q (<= 256 columns) + two 128-column accumulators
constexpr uint32_t ACC0 = 256;
constexpr uint32_t IDESC = idesc_bf16(128, NK, false, false);  // A (q, TMEM) and B (keys) K-major

constexpr int OFF_RING = 0;                                     // NSTG stages
constexpr int OFF_T = OFF_RING + NSTG * STG;                    // 192 KB: per-slot T, 2 item parities
constexpr int OFF_MASK = OFF_T + 2 * TWMAX * 4;                 // slot-validity words, 2 x TWMAX / 32
constexpr int OFF_PART = OFF_MASK + 2 * (TWMAX / 32) * 4;       // (m, s) partials: 2 parities x 2 halves x 128
constexpr int OFF_MISC = OFF_PART + 2 * 2 * H * 8;
constexpr int OFF_KLE = OFF_MISC + 1024;                         // the KL step's exp(x - m) per slot, TWMAX
constexpr int SMEM = OFF_KLE + TWMAX * 4 + 1024;                 // + the 1024-byte alignment slack
static_assert(SMEM <= 232448, "teacher shared memory exceeds the per-block limit");

struct Args {
    Geo g;
    const float *sink;
    const int32_t *ids;
    const __nv_bfloat16 *q;      // cp.async sources (sparse loss): the query rows, the original KV rows and the
    const __nv_bfloat16 *kv;     // compressed keys
    const __nv_bfloat16 *kv_c;
    float *teacher;
    int nkb;                     // D / 64
    int kl;                      // the KL step runs in the helper warp (sparse loss, TW == K): the fields below
    const float *selscore;       // [rows][K] selected scores
    float *gslot;                // g by slot [rows][K], or null
    float *gkey;                 // g by key (row gd_row_of, stride ncp), or null
    int ncp;
    float *row_loss;             // [rows]
};

struct Item {
    long long row;
    int b, s, v;
    long long gid0, key_y;
    int wcount, p_lo;            // window positions [p_lo, p_lo + wcount)
    int nw, ncs, nct;            // window tiles, compressed slots / keys, compressed tiles
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

// Items are the query rows in reverse memory order (the latest positions, with the most keys, first).
__device__ Item decode(const Args &a, int i)
{
    const Geo &g = a.g;
    Item it;
    it.row = (long long)g.rows - 1 - i;
    const Row R = decode_row(g, it.row);
    it.b = R.b;
    it.s = R.s;
    it.v = R.v;
    it.gid0 = key_gid(g, R, 0);
    it.key_y = it.gid0;
    it.wcount = (R.v > 0 && g.window > 0) ? (R.s + 1 < g.window ? R.s + 1 : g.window) : 0;
    it.p_lo = R.s - it.wcount + 1;
    it.nw = (it.wcount + NK - 1) / NK;
    it.ncs = g.sparse ? (R.v < g.K ? R.v : g.K) : R.v;
    it.nct = (it.ncs + NK - 1) / NK;
    return it;
}

// tiles of a row: window, then compressed (pass 1), then compressed again (pass 2)
__device__ __forceinline__ int ntiles(const Item &it) { return it.v > 0 ? it.nw + 2 * it.nct : 0; }
// ring stages of a row: q, window tiles, both passes of the compressed tiles (one stage per K-block)
__device__ __forceinline__ int row_stages(const Args &a, const Item &it) { return a.nkb * (1 + it.nw + 2 * it.nct); }
// the id of slot s of the row (-1 past the K slots)
__device__ __forceinline__ int32_t slot_id(const Args &a, const Item &it, int s)
{
    return s < a.g.K ? __ldg(a.ids + it.row * a.g.K + s) : -1;
}
// a slot holding id is usable when id is a key of the row's segment within its visible range; its kv_c row then
// (row 0, never read for the loss, otherwise)
__device__ __forceinline__ long long id_key_row(const Args &a, const Item &it, int32_t id, bool &ok)
{
    const long long j = (long long)id - it.gid0;
    ok = !(id < 0 || j < 0 || j >= it.v);
    return ok ? key_row(a.g, (long long)id) : 0;
}

__global__ void __launch_bounds__(THREADS, 1)
teacher_h128_tc_kernel(const __grid_constant__ CUtensorMap map_q, const __grid_constant__ CUtensorMap map_kv,
                       const __grid_constant__ CUtensorMap map_kvc, Args a)
{
    extern __shared__ unsigned char smem_raw[];
    // aligned through an integer, unlike the other tensor-core kernels (smem_align1024): with the shared-window
    // form the compiler's register allocation for this kernel spills, and the kernel measured about 1 % slower
    unsigned char *smem = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    unsigned char *ring = smem + OFF_RING;
    float *sT = reinterpret_cast<float *>(smem + OFF_T);             // [2][TWMAX]
    uint32_t *sMask = reinterpret_cast<uint32_t *>(smem + OFF_MASK); // [2][TWMAX / 32]
    float2 *sPart = reinterpret_cast<float2 *>(smem + OFF_PART);     // [2][2][H]
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_MISC);
    // full: one arrival per stage (producer thread 0: a TMA load's expect_tx, or once a gathered stage's copies are
    // visible); empty: the MMA's commit, or the epilogue once it has copied a q stage
    uint64_t *full = bars, *empty = bars + NSTG;
    uint64_t *t_full = bars + 2 * NSTG, *t_empty = t_full + 2, *q_ready = t_full + 4, *mma_done = t_full + 5;
    uint64_t *mask_full = t_full + 6, *t_done = t_full + 8;          // [item parity]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC + 512);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 520);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    const bool sbhd = g.layout == CSA_SBHD;
    const int nkb = a.nkb;
    int *err = &g_teacher_h128_error;
    const int total = g.rows;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NSTG; i++) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, 1);
        }
        for (int i = 0; i < 2; i++) {
            mbar_init(t_full + i, 1);
            mbar_init(t_empty + i, EPI / 32);
            mbar_init(mask_full + i, 1);
            mbar_init(t_done + i, EPI / 32);
        }
        mbar_init(q_ready, 1);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 1) {
        // -------------------------------------------------------------------- MMA issue (whole warp)
        // Rows are decoded lane-parallel (lane l: the CTA's row k + l) and the loop reads the tile count of row k
        // by a shuffle.  Per row: skip its q stages (the epilogue copies them into TMEM), wait for q in
        // TMEM, then per tile and K-block four MMAs of K = 16 with A = q's columns of that K-block.
        // A barrier wait costs the issuing thread a shared-memory round trip even when the phase is complete (under
        // this kernel's shared-memory load, close to a K-block's 256 cycles of MMAs), so the warp waits as rarely as
        // the hand-over allows.  With the sparse loss the producers hand a row's stages over in groups of GRP counted
        // from the row's first stage, one thread arriving on a group's full barriers in order once every copy of the
        // group is visible; the arrivals release and the wait acquires, so a group's last barrier seen complete
        // shows the whole group complete, and the warp waits once per group (on its last stage; a group's stages
        // are at most GRP - 1 ahead, so that barrier cannot be two phases behind).  With the dense loss every stage
        // is a TMA load completing on its own, and each is waited for.  A wait placed at a group's (or a tile's)
        // start overlaps the MMAs still queued from the one before.
        const uint64_t ring_desc = desc_kmajor(ring);  // stage st: + st * STG / 16 in the address field
        int xs = 0, tc = 0, rc = 0, k = 0, nt_lane = 0;  // xs: absolute index of the next stage in the stream
        int ready_to = -1;                               // every stage up to this one is known full
        for (int i = blockIdx.x; i < total; i += gridDim.x, k++) {
            if ((k & 31) == 0) {
                const int il = i + lane * (int)gridDim.x;
                nt_lane = il < total ? ntiles(decode(a, il)) : 0;
            }
            const int nt = __shfl_sync(0xffffffffu, nt_lane, k & 31);
            if (nt == 0) continue;
            const int x0 = xs;                               // the row's first stage (its q)
            const int xend = x0 + nkb * (1 + nt);            // one past the row's last stage (nt = nw + 2 nct)
            xs += nkb;                                       // the row's q stages
            wait_bar(q_ready, rc & 1, abort_flag, err, 62);
            fence_after();
            for (int tt = 0; tt < nt; tt++) {
                const int tb = tc & 1;
                wait_bar(t_empty + tb, ((tc >> 1) & 1) ^ 1, abort_flag, err, 63);
                fence_after();
                const uint32_t d = tmem + ACC0 + (uint32_t)(tb * NK);
                for (int kb = 0; kb < nkb; kb++, xs++) {
                    if (xs > ready_to) {
                        int gl = xs;
                        if (g.sparse) {
                            gl = x0 + ((xs - x0) / GRP) * GRP + GRP - 1;
                            if (gl > xend - 1) gl = xend - 1;
                        }
                        wait_bar(full + gl % NSTG, (gl / NSTG) & 1, abort_flag, err, 64);
                        fence_after();
                        ready_to = gl;
                    }
                    const int st = xs % NSTG;
                    // four MMAs of K = 16 (A: q's columns of K-block kb; B: 32 bytes further per MMA), one commit
                    mma4_ts_w(d, tmem + (uint32_t)(kb * 32), 8, 16, ring_desc + (uint64_t)(st * (STG >> 4)), 2, IDESC,
                              kb != 0 ? 1u : 0u, su32(empty + st));
                }
                mma_commit_w(t_full + tb);
                tc++;
            }
            rc++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    } else if (warp >= EPI_WARP0 && warp < HELPER_WARP) {
        // ---------------------------------------------------------------- epilogue (8 warps)
        // Two warps per TMEM lane quadrant (warp % 4); warp half cq = (warp - 2) / 4 reads the 32-column chunks at
        // columns 32 cq and 32 cq + 64 of every tile, and copies q's K-blocks kb = cq (mod 2) into TMEM.
        const int quad = warp & 3, cq = (warp - EPI_WARP0) >> 2;
        const int h = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const float s2 = g.scale * 1.4426950408889634f;  // logits in log2 units: exp(c) = 2^(x * sigma * log2 e)
        const bool s2_pos = s2 > 0.f;
        auto col_of = [&](int c) { return cq * 32 + c * 64; };
        // copy the q of the row whose stages start at x0 into TMEM, release those stages, signal the MMA
        auto copy_q = [&](int x0) {
            for (int kb = cq; kb < nkb; kb += 2) {
                const int x = x0 + kb, st = x % NSTG;
                wait_bar(full + st, (x / NSTG) & 1, abort_flag, err, 66);
                const unsigned char *src = ring + st * STG;
                uint32_t v[32];
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const uint4 q4 = *reinterpret_cast<const uint4 *>(src + sw128_off((uint32_t)h, (uint32_t)c));
                    v[4 * c] = q4.x;
                    v[4 * c + 1] = q4.y;
                    v[4 * c + 2] = q4.z;
                    v[4 * c + 3] = q4.w;
                }
                tmem_st32(tmem + lane_off + (uint32_t)(kb * 32), v);
            }
            fence_before();
            named_bar(2, EPI);
            if (threadIdx.x == EPI_WARP0 * 32) {
                for (int kb = 0; kb < nkb; kb++) mbar_arrive(empty + (x0 + kb) % NSTG);
                mbar_arrive(q_ready);
            }
        };
        int tc = 0, ic = 0, x = 0;  // x: first stage of the current row
        bool first = true;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            const Item it = decode(a, i);
            const int nt = ntiles(it);
            const int ib = ic & 1;
            float *sTb = sT + ib * TWMAX;
            const uint32_t *sMaskb = sMask + ib * (TWMAX / 32);
            wait_bar(mask_full + ib, (ic >> 1) & 1, abort_flag, err, 67);
            if (nt > 0) {
                if (first) {
                    copy_q(x);
                    first = false;
                }
                const int x_next = x + row_stages(a, it);
                float m = -INFINITY, ssum = 0.f, ell = 0.f;
                float ell4[4] = {0.f, 0.f, 0.f, 0.f};  // l_h of heads g, g + 8, g + 16, g + 24 of the quadrant
                for (int tt = 0; tt < nt; tt++) {
                    const int tb = tc & 1;
                    wait_bar(t_full + tb, (tc >> 1) & 1, abort_flag, err, 68);
                    fence_after();
                    if (tt == nt - 1) {
                        // every MMA of this row has completed: the next row's q may replace it in TMEM
                        for (int j = i + gridDim.x; j < total; j += gridDim.x)
                            if (ntiles(decode(a, j)) > 0) {
                                copy_q(x_next);
                                break;
                            }
                    }
                    const bool win = tt < it.nw;
                    const bool pass2 = tt >= it.nw + it.nct;
                    const int t = win ? tt : (tt - it.nw) % it.nct;
                    if (pass2 && tt == it.nw + it.nct) {
                        // l_h (log2 units) from the two column halves, combined in a fixed order, and the sink
                        float2 *pp = sPart + ib * 2 * H;
                        pp[cq * H + h] = make_float2(m, ssum);
                        named_bar(1, EPI);
                        const float2 p0 = pp[h], p1 = pp[H + h];
                        const float ah = g.lse_nc != nullptr ? __ldg(g.lse_nc + it.row * H + h) * 1.4426950408889634f
                                                             : (g.no_sink ? -INFINITY : __ldg(a.sink + h) * 1.4426950408889634f);
                        const float mm = fmaxf(fmaxf(p0.x, p1.x), ah);
                        float S = 0.f;
                        if (mm != -INFINITY) {
                            if (p0.x != -INFINITY) S += p0.y * ex2(p0.x - mm);
                            if (p1.x != -INFINITY) S += p1.y * ex2(p1.x - mm);
                            if (ah != -INFINITY) S += ex2(ah - mm);
                        }
                        ell = mm + lg2(S);
#pragma unroll
                        for (int k4 = 0; k4 < 4; k4++) ell4[k4] = __shfl_sync(0xffffffffu, ell, (lane >> 2) + 8 * k4);
                    }
                    uint32_t mw[2];
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        const int c0 = t * NK + col_of(c);
                        if (win) mw[c] = range_bits(0, it.wcount - 1 - c0);
                        else if (g.sparse) mw[c] = c0 < it.ncs ? sMaskb[c0 >> 5] & range_bits(0, it.ncs - 1 - c0) : 0u;
                        else mw[c] = range_bits(0, it.ncs - 1 - c0);
                    }
                    // the accumulator goes back to the MMA as soon as this warp holds its columns in registers: the
                    // math below then overlaps the next tiles' MMAs (two accumulators alone would leave the MMA waiting
                    // for the epilogue's whole per-tile latency chain)
                    auto release = [&]() {
                        fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(t_empty + tb);
                    };
                    const uint32_t ca0 = tmem + lane_off + ACC0 + (uint32_t)(tb * NK + col_of(0));
                    const uint32_t ca1 = tmem + lane_off + ACC0 + (uint32_t)(tb * NK + col_of(1));
                    if ((mw[0] | mw[1]) == 0u) {
                        release();
                    } else if (!pass2) {
                        // running sum against a reference max, one 32-column chunk at a time; a chunk is re-based
                        // on its own max only when its sum leaves the safe range
                        uint32_t r0[32], r1[32];
                        if (mw[0] != 0u) tmem_ld32_async(ca0, r0);
                        else
#pragma unroll
                            for (int q = 0; q < 32; q++) r0[q] = 0u;
                        if (mw[1] != 0u) tmem_ld32_async(ca1, r1);
                        else
#pragma unroll
                            for (int q = 0; q < 32; q++) r1[q] = 0u;
                        tmem_wait_ld(r0);
                        tmem_wait_ld(r1);
                        release();
                        const float sc = s2_pos ? s2 : 1.f;
                        auto chunk1 = [&](const uint32_t (&r)[32], uint32_t mwc) {
                            float x[32];
                            if (s2_pos) {
                                if (mwc != 0xffffffffu) {
#pragma unroll
                                    for (int q = 0; q < 32; q++) x[q] = (mwc >> q) & 1u ? __uint_as_float(r[q]) : -INFINITY;
                                } else {
#pragma unroll
                                    for (int q = 0; q < 32; q++) x[q] = __uint_as_float(r[q]);
                                }
                            } else {
#pragma unroll
                                for (int q = 0; q < 32; q++) x[q] = (mwc >> q) & 1u ? __uint_as_float(r[q]) * s2 : -INFINITY;
                            }
                            auto chunk_max = [&]() -> float {
                                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                                for (int q = 0; q < 32; q++) mx[q & 3] = fmaxf(mx[q & 3], x[q]);
                                return fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])) * sc;
                            };
                            auto chunk_sum = [&]() -> float {
                                float2 sm[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
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
                        };
                        if (mw[0] != 0u) chunk1(r0, mw[0]);
                        if (mw[1] != 0u) chunk1(r1, mw[1]);
                    } else {
                        // pass 2 in the 16-lane shape: a thread holds heads g, g + 8, g + 16, g + 24 (g = lane / 4)
                        // of columns 8 p + 2 u + e (u = lane % 4); four heads are added in registers and the eight
                        // threads of a column set reduce-scatter over g
                        const int u4 = lane & 3, g8 = lane >> 2;
                        uint32_t a0[16], b0[16], a1[16], b1[16];
                        if (mw[0] != 0u) {
                            tmem_ld16x256_x4_async(ca0, a0);
                            tmem_ld16x256_x4_async(ca0 + (16u << 16), b0);
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; q++) a0[q] = b0[q] = 0u;
                        }
                        if (mw[1] != 0u) {
                            tmem_ld16x256_x4_async(ca1, a1);
                            tmem_ld16x256_x4_async(ca1 + (16u << 16), b1);
                        } else {
#pragma unroll
                            for (int q = 0; q < 16; q++) a1[q] = b1[q] = 0u;
                        }
                        tmem_wait_ld16(a0);
                        tmem_wait_ld16(b0);
                        tmem_wait_ld16(a1);
                        tmem_wait_ld16(b1);
                        release();
                        auto chunk2 = [&](const uint32_t (&ra)[16], const uint32_t (&rb)[16], uint32_t mwc, int c) {
                            const bool full = mwc == 0xffffffffu;
                            float s8[8];
#pragma unroll
                            for (int p4 = 0; p4 < 4; p4++) {
                                const int col = 8 * p4 + 2 * u4;
                                const bool e0m = full || ((mwc >> col) & 1u), e1m = full || ((mwc >> (col + 1)) & 1u);
                                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                                for (int k4 = 0; k4 < 4; k4++) {
                                    const uint32_t *r = k4 < 2 ? ra : rb;
                                    const int o = 4 * p4 + 2 * (k4 & 1);
                                    const float2 arg = fma2(make_float2(__uint_as_float(r[o]), __uint_as_float(r[o + 1])),
                                                            make_float2(s2, s2), make_float2(-ell4[k4], -ell4[k4]));
                                    const float e0 = ex2(arg.x), e1 = ex2(arg.y);
                                    acc = add2(acc, make_float2(e0m ? e0 : 0.f, e1m ? e1 : 0.f));
                                }
                                s8[2 * p4] = acc.x;
                                s8[2 * p4 + 1] = acc.y;
                            }
#pragma unroll
                            for (int hv = 4; hv >= 1; hv >>= 1) {
                                const int off = hv * 4;
                                const bool up = (lane & off) != 0;
#pragma unroll
                                for (int q = 0; q < hv; q++) {
                                    const float send = up ? s8[q] : s8[q + hv];
                                    const float keep = up ? s8[q + hv] : s8[q];
                                    s8[q] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                                }
                            }
                            const int j = t * NK + col_of(c) + 8 * (g8 >> 1) + 2 * u4 + (g8 & 1);
                            if (j < TWMAX && s8[0] != 0.f) atomicAdd(sTb + j, s8[0]);
                        };
                        if (mw[0] != 0u) chunk2(a0, b0, mw[0], 0);
                        if (mw[1] != 0u) chunk2(a1, b1, mw[1], 1);
                    }
                    tc++;
                }
                x = x_next;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(t_done + ib);
        }
    } else if (warp == HELPER_WARP) {
        // ---------------------------------------------------------------- per-row helper
        // For row ic (buffer ic & 1): zero its T row, build its slot-validity words (sparse loss), signal
        // mask_full; then, once the epilogue has summed row ic - 1 into the other buffer (t_done), L1-normalise
        // that row and write it out, or (a.kl) take the row's KL step from it.  Buffer reuse is ordered by this
        // warp's program order.
        //
        // KL step of a row ([BUG] sec. 2 excerpt; the arithmetic of the KL kernels): p = softmax of the selected
        // scores over the support C (the slots whose id is a visible key of the row, the validity words), t the
        // normalised teacher (0 past the first min(v, K) slots), L = sum_C t (log(t + eps) - log(p + eps)) and
        // g_s = f p_s (A - t_s / (p_s + eps)) with A = sum_C t p / (p + eps).  The scores' maximum and the
        // exponentials exp(x - m) (in sE) need no teacher, so they are taken before waiting for the epilogue.
        float *sE = reinterpret_cast<float *>(smem + OFF_KLE);
        constexpr int KLB = 16;  // score loads in flight per lane
        auto in_support = [&](const uint32_t *mk, int j) { return ((mk[j >> 5] >> (j & 31)) & 1u) != 0u; };
        auto writeout = [&](const Item &it, int icw) {
            const int ib = icw & 1;
            const int K = g.K;
            const uint32_t *mk = sMask + ib * (TWMAX / 32);
            const bool any = it.v > 0;  // otherwise no validity words were built: the support is empty
            float m = -INFINITY, z = 0.f;
            if (a.kl && any) {
                const float *xrow = a.selscore + it.row * K;
                for (int j0 = 0; j0 < K; j0 += 32 * KLB) {
                    float xv[KLB];
#pragma unroll
                    for (int k = 0; k < KLB; k++) {
                        const int j = j0 + 32 * k + lane;
                        xv[k] = j < K && in_support(mk, j) ? __ldg(xrow + j) : -INFINITY;
                    }
#pragma unroll
                    for (int k = 0; k < KLB; k++) {
                        const int j = j0 + 32 * k + lane;
                        if (j < K) sE[j] = xv[k];
                        m = fmaxf(m, xv[k]);
                    }
                }
                m = warp_max(m);
                if (m != -INFINITY) {
                    for (int j = lane; j < K; j += 32) {  // each lane rereads only its own slots
                        const float e = __expf(sE[j] - m);  // 0 off the support (x = -inf)
                        sE[j] = e;
                        z += e;
                    }
                    z = warp_sum(z);
                }
            }
            wait_bar(t_done + ib, (icw >> 1) & 1, abort_flag, err, 69);
            const float *tr = sT + ib * TWMAX;
            float part = 0.f;
            for (int j = lane; j < it.ncs; j += 32) part += tr[j];
            const float inv = 1.f / fmaxf(warp_sum(part), 1e-10f);
            if (!a.kl) {
                float *trow = a.teacher + it.row * g.TW;
                for (int j = lane; j < g.TW; j += 32) trow[j] = j < it.ncs ? tr[j] * inv : 0.f;
                return;
            }
            float *grow = a.gslot != nullptr ? a.gslot + it.row * K : nullptr;
            float *drow = a.gkey != nullptr ? a.gkey + gd_row_of(g, it.b, it.s, it.row) * a.ncp : nullptr;
            if (drow != nullptr) {  // zero the visible range (16-byte stores: the row stride is a multiple of 4)
                for (int j4 = lane; 4 * j4 < it.v; j4 += 32)
                    reinterpret_cast<float4 *>(drow)[j4] = make_float4(0.f, 0.f, 0.f, 0.f);
                __syncwarp();
            }
            if (m == -INFINITY) {  // empty support: no loss, no gradient
                if (grow != nullptr)
                    for (int j = lane; j < K; j += 32) grow[j] = 0.f;
                if (lane == 0) a.row_loss[it.row] = 0.f;
                return;
            }
            const float inv_z = 1.f / z;
            float A = 0.f, L = 0.f;
            for (int j = lane; j < K; j += 32) {
                if (!in_support(mk, j)) continue;
                const float p = sE[j] * inv_z;
                const float t = j < it.ncs ? tr[j] * inv : 0.f;
                A += t * p / (p + kKlEps);
                L += t * (logf(t + kKlEps) - logf(p + kKlEps));
            }
            A = warp_sum(A);
            L = warp_sum(L);
            const int32_t *irow = a.ids + it.row * K;
#pragma unroll 4
            for (int j = lane; j < K; j += 32) {
                const bool in = in_support(mk, j);
                const float p = sE[j] * inv_z;
                const float t = j < it.ncs ? tr[j] * inv : 0.f;
                const float gv = in ? g.factor * p * (A - t / (p + kKlEps)) : 0.f;
                if (grow != nullptr) grow[j] = gv;
                if (drow != nullptr && in) drow[__ldg(irow + j) - it.gid0] = gv;
            }
            if (lane == 0) a.row_loss[it.row] = L;
        };
        Item prev;
        int ic = 0;
        for (int i = blockIdx.x; i < total; i += gridDim.x, ic++) {
            const Item it = decode(a, i);
            const int ib = ic & 1;
            float4 *tz = reinterpret_cast<float4 *>(sT + ib * TWMAX);
            const int nz = (it.ncs + 3) / 4;
            for (int x = lane; x < nz; x += 32) tz[x] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (g.sparse && ntiles(it) > 0) {
                // the teacher reads the words of the first ncs slots; the KL step those of all K slots
                const int nmk = a.kl ? g.K : it.ncs;
                uint32_t *mk = sMask + ib * (TWMAX / 32);
                for (int w0 = 0; w0 < nmk; w0 += 256) {  // eight independent loads in flight per lane
                    int32_t idv[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) idv[k] = w0 + 32 * k + lane < nmk ? slot_id(a, it, w0 + 32 * k + lane) : -1;
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        bool ok;
                        id_key_row(a, it, idv[k], ok);
                        const unsigned bits = __ballot_sync(0xffffffffu, ok);
                        if (lane == 0 && w0 + 32 * k < nmk) mk[(w0 >> 5) + k] = bits;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(mask_full + ib);
            if (ic > 0) writeout(prev, ic - 1);
            prev = it;
        }
        if (ic > 0) writeout(prev, ic - 1);
    } else if (warp >= PROD_WARP0) {
        // ---------------------------------------------------------------- producers (one group, the whole stream)
        // The four producer warps walk every stage of the stream in order and are its only producer.  A barrier
        // tested by parity must never be two phases away from a thread that waits on it; the two loss modes meet
        // that differently.
        //   Dense loss: thread 0 alone issues every stage as a TMA tile load (its full barrier completes with the
        //     copy's bytes) and is the only thread that waits on the empty barriers, each in order.
        //   Sparse loss: every stage (the row's q, its window tiles and its selected compressed keys) is copied by
        //     all 128 threads with 16-byte cp.async copies, each to its chunk of the 128-byte-swizzled row of its
        //     matrix row: thread n takes chunk n % 8 of the rows n / 8 + 16 i (i = 0..7), so the eight consecutive
        //     threads of a row read its whole 128-byte segment and one warp instruction reads four rows.  Each
        //     thread waits on a stage's empty barrier before issuing its copies for it.  A stage is handed over
        //     (one arrival by thread 0) only after a named barrier of the four warps that every thread reaches
        //     once its copies for the stage have completed and been made visible to the async proxy, so no stage
        //     can be filled, let alone consumed, before every thread has passed its empty wait: no thread can
        //     fall a phase behind.  (With TMA stages filled by thread 0 alone, a lagging warp could find a stage
        //     already filled and consumed when it first tests the slot, and would then wait for good.)  The
        //     stages of a row go in groups of GRP, one commit group each; group j is handed over after group
        //     j + 1 has been issued (at most 2 GRP stages unsignalled, well inside the ring), and the row's last
        //     groups at its end.  The ids of each thread's eight key slots are loaded one tile ahead (the first
        //     gathered tile's at the row start), so that no tile waits for them.
        const int n = threadIdx.x - PROD_WARP0 * 32;
        if (g.sparse || n == 0) {
            const int D = g.D;
            int x = 0;
            bool tma_slot[NSTG];  // whether a slot's last stage was a TMA load of thread 0 (drained at the end)
            for (int st = 0; st < NSTG; st++) tma_slot[st] = false;
            auto wait_slot = [&](int y) { wait_bar(empty + y % NSTG, ((y / NSTG) & 1) ^ 1, abort_flag, err, 61); };
            // a TMA stage (dense loss, thread 0): wait for its slot, arm its full barrier, return the destination
            auto tma_dst = [&]() -> unsigned char * {
                const int st = x % NSTG;
                wait_slot(x);
                tma_slot[st] = true;
                mbar_expect_tx(full + st, STG);
                return ring + st * STG;
            };
            auto signal = [&](int y0, int y1) {  // stages [y0, y1): this thread's copies are complete
                fence_proxy_async();
                named_bar(3, NPROD);
                if (n == 0)
                    for (int y = y0; y < y1; y++) mbar_arrive(full + y % NSTG);
            };
            const int cc = n & 7, kq = n >> 3;
            for (int i = blockIdx.x; i < total; i += gridDim.x) {
                const Item it = decode(a, i);
                if (ntiles(it) == 0) continue;
                if (!g.sparse) {  // thread 0 alone
                    for (int kb = 0; kb < nkb; kb++, x++) tma_load_3d(tma_dst(), &map_q, full + x % NSTG, kb * 64, 0, (int)it.row);
                    for (int t = 0; t < it.nw; t++) {
                        const int p = it.p_lo + t * NK;
                        for (int kb = 0; kb < nkb; kb++, x++) {
                            unsigned char *dst = tma_dst();
                            if (sbhd) tma_load_3d(dst, &map_kv, full + x % NSTG, kb * 64, it.b, p);
                            else tma_load_2d(dst, &map_kv, full + x % NSTG, kb * 64, (int)(it.row - it.s + p));
                        }
                    }
                    for (int pass = 0; pass < 2; pass++)
                        for (int t = 0; t < it.nct; t++)
                            for (int kb = 0; kb < nkb; kb++, x++) {
                                unsigned char *dst = tma_dst();
                                if (sbhd) tma_load_3d(dst, &map_kvc, full + x % NSTG, kb * 64, it.b, t * NK);
                                else tma_load_2d(dst, &map_kvc, full + x % NSTG, kb * 64, (int)(it.key_y + t * NK));
                            }
                    continue;
                }
                int32_t idn[8];
                auto load_ids = [&](int t) {
#pragma unroll
                    for (int k = 0; k < 8; k++) idn[k] = slot_id(a, it, t * NK + kq + 16 * k);
                };
                load_ids(0);
                const int nu = 2 * it.nct;      // gathered tiles: both passes
                const int ntl = 1 + it.nw + nu;  // q, window tiles, gathered tiles
                int grp0 = x;                    // first stage of the group being issued
                int pend0 = -1, pend1 = -1;      // the issued group not yet handed over, [pend0, pend1)
                for (int tl = 0; tl < ntl; tl++) {
                    // this thread's eight source rows of the tile (matrix rows kq + 16 i), at chunk cc of K-block 0
                    const __nv_bfloat16 *src[8];
                    if (tl == 0) {  // q: head rows of the query row
#pragma unroll
                        for (int i = 0; i < 8; i++) src[i] = a.q + (it.row * H + kq + 16 * i) * D + cc * 8;
                    } else if (tl <= it.nw) {  // window positions p (past the window: the row's own, never read)
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            const int w = (tl - 1) * NK + kq + 16 * i;
                            const int p = w < it.wcount ? it.p_lo + w : it.s;
                            const long long mr = sbhd ? (long long)p * g.B + it.b : it.row - it.s + p;
                            src[i] = a.kv + mr * D + cc * 8;
                        }
                    } else {  // selected compressed keys
                        const int u = tl - 1 - it.nw;
#pragma unroll
                        for (int i = 0; i < 8; i++) {
                            bool ok;
                            src[i] = a.kv_c + id_key_row(a, it, idn[i], ok) * D + cc * 8;
                        }
                        if (u + 1 < nu) load_ids(u + 1 < it.nct ? u + 1 : u + 1 - it.nct);
                    }
                    for (int kb = 0; kb < nkb; kb++) {
                        wait_slot(x);
                        const int st = x % NSTG;
                        tma_slot[st] = false;
                        // row kq + 16 i, chunk cc; (kq + 16 i) & 7 == kq & 7
                        unsigned char *dst = ring + st * STG + kq * 128 + ((cc ^ (kq & 7)) << 4);
#pragma unroll
                        for (int i = 0; i < 8; i++) cp_async16(dst + i * 16 * 128, src[i] + kb * 64);
                        x++;
                        if (x - grp0 == GRP) {  // the group is complete: commit it, hand over the previous one
                            cp_async_commit();
                            if (pend0 >= 0) {
                                cp_async_wait<1>();
                                signal(pend0, pend1);
                            }
                            pend0 = grp0;
                            pend1 = x;
                            grp0 = x;
                        }
                    }
                }
                if (grp0 < x) cp_async_commit();  // a last, partial group
                cp_async_wait<0>();
                if (pend0 >= 0) signal(pend0, pend1);
                if (grp0 < x) signal(grp0, x);
            }
            // thread 0's TMA loads must land before the CTA exits (a slot whose last stage was gathered held an
            // earlier load only if that load was consumed, i.e. had landed)
            if (n == 0)
                for (int y = x - NSTG < 0 ? 0 : x - NSTG; y < x; y++)
                    if (tma_slot[y % NSTG]) drain_bar(full + y % NSTG, (y / NSTG) & 1, err);
        }
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace tw

// ------------------------------------------------------------------ host side

bool tc_teacher_h128_supported(const Geo &g, bool bf16)
{
    const char *f = getenv("CSA_FORCE_GENERIC");
    if (f != nullptr && f[0] == '1') return false;
    return bf16 && g.H == tw::H && g.D % 64 == 0 && g.D / 64 >= 1 && g.D / 64 <= tw::MAXKB && g.NC >= 1 &&
           g.K >= 1 && g.TW <= tw::TWMAX && g.rows > 0 && g.key_rows > 0;
}

cudaError_t launch_teacher_h128_tc(const Geo &g, const __nv_bfloat16 *q, const __nv_bfloat16 *kv,
                                   const __nv_bfloat16 *kv_c, const float *sink, const int32_t *ids, float *teacher,
                                   const TeacherKl *kl, cudaStream_t st)
{
    using namespace tw;
    CUtensorMap mq, mkv, mkc;
    // q as [rows][H][D] with a 64 x 128 x 1 box (one K-block of a row's 128 heads)
    {
        const cuuint64_t dims[3] = {(cuuint64_t)g.D, (cuuint64_t)g.H, (cuuint64_t)g.rows};
        const cuuint64_t strides[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.H * g.D * 2};
        const cuuint32_t box[3] = {64, (cuuint32_t)g.H, 1};
        if (!tc_encode_bf16(&mq, q, 3, dims, strides, box)) return cudaErrorInvalidValue;
    }
    // kv_c as tiles of 128 keys (dense loss); kv as tiles of 128 positions (window)
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
    if (g.window == 0) {  // no window tile is ever loaded: the kv map is never used
        mkv = mkc;
    } else if (g.layout == CSA_SBHD) {
        const cuuint64_t dkv[3] = {(cuuint64_t)g.D, (cuuint64_t)g.B, (cuuint64_t)g.S};
        const cuuint64_t skv[2] = {(cuuint64_t)g.D * 2, (cuuint64_t)g.B * g.D * 2};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)NK};
        if (!tc_encode_bf16(&mkv, kv, 3, dkv, skv, box)) return cudaErrorInvalidValue;
    } else {
        const cuuint64_t dkv[2] = {(cuuint64_t)g.D, (cuuint64_t)g.rows};
        const cuuint64_t s1[1] = {(cuuint64_t)g.D * 2};
        const cuuint32_t box[2] = {64, (cuuint32_t)NK};
        if (!tc_encode_bf16(&mkv, kv, 2, dkv, s1, box)) return cudaErrorInvalidValue;
    }
    Args a = {};  // every field set below; zero first so none is ever left unset
    a.g = g;
    a.sink = sink;
    a.ids = ids;
    a.q = q;
    a.kv = kv;
    a.kv_c = kv_c;
    a.teacher = teacher;
    a.nkb = g.D / 64;
    if (kl != nullptr) {  // the KL step needs the sparse support and one teacher slot per selected slot
        if (!g.sparse || g.TW != g.K || kl->selscore == nullptr || kl->row_loss == nullptr) return cudaErrorInvalidValue;
        a.kl = 1;
        a.selscore = kl->selscore;
        a.gslot = kl->gslot;
        a.gkey = kl->gkey;
        a.ncp = kl->ncp;
        a.row_loss = kl->row_loss;
    }
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(teacher_h128_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const int grid = g.rows < sms ? g.rows : sms;
    teacher_h128_tc_kernel<<<grid, THREADS, SMEM, st>>>(mq, mkv, mkc, a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
