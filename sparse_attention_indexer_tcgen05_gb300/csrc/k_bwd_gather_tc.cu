// k_bwd_gather_tc.cu -- the row-owner half of the indexer backward (dQ_idx, dW) over each row's selected keys only,
// on the 5th-generation tensor cores (tcgen05 + TMEM), for key axes too long for dense key tiles to pay.
//
// For query row t and its selected keys s (the ids; g_ts = dloss/dI_ts from the KL step, by slot):
//   dQ'[t,j] = sum_s g_ts 1[x_tjs > 0] k_idx[s],   dQ_idx[t,j] = w[t,j] dQ'[t,j],   dW[t,j] = q_idx[t,j] . dQ'[t,j]
// with x_tjs = q_idx[t,j] . k_idx[s] ("[Bug] DSV4 unfused CSA indexer loss ..." (Megatron-LM issue #5776), the
// proposal comment: gradients only for the indexer Q, weights and K; "Megatron-LM PR #8539" item 1: global ids).
//
// Mapping (bf16, H_I = 64, D_I = 128).  A work item is one query row; its selected keys, in slot order, go in tiles
// of 128.  Per tile:
//   MMA1  X[key, h]    = k . q^T      M = 128 keys (A: the gathered k tile, K-major), N = 64 heads (B: the row's
//                                      q_idx, K-major), K = 128 d; fp32 in TMEM (two 64-column buffers);
//   epilogue           G'[key, h] = g_key 1[x > 0] in bf16, written to shared memory as an MN-major B operand
//                      (one 128-byte row of 64 heads per key, 128-byte swizzle); g is read by slot, so keys off the
//                      row's support (g = 0) add nothing;
//   MMA2  dQ'^T[d, h] += k^T . G'     M = 128 d (A: the same k tile read MN-major), N = 64 heads (B: G'), K = 128
//                                      keys; fp32 in TMEM (64 columns), accumulated over the row's tiles;
// and at the row's end the epilogue reads dQ'^T (lane = d), writes dQ_idx = w dQ' and reduces dW = q . dQ' over d.
// The epilogue also stores, per (row, slot), the 64 signs of x (bit h: x[key, h] > 0) for the key-owner kernel,
// which then forms its G = g w 1[x > 0] without recomputing x.
// The k rows of a tile are gathered by four producer warps with 16-byte cp.async copies (16 threads per 256-byte
// row, coalesced), each chunk written to its place in the swizzled tile; tiles are handed to the MMA one tile late
// (after the next tile's copies are issued) once every thread's copies have completed and been made visible to
// the async proxy.  The row's q_idx comes by TMA.
// Roles: warps 0..3 producers (thread 0 also issues the q TMA loads), warps 4..7 epilogue (one per TMEM lane
// quadrant), warp 8 TMEM allocation + MMA issue.  Every barrier has one waiting role that sees each of its phases;
// waits are bounded as in the other tensor-core kernels.
#include "csa_tc.cuh"
#include "tc_ptx.cuh"

#include <stdlib.h>

namespace csa {

static __device__ int g_bwd_gather_error = 0;

cudaError_t bwd_gather_read_clear_error(int *flag)
{
    cudaError_t e = cudaMemcpyFromSymbol(flag, g_bwd_gather_error, sizeof(int));
    if (e != cudaSuccess || *flag == 0) return e;
    int zero = 0;
    return cudaMemcpyToSymbol(g_bwd_gather_error, &zero, sizeof(int));
}

namespace bwg {

using namespace ptx;

constexpr int HI = 64, DI = 128, NKEY = 128;
constexpr int KHALF = NKEY * 64 * 2;            // 16 KB: 128 keys x 64 d
constexpr int KT = 2 * KHALF;                   // 32 KB: a gathered k tile, two 64-wide K-halves
constexpr int NKT = 5;                          // k tiles in the ring
constexpr int QHALF = HI * 64 * 2;              // 8 KB: 64 heads x 64 d
constexpr int QT = 2 * QHALF;                   // 16 KB: a row's q_idx
constexpr int GT = NKEY * HI * 2;               // 16 KB: G' [128 keys][64 heads] bf16
constexpr int THREADS = 288;                    // 9 warps
constexpr int NPROD = 128, EPI = 128;
constexpr int EPI_WARP0 = 4, MMA_WARP = 8;
constexpr int NX = 2;                           // X accumulators and G' tiles in flight (MMA2 runs one tile behind)
constexpr uint32_t TMEM_COLS = 256;             // X buffers at 0, 64; dQ'^T at 192
constexpr uint32_t IDESC_X = idesc_bf16(128, HI, false, false);   // A = k tile, B = q, both K-major
constexpr uint32_t IDESC_DQ = idesc_bf16(128, HI, true, true);    // A = k tile read MN-major, B = G' MN-major

constexpr int OFF_K = 0;                                         // NKT x 32 KB
constexpr int OFF_Q = OFF_K + NKT * KT;                          // 160 KB: 2 x 16 KB
constexpr int OFF_G = OFF_Q + 2 * QT;                            // 192 KB: NX x 16 KB
constexpr int OFF_W = OFF_G + NX * GT;                           // 224 KB: w rows, 2 x 64 fp32
constexpr int OFF_DW = OFF_W + 2 * HI * 4;                       // dW partials, 4 warps x 64 fp32
constexpr int OFF_MISC = OFF_DW + 4 * HI * 4;                    // barriers (< 256 B), TMEM slot, abort flag
constexpr int SMEM = OFF_MISC + 512 + 1024;                      // + slack to align the base to 1024 B
static_assert((2 * NKT + 4 + 4 * NX + 3) * 8 <= 256, "gathered row-owner barriers overlap the TMEM slot");
static_assert(SMEM <= 232448, "gathered row-owner shared memory exceeds the per-block limit");

struct Args {
    Geo g;
    const __nv_bfloat16 *k_idx;   // gather source
    const float *w;
    const int32_t *ids;
    const float *gslot;           // dloss/dI by slot [rows][K]
    __nv_bfloat16 *dq;
    float *dw;
    unsigned long long *sgn;      // [rows][K]: bit h set when x > 0 for head h (0 for slots without a key)
};

struct Item {
    long long row;
    long long gid0;
    int v, ncs, nt;               // visible keys, slots in use (min(K, v)), key tiles
};

// Items are the query rows in reverse memory order (the latest positions, with the most keys, first).
__device__ __forceinline__ Item decode(const Args &a, int i)
{
    const Geo &g = a.g;
    Item it;
    it.row = (long long)g.rows - 1 - i;
    const Row R = decode_row(g, it.row);
    it.gid0 = key_gid(g, R, 0);
    it.v = R.v;
    it.ncs = R.v < g.K ? R.v : g.K;
    it.nt = (it.ncs + NKEY - 1) / NKEY;
    return it;
}

// memory row in k_idx of the key in slot s (row 0 when the slot holds no usable key: its g is 0)
__device__ __forceinline__ long long slot_key_row(const Args &a, const Item &it, int s)
{
    const Geo &g = a.g;
    if (s >= g.K) return 0;
    const int32_t id = __ldg(a.ids + it.row * g.K + s);
    const long long j = (long long)id - it.gid0;
    if (id < 0 || j < 0 || j >= it.v) return 0;
    return key_row(g, (long long)id);
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

__global__ void __launch_bounds__(THREADS, 1)
dq_dw_gather_tc_kernel(const __grid_constant__ CUtensorMap map_q, Args a)
{
    // the key-owner kernel reads nothing this one writes: let it take each SM this kernel leaves
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_align1024(smem_raw);
    unsigned char *sK = smem + OFF_K;
    unsigned char *sQ = smem + OFF_Q;
    unsigned char *sG = smem + OFF_G;
    float *sW = reinterpret_cast<float *>(smem + OFF_W);
    float *sDW = reinterpret_cast<float *>(smem + OFF_DW);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + OFF_MISC);
    uint64_t *k_full = bars, *k_empty = bars + NKT;
    uint64_t *q_full = bars + 2 * NKT, *q_empty = q_full + 2;
    uint64_t *x_full = q_full + 4, *x_empty = x_full + NX, *g_full = x_empty + NX, *g_empty = g_full + NX;
    uint64_t *dq_full = g_empty + NX, *dq_empty = dq_full + 1, *mma_done = dq_full + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + OFF_MISC + 256);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + OFF_MISC + 264);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Geo &g = a.g;
    int *err = &g_bwd_gather_error;
    const int total = g.rows;
    const int K = g.K;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NKT; i++) { mbar_init(k_full + i, 1); mbar_init(k_empty + i, 1); }
        for (int i = 0; i < 2; i++) {
            mbar_init(q_full + i, 1);
            mbar_init(q_empty + i, 2);            // the MMA's last X group of the row, and the epilogue's dW
        }
        for (int i = 0; i < NX; i++) {
            mbar_init(x_full + i, 1);
            mbar_init(x_empty + i, EPI / 32);
            mbar_init(g_full + i, EPI / 32);
            mbar_init(g_empty + i, 1);
        }
        mbar_init(dq_full, 1);
        mbar_init(dq_empty, EPI / 32);
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        init_fence();
    }
    if (warp == MMA_WARP) tmem_alloc(tmem_slot, TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tX = tmem, tDQ = tmem + 192;

    if (warp < EPI_WARP0) {
        // ---------------------------------------------------------------- producers
        // Thread n copies 16-byte chunk n % 16 (K-half (n % 16) / 8, chunk n % 8) of the keys in slots n / 16 + 8 i
        // (i = 0..15) of every tile: the 16 consecutive threads of a slot read its whole 256-byte row.  The CTA's
        // (row, tile) sequence is walked as one stream; the ids of the next tile's slots are loaded one tile ahead
        // (turned into k_idx rows only when used, so the loads never stall the current tile).  One commit group
        // per tile; tile j is handed over after tile j + 1's copies are issued, and the last one at the end.
        const int n = threadIdx.x;
        const int c16 = n & 15, half = c16 >> 3, cc = c16 & 7, kq = n >> 4;
        int x = 0, rq = 0;       // tiles issued, rows whose q was loaded
        int pend = -1;           // the issued tile not yet handed over
        auto signal = [&](int y) {
            fence_proxy_async();
            named_bar(1, NPROD);
            if (n == 0) mbar_arrive(k_full + y % NKT);
        };
        auto next_row = [&](int from, Item &out) -> int {  // the next row with keys at or after item index from
            for (int j = from; j < total; j += gridDim.x) {
                out = decode(a, j);
                if (out.nt > 0) return j;
            }
            return total;
        };
        int32_t id_next[16];     // raw ids of the next tile's slots (-1 past K)
        auto load_ids = [&](const Item &it, int t) {
#pragma unroll
            for (int i2 = 0; i2 < 16; i2++) {
                const int sl = t * NKEY + kq + 8 * i2;
                id_next[i2] = sl < K ? __ldg(a.ids + it.row * K + sl) : -1;
            }
        };
        Item cur;
        int i = next_row(blockIdx.x, cur), t = 0;
        if (i < total) load_ids(cur, 0);
        while (i < total) {
            if (t == 0) {
                if (n == 0) {  // the row's q_idx (both K-halves) by TMA into buffer rq & 1
                    const int qb = rq & 1;
                    wait_bar(q_empty + qb, ((rq >> 1) & 1) ^ 1, abort_flag, err, 51);
                    mbar_expect_tx(q_full + qb, QT);
                    for (int kh = 0; kh < 2; kh++)
                        tma_load_3d(sQ + qb * QT + kh * QHALF, &map_q, q_full + qb, kh * 64, 0, (int)cur.row);
                }
                rq++;
            }
            // this tile's source rows (a slot without a usable key reads row 0; its g is 0)
            const __nv_bfloat16 *src[16];
#pragma unroll
            for (int i2 = 0; i2 < 16; i2++) {
                const long long j = (long long)id_next[i2] - cur.gid0;
                const long long kr = (id_next[i2] >= 0 && j >= 0 && j < cur.v) ? key_row(g, (long long)id_next[i2]) : 0;
                src[i2] = a.k_idx + kr * DI + half * 64 + cc * 8;
            }
            // the next tile: this row's next, or the next row's first
            Item nxt = cur;
            int inext = i, tn = t + 1;
            if (tn == cur.nt) {
                inext = next_row(i + gridDim.x, nxt);
                tn = 0;
            }
            if (inext < total) load_ids(nxt, tn);
            const int st = x % NKT;
            wait_bar(k_empty + st, ((x / NKT) & 1) ^ 1, abort_flag, err, 52);
            // row kq + 8 i of K-half `half`, chunk cc; (kq + 8 i) & 7 == kq & 7
            unsigned char *dst = sK + st * KT + half * KHALF + kq * 128 + ((cc ^ (kq & 7)) << 4);
#pragma unroll
            for (int i2 = 0; i2 < 16; i2++) cp_async16(dst + i2 * 8 * 128, src[i2]);
            cp_async_commit();
            if (pend >= 0) {
                cp_async_wait<1>();
                signal(pend);
            }
            pend = x;
            x++;
            i = inext;
            cur = nxt;
            t = tn;
        }
        cp_async_wait<0>();
        if (pend >= 0) signal(pend);
        if (n == 0)  // our own q copies must land before the CTA exits
            for (int r = rq - 2 < 0 ? 0 : rq - 2; r < rq; r++) drain_bar(q_full + (r & 1), (r >> 1) & 1, err);
    } else if (warp < MMA_WARP) {
        // ---------------------------------------------------------------- epilogue (4 warps, one per lane quadrant)
        const int quad = warp & 3, et = threadIdx.x - EPI_WARP0 * 32;
        const int r_lane = quad * 32 + lane;          // TMEM lane: a key of the tile (X), or a d (dQ'^T)
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int xc = 0, rq = 0, rc = 0;                   // tiles converted, rows with tiles, rows
        for (int i = blockIdx.x; i < total; i += gridDim.x, rc++) {
            const Item it = decode(a, i);
            const long long row = it.row;
            if (it.nt == 0) {  // no key: dQ_idx and dW are zero
                for (int e = et; e < HI * DI / 8; e += EPI)
                    reinterpret_cast<uint4 *>(a.dq + row * (HI * DI))[e] = make_uint4(0, 0, 0, 0);
                if (et < HI) a.dw[row * HI + et] = 0.f;
                continue;
            }
            const int qb = rq & 1;
            if (et < HI) sW[qb * HI + et] = __ldg(a.w + row * HI + et);
            const float *grow = a.gslot + row * K;
            // g of this key's slot, loaded one tile ahead
            float g_next = r_lane < K ? __ldg(grow + r_lane) : 0.f;
            for (int t = 0; t < it.nt; t++, xc++) {
                const int xb = xc % NX;
                const float gk = g_next;
                const int s1 = (t + 1) * NKEY + r_lane;
                if (t + 1 < it.nt) g_next = s1 < K ? __ldg(grow + s1) : 0.f;
                wait_bar(x_full + xb, (xc / NX) & 1, abort_flag, err, 53);
                fence_after();
                uint32_t xr[64];
                tmem_ld32_async(tX + lane_off + (uint32_t)(xb * 64), *reinterpret_cast<uint32_t(*)[32]>(xr));
                tmem_ld32_async(tX + lane_off + (uint32_t)(xb * 64 + 32), *reinterpret_cast<uint32_t(*)[32]>(xr + 32));
                tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(xr));
                tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(xr + 32));
                fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(x_empty + xb);
                const int sl = t * NKEY + r_lane;
                if (sl < K) {
                    unsigned long long m = 0ull;
#pragma unroll
                    for (int h = 0; h < HI; h++) m |= (unsigned long long)(__uint_as_float(xr[h]) > 0.f) << h;
                    a.sgn[row * K + sl] = gk != 0.f ? m : 0ull;
                }
                // G' of this key over the 64 heads into buffer xb, row r_lane of the MN-major tile
                wait_bar(g_empty + xb, ((xc / NX) & 1) ^ 1, abort_flag, err, 54);
                unsigned char *gt = sG + xb * GT + r_lane * 128;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    uint4 o;
                    o.x = pack_bf16(__uint_as_float(xr[8 * c + 0]) > 0.f ? gk : 0.f, __uint_as_float(xr[8 * c + 1]) > 0.f ? gk : 0.f);
                    o.y = pack_bf16(__uint_as_float(xr[8 * c + 2]) > 0.f ? gk : 0.f, __uint_as_float(xr[8 * c + 3]) > 0.f ? gk : 0.f);
                    o.z = pack_bf16(__uint_as_float(xr[8 * c + 4]) > 0.f ? gk : 0.f, __uint_as_float(xr[8 * c + 5]) > 0.f ? gk : 0.f);
                    o.w = pack_bf16(__uint_as_float(xr[8 * c + 6]) > 0.f ? gk : 0.f, __uint_as_float(xr[8 * c + 7]) > 0.f ? gk : 0.f);
                    *reinterpret_cast<uint4 *>(gt + ((c ^ (r_lane & 7)) << 4)) = o;
                }
                fence_proxy_async();  // generic-proxy writes of G', read by the MMA
                __syncwarp();
                if (lane == 0) mbar_arrive(g_full + xb);
            }
            // ---- the row's end: dQ'^T (lane = d, column = head)
            wait_bar(dq_full, rq & 1, abort_flag, err, 55);
            fence_after();
            uint32_t vr[64];
            tmem_ld32_async(tDQ + lane_off, *reinterpret_cast<uint32_t(*)[32]>(vr));
            tmem_ld32_async(tDQ + lane_off + 32u, *reinterpret_cast<uint32_t(*)[32]>(vr + 32));
            tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(vr));
            tmem_wait_ld(*reinterpret_cast<uint32_t(*)[32]>(vr + 32));
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(dq_empty);
            named_bar(2, EPI);  // the w row is in
            const int d = r_lane;
            const float *wr = sW + qb * HI;
            __nv_bfloat16 *dqr = a.dq + row * (HI * DI) + d;
            // q_idx[h][d] from the row's q tile (K-major, 128-byte swizzle: K-half d / 64, chunk (d % 64) / 8)
            const unsigned char *qt = sQ + qb * QT + (d >> 6) * QHALF;
            const uint32_t qc = (uint32_t)((d & 63) >> 3), qe = (uint32_t)(d & 7);
            float p[64];
#pragma unroll
            for (int h = 0; h < HI; h++) {
                const float dqv = __uint_as_float(vr[h]);
                dqr[h * DI] = __float2bfloat16_rn(wr[h] * dqv);
                const __nv_bfloat16 qv = *reinterpret_cast<const __nv_bfloat16 *>(qt + sw128_off((uint32_t)h, qc) + 2 * qe);
                p[h] = __bfloat162float(qv) * dqv;
            }
            // dW = sum over d: reduce-scatter over the warp's 32 lanes (lane l ends with heads 2 l, 2 l + 1), then
            // the four warps' partials in a fixed order
#pragma unroll
            for (int hv = 32; hv >= 2; hv >>= 1) {
                const int m = hv >> 1;  // xor mask of this step: 16, 8, 4, 2, 1
                const bool up = (lane & m) != 0;
#pragma unroll
                for (int q = 0; q < hv; q++) {
                    const float send = up ? p[q] : p[q + hv];
                    const float keep = up ? p[q + hv] : p[q];
                    p[q] = keep + __shfl_xor_sync(0xffffffffu, send, m);
                }
            }
            sDW[quad * HI + 2 * lane] = p[0];
            sDW[quad * HI + 2 * lane + 1] = p[1];
            named_bar(2, EPI);
            if (et < HI) a.dw[row * HI + et] = (sDW[et] + sDW[HI + et]) + (sDW[2 * HI + et] + sDW[3 * HI + et]);
            named_bar(2, EPI);  // sDW and this row's w are read before the next row overwrites them
            if (et == 0) mbar_arrive(q_empty + qb);  // the q tile is no longer read
            rq++;
        }
    } else {
        // ---------------------------------------------------------------- MMA issue (whole warp)
        // Per row: MMA1 of tile t, then MMA2 of tile t - 1 (whose G' the epilogue has had MMA1's time to write);
        // the row's last MMA2 closes it.  (Two tiles of lag would hold each k tile one tile longer, and the k ring's
        // prefetch, not the epilogue, sets this kernel's pace.)
        // Barrier tests cost the issuing thread a shared-memory round trip, so after each MMA group the barriers
        // the next groups need are probed (two per round trip) while the MMAs just issued run; the warp waits only
        // on a barrier no probe has seen complete.  (None of them can be two phases behind: their previous uses
        // have been consumed.)
        int x = 0, rq = 0;
        bool g_rdy = false, k_rdy = false, x_rdy = false;  // G' of the next MMA2; k tile and X slot of the next tile
        auto mma2 = [&](int y, int t_in_row) {  // dQ'^T += k^T G' for the tile at ring position y
            const int gb = y % NX;
            if (t_in_row == 0) wait_bar(dq_empty, (rq & 1) ^ 1, abort_flag, err, 56);
            if (!g_rdy) wait_bar(g_full + gb, (y / NX) & 1, abort_flag, err, 57);
            g_rdy = false;
            fence_after();
            // eight MMAs of K = 16 (both operands MN-major, 2 KB further per MMA) in two groups of four
            const uint64_t dk = desc_sw128(sK + (y % NKT) * KT, KHALF, 1024), dg = desc_sw128(sG + gb * GT, GT, 1024);
            mma4_ss_w(tDQ, dk, 2048 >> 4, dg, 2048 >> 4, IDESC_DQ, t_in_row == 0 ? 0u : 1u, 0u);
            mma4_ss_w(tDQ, dk + (4 * 2048 >> 4), 2048 >> 4, dg + (4 * 2048 >> 4), 2048 >> 4, IDESC_DQ, 1u,
                      su32(k_empty + y % NKT));
            mma_commit_w(g_empty + gb);
            // the next tile's X slot (and its k tile, if not yet seen), while these MMAs run
            const uint32_t m = mbar_test2(x_empty + x % NX, ((x / NX) & 1) ^ 1, k_full + x % NKT, (x / NKT) & 1);
            x_rdy = (m & 1u) != 0u;
            k_rdy = k_rdy || (m & 2u) != 0u;
        };
        for (int i = blockIdx.x; i < total; i += gridDim.x) {
            const Item it = decode(a, i);
            if (it.nt == 0) continue;
            const int qb = rq & 1;
            wait_bar(q_full + qb, (rq >> 1) & 1, abort_flag, err, 58);
            fence_after();
            const unsigned char *pq = sQ + qb * QT;
            const int x0 = x;
            for (int t = 0; t < it.nt; t++) {
                const int st = x % NKT, xb = x % NX;
                if (!k_rdy) wait_bar(k_full + st, (x / NKT) & 1, abort_flag, err, 59);
                if (!x_rdy) wait_bar(x_empty + xb, ((x / NX) & 1) ^ 1, abort_flag, err, 60);
                k_rdy = x_rdy = false;
                fence_after();
                const unsigned char *pk = sK + st * KT;
                // per 64-wide K-half four MMAs of K = 16 (both operands K-major, 32 bytes further per MMA)
                mma4_ss_w(tX + (uint32_t)(xb * 64), desc_kmajor(pk), 2, desc_kmajor(pq), 2, IDESC_X, 0u, 0u);
                mma4_ss_w(tX + (uint32_t)(xb * 64), desc_kmajor(pk + KHALF), 2, desc_kmajor(pq + QHALF), 2, IDESC_X, 1u,
                          su32(x_full + xb));
                if (t == it.nt - 1) mma_commit_w(q_empty + qb);  // the row's q is read by its X groups only
                x++;
                if (t >= 1) {
                    // G' of tile t - 1 and the next tile's k, while MMA1 runs
                    const int y = x - 2;
                    const uint32_t m = mbar_test2(g_full + y % NX, (y / NX) & 1, k_full + x % NKT, (x / NKT) & 1);
                    g_rdy = (m & 1u) != 0u;
                    k_rdy = (m & 2u) != 0u;
                    mma2(y, t - 1);
                }
            }
            mma2(x0 + it.nt - 1, it.nt - 1);
            mma_commit_w(dq_full);
            rq++;
        }
        mma_commit_w(mma_done);
        drain_bar(mma_done, 0, err);
    }
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == MMA_WARP) tmem_dealloc(tmem, TMEM_COLS);
}

}  // namespace bwg

// ------------------------------------------------------------------ host side

cudaError_t launch_dq_dw_gather_tc(const Geo &g, const __nv_bfloat16 *q_idx, const float *w, const __nv_bfloat16 *k_idx,
                                   const int32_t *ids, const float *gslot, __nv_bfloat16 *dq, float *dw,
                                   unsigned long long *sgn, cudaStream_t st)
{
    using namespace bwg;
    CUtensorMap mq;
    if (!tc_encode_q_map(&mq, q_idx, g)) return cudaErrorInvalidValue;
    Args a = {};  // every field set below; zero first so none is ever left unset
    a.g = g;
    a.k_idx = k_idx;
    a.w = w;
    a.ids = ids;
    a.gslot = gslot;
    a.dq = dq;
    a.dw = dw;
    a.sgn = sgn;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(dq_dw_gather_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    const int grid = g.rows < sms ? g.rows : sms;
    dq_dw_gather_tc_kernel<<<grid, THREADS, SMEM, st>>>(mq, a);
    note_launches(1);
    return cudaGetLastError();
}

}  // namespace csa
