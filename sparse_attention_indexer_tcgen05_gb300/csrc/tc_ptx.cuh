// tc_ptx.cuh -- inline-PTX building blocks of the sm_103a tensor-core kernels: mbarriers with bounded
// waits, TMA tile loads, shared-memory matrix descriptors (128-byte swizzle, K-major and MN-major),
// tcgen05.mma / commit / fences, TMEM loads and named barriers.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace csa {
namespace ptx {

constexpr long long kTimeoutCycles = 4000000000LL;  // ~2 s at 2 GHz

__device__ __forceinline__ uint32_t su32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

// The dynamic shared memory aligned up to 1024 bytes (what 128-byte-swizzled TMA and MMA tiles need), by pointer
// arithmetic on the __shared__ array itself: the compiler then knows that every access through the result is a
// shared-memory one.  (Rounding the address through an integer hides that, and every load, store and atomic made
// through such a pointer becomes a generic-address one, which measured slower in the latency-bound loops.)  The
// alignment is taken on the shared-window address, the one TMA and the MMA descriptors use.
__device__ __forceinline__ unsigned char *smem_align1024(unsigned char *raw)
{
    return raw + ((1024u - (su32(raw) & 1023u)) & 1023u);
}

__device__ __forceinline__ void mbar_init(uint64_t *b, uint32_t n)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(n));
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *b, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *b)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(su32(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Non-blocking probe of a phase.  Its result is consumed later, so an MMA issuer can overlap the barrier's
// shared-memory round trip with the tensor work it issues in between.
__device__ __forceinline__ bool mbar_test(uint64_t *b, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok)
                 : "r"(su32(b)), "r"(parity)
                 : "memory");
    return ok != 0;
}
// Two non-blocking probes in one shared-memory round trip: bit 0 = phase `p0` of b0 complete, bit 1 = phase
// `p1` of b1 complete.  Meant to be issued right after a group of MMAs, so that the round trip overlaps the MMAs
// already queued on the tensor pipe (a probe placed before them leaves the pipe idle for its latency).
__device__ __forceinline__ uint32_t mbar_test2(uint64_t *b0, uint32_t p0, uint64_t *b1, uint32_t p1)
{
    uint32_t r;
    asm volatile("{\n\t.reg .pred q0, q1;\n\t.reg .b32 r0, r1;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 q0, [%1], %2;\n\t"
                 "mbarrier.test_wait.parity.shared::cta.b64 q1, [%3], %4;\n\t"
                 "selp.u32 r0, 1, 0, q0;\n\tselp.u32 r1, 2, 0, q1;\n\t"
                 "or.b32 %0, r0, r1;\n\t}"
                 : "=r"(r)
                 : "r"(su32(b0)), "r"(p0), "r"(su32(b1)), "r"(p1)
                 : "memory");
    return r;
}
__device__ __forceinline__ void init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// make generic-proxy shared-memory writes (st.shared) visible to the tensor core's async proxy

// Bounded wait.  Once any role has given up (abort set), waits return at once so control flow stays
// uniform and the kernel runs to its end; `err` receives the site code of the first expiry.  The phase is
// tried before the abort flag is read: on the fast path the flag's load latency would sit in the MMA
// issuer's critical path.
__device__ __forceinline__ void wait_bar_for(uint64_t *b, uint32_t parity, volatile int *abort_flag, int *err, int site,
                                             long long limit_cycles)
{
    if (mbar_try(b, parity)) return;
    if (*abort_flag) return;
    const long long t0 = clock64();
    while (!mbar_try(b, parity)) {
        if (*abort_flag) return;
        if (clock64() - t0 > limit_cycles) {
            *abort_flag = 1;
            atomicExch(err, site);
            return;
        }
    }
}
__device__ __forceinline__ void wait_bar(uint64_t *b, uint32_t parity, volatile int *abort_flag, int *err, int site)
{
    wait_bar_for(b, parity, abort_flag, err, site, kTimeoutCycles);
}
// Timer-only bounded wait, used to drain a kernel's own copies / MMAs even after an abort.
__device__ __forceinline__ void drain_bar(uint64_t *b, uint32_t parity, int *err)
{
    const long long t0 = clock64();
    while (!mbar_try(b, parity))
        if (clock64() - t0 > kTimeoutCycles) {
            atomicExch(err, 99);
            return;
        }
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y)
{
    asm volatile("cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
                 ::"r"(su32(dst)), "l"(map), "r"(su32(bar)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
                 ::"r"(su32(dst)), "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z, int w)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6}], [%2];"
                 ::"r"(su32(dst)), "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
}
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z, int w,
                                            int v)
{
    asm volatile("cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5, %6, %7}], [%2];"
                 ::"r"(su32(dst)), "l"(map), "r"(su32(bar)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(v)
                 : "memory");
}

// Shared-memory matrix descriptor, 128-byte swizzle, version 1 (bits 46-47), layout SWIZZLE_128B (bits 61-63 = 2).
//   K-major:  rows of 128 B (64 bf16 of K) per M/N index, 8-row atoms of 1024 B: SBO = 1024 B; LBO unused.
//   MN-major: 64 consecutive M/N elements per 128-B row, one row per K index, 8-row atoms of 1024 B along K:
//             SBO = 1024 B (next 8 K), LBO = byte distance between consecutive 64-wide M/N blocks.
__device__ __forceinline__ uint64_t desc_sw128(const void *p, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    const uint64_t a = su32(p);
    return ((a & 0x3FFFFull) >> 4) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFF) << 16) |
           ((uint64_t)((sbo_bytes >> 4) & 0x3FFF) << 32) | (1ull << 46) | (2ull << 61);
}
__device__ __forceinline__ uint64_t desc_kmajor(const void *p) { return desc_sw128(p, 16, 1024); }

// Instruction descriptor, kind::f16 with bf16 A/B and fp32 D: bits 4-5 D fmt (1 = f32), 7-9 A fmt (1 = bf16),
// 10-12 B fmt (1 = bf16), 15 A major (1 = MN), 16 B major (1 = MN), 17-22 N >> 3, 24-28 M >> 4.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn, bool b_mn)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Warp-wide forms: the whole warp runs the issue loop (its stage indices and descriptors are warp-uniform)
// and one lane chosen by elect.sync issues the instruction.
__device__ __forceinline__ void mma_bf16_w(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate));
}
// A operand from TMEM (lane = row m, 32-bit column c holds K elements 2c, 2c + 1 of the 16-bit type), B from
// shared memory; warp-wide, one elected lane issues.
__device__ __forceinline__ void mma_bf16_ts_w(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 ::"r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate));
}
// Four MMAs of K = 16 under one elect.sync, for issuing warps that share their scheduler with busy warps (every
// instruction of the issue loop then waits for an issue slot): A from TMEM columns a, a + s1, a + s2, a + s1 + s2
// (s1 = 8, s2 = 16: four consecutive K-steps of 16 bf16), B the shared-memory descriptor b advanced by db per MMA (db in the descriptor's 16-byte address units; the address field must not
// carry, i.e. the operands lie below 256 KB of shared memory), k = 0..3.  D is accumulated except by the first
// MMA when acc0 == 0.  If bar != 0 (a shared-memory address), the four MMAs (and every earlier one of this
// thread) are then committed to that mbarrier.
__device__ __forceinline__ void mma4_ts_w(uint32_t d, uint32_t a, uint32_t s1, uint32_t s2, uint64_t b, uint64_t db,
                                          uint32_t idesc, uint32_t acc0, uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e, p, t, c, ec;\n\t.reg .b64 b1, b2, b3;\n\t.reg .b32 a1, a2, a3;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 p, %5, 0;\n\t"
                 "setp.ne.b32 t, %4, 0;\n\t"  // the instruction descriptor is never 0: always true
                 "setp.ne.b32 c, %6, 0;\n\t"
                 "and.pred ec, e, c;\n\t"
                 "add.s64 b1, %2, %3;\n\tadd.s64 b2, b1, %3;\n\tadd.s64 b3, b2, %3;\n\t"
                 "add.u32 a1, %1, %7;\n\tadd.u32 a2, %1, %8;\n\tadd.u32 a3, a1, %8;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %4, p;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a1], b1, %4, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a2], b2, %4, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [a3], b3, %4, t;\n\t"
                 "@ec tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%6];\n\t}"
                 ::"r"(d), "r"(a), "l"(b), "l"(db), "r"(idesc), "r"(acc0), "r"(bar), "r"(s1), "r"(s2)
                 : "memory");
}
// The same with A also in shared memory: A descriptor a advanced by da per MMA.
__device__ __forceinline__ void mma4_ss_w(uint32_t d, uint64_t a, uint64_t da, uint64_t b, uint64_t db, uint32_t idesc,
                                          uint32_t acc0, uint32_t bar)
{
    asm volatile("{\n\t.reg .pred e, p, t, c, ec;\n\t.reg .b64 a1, a2, a3, b1, b2, b3;\n\t"
                 "elect.sync _|e, 0xffffffff;\n\t"
                 "setp.ne.b32 p, %6, 0;\n\t"
                 "setp.ne.b32 t, %5, 0;\n\t"
                 "setp.ne.b32 c, %7, 0;\n\t"
                 "and.pred ec, e, c;\n\t"
                 "add.s64 a1, %1, %2;\n\tadd.s64 a2, a1, %2;\n\tadd.s64 a3, a2, %2;\n\t"
                 "add.s64 b1, %3, %4;\n\tadd.s64 b2, b1, %4;\n\tadd.s64 b3, b2, %4;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %3, %5, p;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a1, b1, %5, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a2, b2, %5, t;\n\t"
                 "@e tcgen05.mma.cta_group::1.kind::f16 [%0], a3, b3, %5, t;\n\t"
                 "@ec tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%7];\n\t}"
                 ::"r"(d), "l"(a), "l"(da), "l"(b), "l"(db), "r"(idesc), "r"(acc0), "r"(bar)
                 : "memory");
}
__device__ __forceinline__ void mma_commit_w(uint64_t *bar)
{
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
                 "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(su32(bar))
                 : "memory");
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t cols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(su32(slot)), "r"(cols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t cols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols));
}

// 32 consecutive fp32 columns of this thread's TMEM lane (warp-collective), waited.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

// 32 consecutive fp32 columns of this thread's TMEM lane, NOT waited: other loads can be issued before
// tmem_wait_ld, which takes the registers so that no use of them moves above the wait.
__device__ __forceinline__ void tmem_ld32_async(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld(uint32_t (&r)[32])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
}

// 16 lanes x 32 columns in the 16x256b shape, repeated 4 times along the columns, then waited: with g = lane / 4
// and u = lane % 4, register 4 p + e holds (lane base + g, column 8 p + 2 u + e) and register 4 p + 2 + e holds
// (lane base + g + 8, the same column), p = 0..3, e = 0..1.
__device__ __forceinline__ void tmem_ld16x256_x4(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// The same load without the wait; tmem_wait_ld16 (which takes the registers, so that no use of them moves above
// it) completes every earlier load of the thread.
__device__ __forceinline__ void tmem_ld16x256_x4_async(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile("tcgen05.ld.sync.aligned.16x256b.x4.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane from registers (warp-collective), then waited.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                   "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane from registers (warp-collective), then waited.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&v)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 ::"r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                   "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
                   "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]),
                   "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16-byte asynchronous global -> shared copy (L2 only), its commit group and the wait for all but the n most
// recent groups; the proxy fence that makes completed generic-proxy writes of shared memory visible to the
// tensor core's async proxy.
__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(su32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N> __device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Paired fp32 arithmetic (one instruction for two values, the same rounding as two scalar operations).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    float2 r;
    asm("{\n\t.reg .b64 a, b, c, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\tmov.b64 c, {%6, %7};\n\t"
        "fma.rn.f32x2 d, a, b, c;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return r;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "add.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b)
{
    float2 r;
    asm("{\n\t.reg .b64 a, b, d;\n\tmov.b64 a, {%2, %3};\n\tmov.b64 b, {%4, %5};\n\t"
        "mul.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, d;\n\t}"
        : "=f"(r.x), "=f"(r.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return r;
}

__device__ __forceinline__ void named_bar(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// byte offset of 16-byte chunk c of row r inside a 128-byte-swizzled tile (rows of 128 B, 1024-B aligned)
__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk)
{
    return row * 128u + ((chunk ^ (row & 7u)) << 4);
}

}  // namespace ptx
}  // namespace csa
