// ptx.cuh -- thin inline-PTX wrappers for sm_103a: mbarrier, TMA
// (cp.async.bulk.tensor), tcgen05 (TMEM alloc, MMA, commit, ld/st) and the
// bounded waits every kernel in this library uses.  Written from the public
// PTX ISA description of these instructions.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#define DEVI __device__ __forceinline__

namespace gqa {

// Device error word codes (bit flags, OR-ed together by failing threads).
enum : unsigned {
    kErrTimeout = 1u,  // a bounded wait gave up
    kErrIndex = 2u,    // a device-side index check failed (e.g. cache slot out of range)
    kErrRange = 4u,    // a value beyond the binary16 range was clamped
};

// Default limit of a bounded wait: 1 s of %globaltimer.  Every legitimate
// wait in these kernels lasts microseconds.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

DEVI uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

DEVI uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier

DEVI void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async proxy (TMA, tcgen05).
DEVI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

// Order this thread's generic-proxy shared-memory writes before later
// async-proxy reads (tcgen05.mma operands written with st.shared).
DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

DEVI void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

DEVI void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Arrive once without release semantics.  For hand-offs of TMEM contents
// only (see mbar_arrive_cluster_relaxed).
DEVI void mbar_arrive_relaxed(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// CLUSTER: acquire at cluster scope (the phase completes with arrivals from
// another CTA of the cluster whose earlier writes must be visible).
template <bool CLUSTER = false>
DEVI bool mbar_try_wait(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    if constexpr (CLUSTER)
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    else
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
    return ok != 0;
}

// Wait until the phase with the given parity has completed.  Gives up after
// limit_ns (recording kErrTimeout in *err) or as soon as another thread of the
// grid has recorded a timeout.  Returns true when the phase completed.
template <bool CLUSTER = false>
DEVI bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned *err, uint64_t limit_ns = kWaitLimitNs)
{
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait<CLUSTER>(a, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait<CLUSTER>(a, parity)) return true;
        if ((i & 63u) == 0) {
            if (*(volatile unsigned *)err & kErrTimeout) return false;
            if (globaltimer() - t0 > limit_ns) {
                atomicOr(err, kErrTimeout);
                return false;
            }
        }
    }
}

// ------------------------------------------------------ bf16 -> binary16

// Two bf16 values (one 32-bit word) as binary16, saturated to +-65504;
// `over` collects bit 15 of each half of (|x| bits + 0x3880), which is set
// exactly when |x| >= 2^16 (the bf16 values beyond binary16's range: every
// bf16 below 2^16 is at most 65280) or x is not finite.
DEVI uint32_t bf16x2_to_f16x2(uint32_t x, uint32_t &over)
{
    over |= (x & 0x7fff7fffu) + 0x38803880u;
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r)
        : "f"(__uint_as_float(x & 0xffff0000u)), "f"(__uint_as_float(x << 16)));
    return r;
}

// ------------------------------------------------ programmatic dependent launch

// Wait until the grids this one depends on (the previous kernel in the stream,
// when this one was launched as its programmatic dependent) have completed and
// their memory operations are visible.  Returns at once otherwise.
DEVI void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel in the stream, if launched as a programmatic dependent,
// be scheduled (its own grid_dep_wait still orders it after this grid).
DEVI void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- clusters

// Rank of this CTA in its thread-block cluster.
DEVI uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Every thread of every CTA of the cluster: shared-memory writes before it
// (local or remote) are visible to every thread after it.
DEVI void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// The shared::cluster address of the same offset in CTA `rank`'s shared memory.
DEVI uint32_t cluster_map(uint32_t local_addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_addr), "r"(rank));
    return r;
}

DEVI void st_cluster_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.shared::cluster.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
                 : "memory");
}

// --------------------------------------------------------------------- TMA

DEVI void tma_prefetch_desc(const CUtensorMap *tm)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"((uint64_t)tm) : "memory");
}

DEVI void tma_load_2d(void *dst, const CUtensorMap *tm, int x, int y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(smem_u32(bar))
        : "memory");
}

DEVI void tma_load_3d(void *dst, const CUtensorMap *tm, int x, int y, int z, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(smem_u32(bar))
        : "memory");
}

// Plain bulk copy global -> shared (both 16-byte aligned, bytes % 16 == 0).
DEVI void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"((uint64_t)src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------------------------ tcgen05

// Shared-memory matrix descriptor for a 128-byte-swizzled operand tile:
// start address, leading / stride byte offsets, descriptor version 1, swizzle
// mode "128B".  The tile base must be 1024-byte aligned.
DEVI uint64_t sw128_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1u << 46;  // version
    d |= (uint64_t)2u << 61;  // 128-byte swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16 with fp32 D: A and B both
// bf16 (ab_fmt 1) or both binary16 (ab_fmt 0), M x N tile, each operand
// K-major (0) or MN-major (1).
__host__ __device__ constexpr uint32_t idesc_f32acc(int M, int N, int a_mn_major, int b_mn_major, uint32_t ab_fmt)
{
    return (1u << 4)                        // D format f32
           | (ab_fmt << 7)                  // A format
           | (ab_fmt << 10)                 // B format
           | ((uint32_t)a_mn_major << 15)   // A major
           | ((uint32_t)b_mn_major << 16)   // B major
           | ((uint32_t)(N >> 3) << 17)     // N / 8
           | ((uint32_t)(M >> 4) << 24);    // M / 16
}
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major, int b_mn_major)
{
    return idesc_f32acc(M, N, a_mn_major, b_mn_major, 1u);
}
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N, int a_mn_major, int b_mn_major)
{
    return idesc_f32acc(M, N, a_mn_major, b_mn_major, 0u);
}

// Whole warp: allocate ncols TMEM columns (power of two >= 32); the base
// address is written to shared memory at dst.
DEVI void tmem_alloc(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// D[tmem] (+)= A[smem desc] * B[smem desc]^T, kind::f16 (bf16 or binary16
// operands as the instruction descriptor says); one thread issues.
DEVI void umma_f16_ss(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem desc]^T, kind::f16: A (M rows in TMEM lanes,
// K packed two 16-bit values per 32-bit column) read from tensor memory.
DEVI void umma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive (once) on an mbarrier when every tcgen05 op issued so far by this
// thread has completed.
DEVI void umma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ------------------------------------------------ CTA pairs (.cta_group::2)
// The two CTAs of a 2-CTA cluster share one MMA of M = 256: A rows 0-127 and
// B rows 0 .. N/2-1 come from the even CTA's shared memory, A rows 128-255
// and B rows N/2 .. N-1 from the odd CTA's (the same offsets in both), and
// the accumulator rows sit in the two CTAs' TMEM (rows 0-127 in the even CTA,
// 128-255 in the odd one), at the same address.  A kernel that uses these
// uses no .cta_group::1 form.

// One warp of EACH CTA of the pair: allocate ncols TMEM columns in both.
DEVI void tmem_alloc_pair(uint32_t *dst, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

// One warp of EACH CTA of the pair.
DEVI void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// One thread of the even CTA: D (+)= A * B^T over the pair.
DEVI void umma_f16_ss_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// The issuing thread: when its pair MMAs so far have completed, arrive once on
// the mbarrier at this offset in every CTA of cta_mask.
DEVI void umma_commit_pair(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// Tensor copy into this CTA's shared memory whose completion (bytes) is
// counted on the mbarrier at cluster address bar_cl, which may be the peer
// CTA's.
DEVI void tma_load_2d_pair(void *dst, const CUtensorMap *tm, int x, int y, uint32_t bar_cl)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(bar_cl)
        : "memory");
}

// 3-D form of tma_load_2d_pair.
DEVI void tma_load_3d_pair(void *dst, const CUtensorMap *tm, int x, int y, int z, uint32_t bar_cl)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(smem_u32(dst)),
        "l"((uint64_t)tm), "r"(x), "r"(y), "r"(z), "r"(bar_cl)
        : "memory");
}

// One thread of the even CTA: D (+)= A * B over the pair, A from TMEM (each
// CTA's 128 rows at the same TMEM address), B from shared memory as in
// umma_f16_ss_pair.
DEVI void umma_f16_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier at cluster address bar_cl (this or another CTA).
DEVI void mbar_arrive_cluster(uint32_t bar_cl)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

// As mbar_arrive_cluster without release semantics.  For hand-offs of TMEM
// contents only: the arriving thread has completed its TMEM accesses
// (tcgen05.wait::ld / wait::st) and issued tcgen05.fence::before_thread_sync,
// and the waiting side issues tcgen05.fence::after_thread_sync before its MMAs;
// no shared or global memory written before the arrival is read after the
// wait.  A release at cluster scope costs ~1000 SM clocks per arrival here.
DEVI void mbar_arrive_cluster_relaxed(uint32_t bar_cl)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cl) : "memory");
}

DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// TMEM -> registers, 32 lanes x 32 bits, 16 consecutive columns per thread.
// The wait is part of the same statement so no use of r can be scheduled
// before the data has arrived.
DEVI void tmem_ld16(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}

DEVI void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

// TMEM -> registers, 32 lanes x 32 bits, 128 consecutive columns (a whole
// 128-wide row per thread) in one instruction, then wait.
#define GQA_R8(i) "=r"(r[i]), "=r"(r[i + 1]), "=r"(r[i + 2]), "=r"(r[i + 3]), "=r"(r[i + 4]), "=r"(r[i + 5]), \
                  "=r"(r[i + 6]), "=r"(r[i + 7])
DEVI void tmem_ld128(uint32_t taddr, uint32_t (&r)[128])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x128.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,"
        "%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,"
        "%64,%65,%66,%67,%68,%69,%70,%71,%72,%73,%74,%75,%76,%77,%78,%79,"
        "%80,%81,%82,%83,%84,%85,%86,%87,%88,%89,%90,%91,%92,%93,%94,%95,"
        "%96,%97,%98,%99,%100,%101,%102,%103,%104,%105,%106,%107,%108,%109,%110,%111,"
        "%112,%113,%114,%115,%116,%117,%118,%119,%120,%121,%122,%123,%124,%125,%126,%127}, [%128];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : GQA_R8(0), GQA_R8(8), GQA_R8(16), GQA_R8(24), GQA_R8(32), GQA_R8(40), GQA_R8(48), GQA_R8(56),
          GQA_R8(64), GQA_R8(72), GQA_R8(80), GQA_R8(88), GQA_R8(96), GQA_R8(104), GQA_R8(112), GQA_R8(120)
        : "r"(taddr)
        : "memory");
}
#undef GQA_R8

// max of three floats in one instruction (sm_100+)
DEVI float fmax3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// registers -> TMEM, 32 lanes x 32 bits, 16 consecutive columns (no wait).
DEVI void tmem_st16_nowait(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

DEVI void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// registers -> TMEM, 32 lanes x 32 bits, 32 consecutive columns, then wait.
DEVI void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
        "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
        "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// ----------------------------------------------------- warp-level MMA (mma.sync)

// Four 8x8 16-bit matrices from shared memory; lane i gives the address of row
// i%8 of matrix i/8; lane t receives (row t/4, columns 2(t%4), 2(t%4)+1) of
// each matrix (transposed matrices with .trans).
DEVI void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}
DEVI void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// D = A(16x16, row) * B(16x8, col) + C, bf16 inputs, fp32 accumulators.
DEVI void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                         uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A(16x16, row) * B(16x8, col) + C, binary16 inputs, fp32 accumulators.
DEVI void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                        uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// ------------------------------------------------------------------- FP8

// Four E4M3 codes (byte 0 first) -> two binary16x2 words: lo = codes 0, 1,
// hi = codes 2, 3 (the lower code in the lower half).  Exact: every E4M3
// value is a binary16 value.
DEVI void e4m3x4_to_f16x4(uint32_t four_codes, uint32_t &lo, uint32_t &hi)
{
    asm("{\n\t.reg .b16 c01, c23;\n\t"
        "mov.b32 {c01, c23}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, c01;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, c23;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
}

// Two floats -> two E4M3 codes (lo in the low byte), nearest with ties to
// even, saturating at +-448.
DEVI uint32_t f32x2_to_e4m3x2(float lo, float hi)
{
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
}

// Byte permute: result byte i = byte sel[i] of (b:a) (a bytes 0-3, b bytes 4-7).
DEVI uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// ------------------------------------------------------------------- misc

DEVI float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
DEVI float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// Two floats -> packed bf16x2 (round to nearest even), lo in the low half.
DEVI uint32_t pack_bf16(float lo, float hi)
{
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

// Two floats -> packed binary16x2 (round to nearest even), lo in the low half.
DEVI uint32_t pack_f16(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&h);
}

constexpr float kHalfMax = 65504.0f;  // largest finite binary16

DEVI float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace gqa
