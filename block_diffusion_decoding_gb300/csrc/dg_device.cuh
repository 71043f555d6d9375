// dg_device.cuh -- device building blocks for sm_103a: mbarrier, TMA,
// tcgen05 (UMMA + TMEM) wrappers in inline PTX, bounded waits, Philox4x32-10
// and the sampler's fp32 logarithm.  Included by every kernel file.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/dg.h"

#define DG_DEVICE __device__ __forceinline__

namespace dg {

// ------------------------------------------------------------------------
// Workspace header: the first 256 bytes of every workspace.
// ------------------------------------------------------------------------
struct WsHeader {
    int32_t status;          // 0 or a DG_ERR_* code (first error wins)
    int32_t where;           // kernel-specific location of the first error
    // Row-bound sharing of the LM-head units (see LmHeadArgs::rowkey): the
    // launch count, the count + 1 once the running launch cleared the row
    // keys, and the units finished in the running launch (0 between launches)
    uint32_t lm_epoch;
    uint32_t lm_ready;
    uint32_t lm_done;
    int32_t pad[59];
};
static_assert(sizeof(WsHeader) == 256, "workspace header is 256 bytes");

DG_DEVICE uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

DG_DEVICE uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Atomic add with acquire-release semantics at GPU scope: the caller's earlier
// writes are visible to whoever observes the new value, and the writes that
// preceded the values it observes are visible to the caller afterwards.
DG_DEVICE int atomic_add_acq_rel_gpu(int *p, int v)
{
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

DG_DEVICE void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Order-preserving map of fp32 scores to u32 keys (larger score, larger key;
// -inf > key 0, which stands for "no bound").
DG_DEVICE uint32_t score_key(float f)
{
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

DG_DEVICE float key_score(uint32_t k)
{
    if (k == 0u) return -INFINITY;
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

DG_DEVICE void report_error(WsHeader *ws, int code, int where)
{
    if (ws != nullptr && atomicCAS(&ws->status, 0, code) == 0) ws->where = where;
}

// ------------------------------------------------------------------------
// Small PTX helpers
// ------------------------------------------------------------------------
DG_DEVICE uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

DG_DEVICE uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------------
// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel of the stream runs; it
// waits here before touching memory that kernel reads or writes.  Without
// the launch attribute both are no-ops.
// ------------------------------------------------------------------------
DG_DEVICE void griddep_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel of the stream launch (once every CTA of this grid has
// called this or exited).
DG_DEVICE void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------
// mbarrier
// ------------------------------------------------------------------------
DG_DEVICE void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

DG_DEVICE void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

DG_DEVICE void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

DG_DEVICE void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

DG_DEVICE bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Every wait in the library is bounded: after ~1 s of wall time it records
// DG_ERR_TIMEOUT in the workspace status word and returns false, and the
// caller winds down without touching the resource it waited for.
constexpr uint64_t kWaitLimitNs = 1000000000ull;

DG_DEVICE bool mbar_wait_limit(uint64_t *bar, uint32_t parity, WsHeader *ws, int where,
                               uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && globaltimer_ns() - t0 > limit_ns) {
            report_error(ws, DG_ERR_TIMEOUT, where);
            return false;
        }
    }
}

DG_DEVICE bool mbar_wait(uint64_t *bar, uint32_t parity, WsHeader *ws, int where)
{
    return mbar_wait_limit(bar, parity, ws, where, kWaitLimitNs);
}

// ------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor), completion on an mbarrier (complete_tx)
// ------------------------------------------------------------------------
DG_DEVICE void tma_prefetch_desc(const CUtensorMap *map)
{
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

DG_DEVICE void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y,
                           uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

// TMA loads of a 2-SM UMMA pair: the data lands in this CTA's shared memory,
// the completion (complete_tx) goes to the mbarrier at cluster address
// bar_cluster, which may be the even CTA's.
DG_DEVICE void tma_load_2d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                int y, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_3d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                int y, int z, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z),
        "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_3d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z,
                           uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z),
        "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_4d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z,
                           int w, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w),
        "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_5d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y, int z,
                           int w, int v, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(v), "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_4d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                int y, int z, int w, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z), "r"(w),
        "l"(policy)
        : "memory");
}

DG_DEVICE void tma_load_5d_pair(void *dst, const CUtensorMap *map, uint32_t bar_cluster, int x,
                                int y, int z, int w, int v, uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6, %7}], [%2], %8;" ::"r"(smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(x), "r"(y), "r"(z), "r"(w),
        "r"(v), "l"(policy)
        : "memory");
}

DG_DEVICE uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

DG_DEVICE uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (the tensor cores read operands through it).
DG_DEVICE void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------------
// tcgen05: TMEM allocation, UMMA issue/commit, TMEM loads/stores
// ------------------------------------------------------------------------
// Must be executed by one whole warp.  Writes the TMEM base address to *dst.
DG_DEVICE void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

DG_DEVICE void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

DG_DEVICE void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

DG_DEVICE void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

DG_DEVICE void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], kind::f16 (bf16 inputs, fp32 accumulate).
DG_DEVICE void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                         uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16.  A (M = 128 rows) sits in the
// 128 TMEM lanes, row i in lane i, two bf16 K-elements per 32-bit column
// (the lower K index in the low half); a_tmem is its first column.
DG_DEVICE void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                            uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive on *bar once every tcgen05.mma issued so far by this thread is done.
DG_DEVICE void umma_commit(uint64_t *bar)
{
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

// ---- 2-SM UMMA (cta_group::2): the CTA pair of a 2-CTA cluster acts as one
// MMA unit.  One warp of each CTA allocates (collectively) the same TMEM
// columns in both; the even CTA issues the MMAs; A (M = 256) is rows 0-127
// from the even CTA's shared memory and 128-255 from the odd one's at the
// same offset, B's N columns are split in halves the same way, and D rows
// 0-127 / 128-255 land in the even / odd CTA's TMEM at the same address.
DG_DEVICE void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}

DG_DEVICE void tmem_relinquish_pair()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

DG_DEVICE void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

DG_DEVICE void umma_bf16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// 2-SM UMMA of E4M3 operands (kind::f8f6f4: K = 32 per instruction, fp32
// accumulator), both from shared memory.
DG_DEVICE void umma_e4m3_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

DG_DEVICE void umma_bf16_pair_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                 uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrival on the mbarrier at this shared offset in every CTA of cta_mask once
// the pair MMAs issued so far by this thread are done.
DG_DEVICE void umma_commit_pair(uint64_t *bar, uint16_t cta_mask)
{
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
        " [%0], %1;" ::"r"(smem_u32(bar)),
        "h"(cta_mask)
        : "memory");
}

// ------------------------------------------------------------------------
// Paired fp32 arithmetic (two lanes of a 64-bit register pair per
// instruction) and a three-input maximum.
// ------------------------------------------------------------------------
DG_DEVICE float2 fma2(float2 a, float2 b, float2 c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)),
          "l"(*reinterpret_cast<const uint64_t *>(&c)));
    return *reinterpret_cast<const float2 *>(&d);
}

DG_DEVICE float2 add2(float2 a, float2 b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<const float2 *>(&d);
}

DG_DEVICE float2 mul2(float2 a, float2 b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<const uint64_t *>(&a)), "l"(*reinterpret_cast<const uint64_t *>(&b)));
    return *reinterpret_cast<const float2 *>(&d);
}

DG_DEVICE float max3(float a, float b, float c)
{
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// ------------------------------------------------------------------------
// Thread-block clusters
// ------------------------------------------------------------------------
// Address of the same shared-memory location in CTA `rank` of the cluster.
DG_DEVICE uint32_t mapa_shared(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

// Arrive (release at cluster scope) on an mbarrier given by its cluster address.
DG_DEVICE void mbar_arrive_cluster(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Arrive without ordering (relaxed, cluster scope) on an mbarrier given by its
// cluster address.  For signals that only say "my tcgen05 loads / stores are
// complete": the caller has already waited for them (tcgen05.wait::ld / ::st)
// and fenced (tcgen05.fence::before_thread_sync), so no memory needs to be
// released.  A release at cluster scope here costs 0.5-1.3 us per arrival on
// this GPU (measured), on the critical path of every key tile.
DG_DEVICE void mbar_arrive_cluster_relaxed(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
                 : "memory");
}

// Bounded wait that acquires at cluster scope (for barriers that other CTAs
// of the cluster arrive on).
DG_DEVICE bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Non-blocking probes of a phase (CTA / cluster acquire) and a bounded
// polling wait on them: it returns as soon as the phase completes, also when
// the completion comes from another CTA of the cluster or from a multicast
// commit.
DG_DEVICE bool mbar_test_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

DG_DEVICE bool mbar_test_wait_cluster(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

DG_DEVICE bool mbar_poll(uint64_t *bar, uint32_t parity, bool cluster, WsHeader *ws, int where)
{
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0;; ++it) {
        if (cluster ? mbar_test_wait_cluster(bar, parity) : mbar_test_wait(bar, parity)) return true;
        if ((it & 1023u) == 1023u && globaltimer_ns() - t0 > kWaitLimitNs) {
            report_error(ws, DG_ERR_TIMEOUT, where);
            return false;
        }
    }
}

DG_DEVICE bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, WsHeader *ws, int where)
{
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if ((it & 63u) == 0 && globaltimer_ns() - t0 > kWaitLimitNs) {
            report_error(ws, DG_ERR_TIMEOUT, where);
            return false;
        }
    }
}
DG_DEVICE uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

DG_DEVICE uint32_t cluster_id_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%clusterid.x;" : "=r"(r));
    return r;
}

DG_DEVICE uint32_t num_clusters_x()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%nclusterid.x;" : "=r"(r));
    return r;
}

// All threads of every CTA of the cluster arrive and wait (release/acquire).
DG_DEVICE void cluster_sync_all()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\t"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Instruction descriptor, kind::f16: D fp32, A/B bf16, A K-major,
// B K-major (b_mn_major = 0) or MN-major (1), shape M x N.
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, int b_mn_major)
{
    return (1u << 4)                                   // D format: f32
           | (1u << 7)                                 // A format: bf16
           | (1u << 10)                                // B format: bf16
           | (0u << 15)                                // A major: K
           | (static_cast<uint32_t>(b_mn_major) << 16) // B major
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Instruction descriptor of kind::f8f6f4 with E4M3 A and B (format code 0),
// both K-major, fp32 accumulator.
__host__ __device__ constexpr uint32_t make_idesc_e4m3(int M, int N)
{
    return (1u << 4)                                   // D format: f32
           | (0u << 7)                                 // A format: E4M3
           | (0u << 10)                                // B format: E4M3
           | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
           | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// Shared-memory matrix descriptor, 128-byte swizzle, tcgen05 format
// (version bits = 1).  lbo/sbo in bytes.
DG_DEVICE uint64_t make_sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo)
{
    return static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4) |
           (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
           (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// 32 lanes x 32 bit, 16 consecutive columns per thread, issued without
// waiting: the registers are valid only after tmem_wait_ld16 on them.
DG_DEVICE void tmem_ld16_issue(uint32_t taddr, uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

// Waits for this thread's TMEM loads; the registers pass through the wait so
// that no use of them can be scheduled before it.
DG_DEVICE void tmem_wait_ld16(uint32_t (&r)[16])
{
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]),
                   "+r"(r[6]), "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]),
                   "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
                 :
                 : "memory");
}

DG_DEVICE void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t r[16];
    tmem_ld16_issue(taddr, r);
    tmem_wait_ld16(r);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 32 bit, 32 consecutive columns per thread (no wait; call
// tmem_wait_ld before using the values).
DG_DEVICE void tmem_ld32_nowait(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

DG_DEVICE void tmem_wait_ld()
{
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

DG_DEVICE void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, "
        "%17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

// 32 lanes x 32 bit, 16 consecutive columns per thread.
DG_DEVICE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

DG_DEVICE void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, SC'11): 4 x 32-bit counter,
// 2 x 32-bit key, ten rounds of two 32x32->64 multiplies, the high halves
// xor'ed into the other words with the round key, key bumped by the Weyl
// constants between rounds.
// ------------------------------------------------------------------------
DG_DEVICE uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint64_t p0 = static_cast<uint64_t>(c.x) * 0xD2511F53u;   // one wide multiply
        const uint64_t p1 = static_cast<uint64_t>(c.z) * 0xCD9E8D57u;
        const uint32_t lo0 = static_cast<uint32_t>(p0), hi0 = static_cast<uint32_t>(p0 >> 32);
        const uint32_t lo1 = static_cast<uint32_t>(p1), hi1 = static_cast<uint32_t>(p1 >> 32);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Four Philox4x32-10 blocks under one key, advanced round by round: the
// same words as four philox4x32_10 calls, with one key-schedule update per
// round for all four and four independent multiply chains in flight.
DG_DEVICE void philox4x32_10_x4(uint4 (&c)[4], uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int round = 0; round < 10; ++round) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint64_t p0 = static_cast<uint64_t>(c[q].x) * 0xD2511F53u;
            const uint64_t p1 = static_cast<uint64_t>(c[q].z) * 0xCD9E8D57u;
            const uint32_t lo0 = static_cast<uint32_t>(p0), hi0 = static_cast<uint32_t>(p0 >> 32);
            const uint32_t lo1 = static_cast<uint32_t>(p1), hi1 = static_cast<uint32_t>(p1 >> 32);
            c[q] = make_uint4(hi1 ^ c[q].y ^ k0, lo1, hi0 ^ c[q].w ^ k1, lo0);
        }
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
}

// Philox streams of the sampler: counter (lane, row, step, stream).
enum : uint32_t { kStreamGumbel = 0u, kStreamRenoise = 1u, kStreamInit = 2u };

DG_DEVICE uint32_t token_from_word(uint32_t x, uint32_t V)
{
    return static_cast<uint32_t>((static_cast<uint64_t>(x) * V) >> 32);
}

// ------------------------------------------------------------------------
// The sampler's fp32 natural log: reduce x = 2^e m, m in [sqrt(1/2),
// sqrt(2)); with f = m - 1 and s = f / (2 + f), ln m = 2 atanh s, summed as
// 2s + 2s s^2 (1/3 + s^2 (1/5 + s^2 (1/7 + s^2 (1/9 + s^2/11)))); then add
// e ln 2 with ln 2 split in a 16-bit head (exact products) and a tail.
// Every operation is an explicit round-to-nearest intrinsic, so the result
// is a fixed function of x.  Valid for positive normal x.
// ------------------------------------------------------------------------
DG_DEVICE float sampler_logf(float x)
{
    const uint32_t bits = __float_as_uint(x);
    int e = static_cast<int>(bits >> 23) - 127;
    uint32_t mb = (bits & 0x007FFFFFu) | 0x3F800000u;
    if (mb > 0x3FB504F3u) {      // m > sqrt(2): halve m
        mb -= 0x00800000u;
        e += 1;
    }
    const float m = __uint_as_float(mb);
    const float f = __fsub_rn(m, 1.0f);
    const float s = __fdiv_rn(f, __fadd_rn(2.0f, f));
    const float w = __fmul_rn(s, s);
    float p = __uint_as_float(0x3DBA2E8Cu);                  // 1/11
    p = __fmaf_rn(p, w, __uint_as_float(0x3DE38E39u));       // 1/9
    p = __fmaf_rn(p, w, __uint_as_float(0x3E124925u));       // 1/7
    p = __fmaf_rn(p, w, __uint_as_float(0x3E4CCCCDu));       // 1/5
    p = __fmaf_rn(p, w, __uint_as_float(0x3EAAAAABu));       // 1/3
    const float t = __fadd_rn(s, s);
    const float r = __fmaf_rn(__fmul_rn(t, w), p, t);
    const float ef = static_cast<float>(e);
    return __fmaf_rn(ef, __uint_as_float(0x3F317200u),          // ln2 head
                     __fmaf_rn(ef, __uint_as_float(0x35BFBE8Eu), r));  // ln2 tail
}

// u = ((x >> 9) + 1/2) 2^-23 in (0,1), exact; G = -ln(-ln u).
DG_DEVICE float gumbel_from_bits(uint32_t x)
{
    const float u = __fmul_rn(__fadd_rn(static_cast<float>(x >> 9), 0.5f),
                              __uint_as_float(0x34000000u));
    const float e1 = -sampler_logf(u);
    return -sampler_logf(e1);
}

}  // namespace dg
