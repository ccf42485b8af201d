// q4mm_device.cuh -- inline-PTX helpers for the sm_103a kernels of libq4mm:
// mbarriers with time-bounded waits, 1-D bulk async copies (TMA engine),
// proxy fences, programmatic dependent launch, bf16 packing, nibble
// unpacking, and the tcgen05 (5th-gen tensor core / TMEM) calls.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "q4mm_internal.h"

namespace q4 {

// ----------------------------------------------------------------- basics --

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// In-kernel event trace (profiling builds only, -DQ4MM_TRACE). Records are
// 16 bytes {globaltimer ns, event << 16 | warp << 8 | lane, argument}; each
// recording thread (lanes 0..3 of a warp) owns a region of `cap` records in
// the device buffer the host registered with q4_debug_set_trace, indexed by a
// shared-memory counter, so recording is a fire-and-forget store. Only the
// CTA chosen there records. Compiles to nothing in normal builds.
struct TraceRef {
    unsigned long long *buf; // regions of `cap` records, region = 4 * warp + lane
    unsigned cap;            // records per region
    unsigned cta;            // blockIdx.x that records
};

enum TraceEvent : unsigned {
    kTrStart = 1, kTrPdl = 2, kTrXStaged = 3, kTrWIssue = 4, kTrWFull = 5, kTrDeqDone = 6,
    kTrMmaIssue = 7, kTrBIssue = 8, kTrDone = 9, kTrEpiDone = 10, kTrEnd = 11, kTrBFull = 12,
    kTrSetup = 13, kTrTile = 14, kTrAlloc = 15, kTrXLoaded = 16, kTrXScaled = 17, kTrRed = 18, kTrAFull = 19
};

#ifdef Q4MM_TRACE
__device__ __forceinline__ unsigned *trace_counters()
{
    __shared__ unsigned counters[kTraceRegions];
    return counters;
}
#endif

// Zero the per-region counters; call before the kernel's first barrier.
__device__ __forceinline__ void trace_init()
{
#ifdef Q4MM_TRACE
    if (threadIdx.x < kTraceRegions) trace_counters()[threadIdx.x] = 0u;
#endif
}

__device__ __forceinline__ void trace(const TraceRef &t, unsigned ev, unsigned arg)
{
#ifdef Q4MM_TRACE
    const unsigned lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (t.buf && blockIdx.x == t.cta && lane < 4 && warp < kTraceRegions / 4) {
        const unsigned region = warp * 4 + lane;
        const unsigned i = trace_counters()[region]++;
        if (i < t.cap) {
            unsigned long long now;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
            unsigned long long *r = t.buf + 2ull * (static_cast<unsigned long long>(region) * t.cap + i);
            r[0] = now;
            r[1] = (static_cast<unsigned long long>((ev << 16) | (warp << 8) | lane) << 32) | arg;
        }
    }
#else
    (void)t, (void)ev, (void)arg;
#endif
}

// Record a device-side failure in the status word (first writer wins).
__device__ __forceinline__ void record_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// Range check of the checked build (-DQ4MM_CHECKED): true when `ok`; else
// records Q4_ERR_DEVICE_CHECK (10) and returns false, so that the caller
// skips the access. Always true in the ordinary build.
__device__ __forceinline__ bool q4_check(bool ok, int *status)
{
#ifdef Q4MM_CHECKED
    if (!ok) record_status(status, 10);
    return ok;
#else
    (void)ok;
    (void)status;
    return true;
#endif
}

// ---------------------------------------------------------------- mbarrier --

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Make barrier initialisation visible to the async proxy and the cluster.
__device__ __forceinline__ void fence_barrier_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
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

// The same test with cluster-scope acquire: for barriers that CTAs of the
// cluster arrive on remotely, after writing this CTA's shared memory.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity)
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


// Arrive, with cluster-scope release, on a barrier in another CTA of the
// cluster (`cluster_addr` from mapa_shared).
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Wait for the phase of `bar` with parity `parity` to complete, for at most
// limit_ns nanoseconds. Returns false if the limit ran out. Each try_wait may
// suspend the thread for a system-dependent time; it resumes when the phase
// completes (measured on GB300: ~170 ns after a local arrival, ~450 ns after
// a remote one; a try_wait given a suspend-time hint resumed ~560 ns after a
// local arrival, so none is given).
// Non-blocking test of a phase (this CTA's barrier, or acquire at cluster scope).
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity)
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
__device__ __forceinline__ bool mbar_test_wait_cluster(uint64_t *bar, uint32_t parity)
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

// Below this limit a wait polls without suspending (try_wait may sleep for
// longer than the limit inside one call), so that the limit is honoured.
constexpr uint64_t kShortWaitNs = 100000;

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (limit_ns < kShortWaitNs) {
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            if (mbar_test_wait(bar, parity)) return true;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (limit_ns < kShortWaitNs) {
        const uint64_t t0 = globaltimer_ns();
        while (true) {
            if (mbar_test_wait_cluster(bar, parity)) return true;
            if (globaltimer_ns() - t0 > limit_ns) return false;
        }
    }
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// ------------------------------------------------------------ bulk copies --

// 1-D bulk copy global -> shared (this CTA), completion counted in bytes on
// `bar`. dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Same, with an L2 eviction-priority policy created by createpolicy.
__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                             uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], "
        "%4;" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// Asynchronous prefetch of `bytes` at `src` into L2 (no completion signal).
// src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_prefetch_l2(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_last()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Generic-proxy writes to shared memory -> visible to the async proxy
// (tensor core operand reads).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------ programmatic dependent launch

// Block until the grids this launch depends on have completed and their
// memory is visible (no-op when launched without a programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the dependent grid in the stream to start launching.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ----------------------------------------------------------------- loads --

__device__ __forceinline__ uint4 lds128(const void *p)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ void sts128(void *p, uint4 v)
{
    asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(smem_u32(p)), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// ------------------------------------------------------------------- bf16 --

// Round-to-nearest-even fp32 -> bf16 bits.
__device__ __forceinline__ uint32_t bf16_rn_bits(float x)
{
    return static_cast<uint32_t>(__bfloat16_as_ushort(__float2bfloat16_rn(x)));
}

// Two fp32 -> packed bf16x2 (lo in bits 0..15), round to nearest even.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi)
{
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Packed bf16x2 arithmetic, each lane rounded once to nearest even.
__device__ __forceinline__ uint32_t bf16x2_sub(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
// (w & 0x000F000F) | 0x43004300 : two nibbles into bf16 128 + q (exact).
__device__ __forceinline__ uint32_t nib2_bf16_biased(uint32_t w)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(0x000F000Fu), "r"(0x43004300u));
    return r;
}

// One 4-byte word of split-half nibbles (bytes qs[4c..4c+3] of a block) into
// four bf16x2 values of (q - 8), exact. With e = 4c the word's element base:
//   v[0] = (e,    e+2)   v[1] = (e+16, e+18)
//   v[2] = (e+1,  e+3)   v[3] = (e+17, e+19)
// i.e. the eight weights in the order e + {0,2,16,18,1,3,17,19}.
__device__ __forceinline__ void unpack_word_bf16(uint32_t w, uint32_t v[4])
{
    const uint32_t k136 = 0x43084308u; // bf16 (136, 136)
    v[0] = bf16x2_sub(nib2_bf16_biased(w), k136);
    v[1] = bf16x2_sub(nib2_bf16_biased(w >> 4), k136);
    v[2] = bf16x2_sub(nib2_bf16_biased(w >> 8), k136);
    v[3] = bf16x2_sub(nib2_bf16_biased(w >> 12), k136);
}

// Same eight weights as fp16 (q - 8), exact. The high nibble of each byte is
// taken in place at bits 4..7 of an fp16 mantissa (1024 + 16q) and brought
// down by an exact fused multiply-add.
__device__ __forceinline__ uint32_t hsub2_bits(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t hfma2_bits(uint32_t a, uint32_t b, uint32_t c)
{
    uint32_t r;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
    return r;
}
__device__ __forceinline__ uint32_t hmul2_bits(uint32_t a, uint32_t b)
{
    uint32_t r;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t w, uint32_t mask, uint32_t magic)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(magic));
    return r;
}
__device__ __forceinline__ void unpack_word_f16(uint32_t w, uint32_t v[4])
{
    const uint32_t magic = 0x64006400u;   // fp16 (1024, 1024)
    const uint32_t k1032 = 0x64086408u;   // fp16 (1032, 1032)
    const uint32_t k1_16 = 0x2C002C00u;   // fp16 (1/16, 1/16)
    const uint32_t km72 = 0xD480D480u;    // fp16 (-72, -72)
    const uint32_t w8 = w >> 8;
    v[0] = hsub2_bits(lop3_and_or(w, 0x000F000Fu, magic), k1032);
    v[1] = hfma2_bits(lop3_and_or(w, 0x00F000F0u, magic), k1_16, km72);
    v[2] = hsub2_bits(lop3_and_or(w8, 0x000F000Fu, magic), k1032);
    v[3] = hfma2_bits(lop3_and_or(w8, 0x00F000F0u, magic), k1_16, km72);
}

// ------------------------------------------------------------ tcgen05 --

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols)
{
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish()
{
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols)
{
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D[tmem] (+)= A[smem desc] * B[smem desc], kind::f16 (bf16 in, fp32 acc).
__device__ __forceinline__ void tc_mma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on `bar` when every tcgen05 operation issued so far by this
// thread has completed.
__device__ __forceinline__ void tc_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}

// 32 lanes x 32 bits, 16 consecutive columns: thread i of the warp receives
// lane (base lane + i), columns col..col+15.
__device__ __forceinline__ void tmem_ld_32x32b_x2(uint32_t taddr, uint32_t r[2])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x2.b32 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr) : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x4(uint32_t taddr, uint32_t r[4])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr)
                 : "memory");
}
// Width-generic load of W consecutive columns (W in 2, 4, 8, 16, 32).
template <int W>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, uint32_t *r);
__device__ __forceinline__ void tmem_ld_32x32b_x8(uint32_t taddr, uint32_t r[8])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
}
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t r[16])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 32 lanes x 32 bits, 32 consecutive columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t r[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
template <> __device__ __forceinline__ void tmem_ld_cols<2>(uint32_t t, uint32_t *r) { tmem_ld_32x32b_x2(t, r); }
template <> __device__ __forceinline__ void tmem_ld_cols<4>(uint32_t t, uint32_t *r) { tmem_ld_32x32b_x4(t, r); }
template <> __device__ __forceinline__ void tmem_ld_cols<8>(uint32_t t, uint32_t *r) { tmem_ld_32x32b_x8(t, r); }
template <> __device__ __forceinline__ void tmem_ld_cols<16>(uint32_t t, uint32_t *r) { tmem_ld_32x32b_x16(t, r); }
template <> __device__ __forceinline__ void tmem_ld_cols<32>(uint32_t t, uint32_t *r) { tmem_ld_32x32b_x32(t, r); }

// Thread i of the warp writes its 16 registers to lane (base lane + i),
// columns col..col+15.
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t r[16])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// Thread i of the warp writes its 32 registers to lane (base lane + i),
// columns col..col+31.
__device__ __forceinline__ void tmem_st_32x32b_x32(uint32_t taddr, const uint32_t r[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
        "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]),
        "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// D[tmem] (+)= A[tmem] * B[smem desc], kind::f16 (A read from tensor memory:
// lane = row of A, column c = elements 2c, 2c+1 of that row's K).
__device__ __forceinline__ void tc_mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                              uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// ------------------------------------------------------------- clusters --

__device__ __forceinline__ uint32_t cluster_ctarank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
// Every thread of every CTA in the cluster arrives, then waits for all.
__device__ __forceinline__ void cluster_sync()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t mapa_shared(uint32_t saddr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v)
{
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Shared-memory matrix descriptor for a K-major operand in the 128-byte
// swizzled canonical layout: rows of 128 bytes, 8-row atoms 1024 bytes apart.
// The tile base must be 1024-byte aligned; K steps inside the 128-byte row
// advance the start address by 32 bytes per 16 bf16 elements.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t saddr)
{
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFF);        // start address
    d |= static_cast<uint64_t>(1) << 16;                        // leading byte offset (unused, 16 B)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;                // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                        // descriptor version (sm_100 family)
    d |= static_cast<uint64_t>(2) << 61;                        // swizzle: 128 B
    return d;
}

// Instruction descriptor, kind::f16: bf16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(uint32_t M, uint32_t N)
{
    return (1u << 4)              // D format: f32
           | (1u << 7)            // A format: bf16
           | (1u << 10)           // B format: bf16
           | ((N >> 3) << 17)     // N / 8
           | ((M >> 4) << 24);    // M / 16
}

// Instruction descriptor, kind::f16: fp16 A and B (both K-major), fp32 D.
__host__ __device__ constexpr uint32_t idesc_f16_f32(uint32_t M, uint32_t N)
{
    return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

} // namespace q4
