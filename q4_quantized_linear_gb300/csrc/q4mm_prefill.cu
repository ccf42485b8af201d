// q4mm_prefill.cu -- the tensor-core path for m > 16 token rows: reading a
// prompt, where wide passes switch from the mat-vec to tiled products (golem,
// "Reading a prompt on the card"; goinfer ch. 10, "What the kernels are":
// GEMM is prefill's workhorse). This is the one case that is a real dense
// contraction, so it runs on the 5th-generation tensor cores.
//
// Two kernels per call:
//   1. xcast: X fp32 -> bf16 (round to nearest even), written once into a
//      workspace already laid out as the shared-memory image the MMA reads
//      (K-major, 128-byte rows, 128-byte swizzle; within each block the
//      elements follow the order the weight dequantiser emits), so the GEMM
//      fetches each X tile with one 1-D bulk copy.
//   2. gemm: one CTA per (128 weight rows) x (T tokens). Warp roles:
//        warp 0     X-tile producer (one lane), ring as deep as shared
//                   memory allows: its copies take over a microsecond to land
//        warp 1     tensor-memory allocation; MMA thread for the first half
//                   of the token columns (all of them when T = 16)
//        warps 2-9  dequantise: each thread owns one weight row and writes
//                   the pair's 64 bf16 weights, (q - 8) times d, straight
//                   into tensor memory (two warps per TMEM sub-partition,
//                   alternating pairs); then the epilogue, TMEM -> Y
//        warp 10    weight-record producer (one lane), its own ring. The two
//                   producers sit in different warps: a lane asleep in a
//                   suspend-hinted barrier wait holds up its whole warp.
//        warp 11    MMA thread for the other half of the token columns.
//                   A thread gets only a few hundred cycles of MMA work
//                   ahead of the tensor pipe before its issue blocks, so each
//                   thread's waits and commits between pairs would leave the
//                   pipe idle; with two issuers one fills the other's gaps.
//      tcgen05.mma kind::f16 (bf16, fp32 accumulate in TMEM), A = the
//      dequantised weights read from tensor memory, B = the X tile in shared
//      memory, M = 128 weight rows, N = T tokens (two near-equal MMAs per
//      K step, one from each MMA thread, when T >= 32).
//      The weight operand never touches shared memory, which leaves shared
//      bandwidth to the X tiles. Every ring is an mbarrier pipeline; every
//      wait is time-bounded.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>
#include <cuda_runtime.h>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5;
constexpr int kDequantWarps = 8;
constexpr int kWProducerWarp = 2 + kDequantWarps;
constexpr int kMma2Warp = 3 + kDequantWarps;
constexpr int kWPrefetch = 8; // weight records requested into L2 beyond the ring
constexpr int kThreads = (4 + kDequantWarps) * 32;
constexpr size_t kStageChunkBytes = 16 * 128 * 4; // 16 tokens x 128 fp32 outputs

// ------------------------------------------------------------- xcast -----

__global__ void __launch_bounds__(256) xcast_kernel(const XcastArgs a)
{
    // The GEMM that follows may be scheduled at once: before its own
    // dependency wait it only streams and dequantises weights.
    pdl_launch_dependents();
    pdl_wait();
    const int64_t total = static_cast<int64_t>(a.ts) * a.np * a.T * 8;
    for (int64_t it = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; it < total;
         it += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int c = static_cast<int>(it & 7);
        const int64_t rowid = it >> 3;                 // (j * np + p) * T + r
        const int r = static_cast<int>(rowid % a.T);
        const int64_t jp = rowid / a.T;
        const int p = static_cast<int>(jp % a.np);
        const int j = static_cast<int>(jp / a.np);
        const int tok = j * a.T + r;
        const int blk = c >> 2, quad = c & 3;
        const int b = 2 * p + blk;
        uint4 out = make_uint4(0u, 0u, 0u, 0u);
        if (tok < a.m && b < a.nb) {
            const int64_t row = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
            const float *xr = a.X + row * a.ldx + 32 * b;
            const float4 xa = __ldg(reinterpret_cast<const float4 *>(xr + 4 * quad));
            const float4 xb = __ldg(reinterpret_cast<const float4 *>(xr + 16 + 4 * quad));
            // block elements 4*quad + {0,2,16,18,1,3,17,19}
            out.x = pack_bf16x2_rn(xa.x, xa.z);
            out.y = pack_bf16x2_rn(xb.x, xb.z);
            out.z = pack_bf16x2_rn(xa.y, xa.w);
            out.w = pack_bf16x2_rn(xb.y, xb.w);
        }
        uint8_t *dst = a.ximg + rowid * 128 + ((c ^ (r & 7)) << 4);
        *reinterpret_cast<uint4 *>(dst) = out;
    }
}

// -------------------------------------------------------------- gemm -----

struct Smem {
    uint8_t *b, *w;
    uint64_t *full_b, *empty_b, *full_w, *empty_w, *full_a, *empty_a, *done;
    uint32_t *tmem_slot;
    int *abort;
};

__device__ __forceinline__ bool aborted(const Smem &sm) { return *reinterpret_cast<volatile int *>(sm.abort) != 0; }

__device__ __forceinline__ void fail(const Smem &sm, const PrefillArgs &a)
{
    *reinterpret_cast<volatile int *>(sm.abort) = 1;
    record_status(a.status, kErrTimeout);
}

// Bounded wait by every lane of a warp with one outcome for the whole warp:
// a timeout must not leave a warp diverged in front of .aligned tcgen05 code.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns)) != 0;
}

// One row's pair of blocks -> 32 bf16x2 columns of tensor memory, in the
// order the MMA's K runs: column 16 blk + 4 wd + j holds v[j] of nibble word
// wd of block blk, i.e. block elements 4 wd + {0,2 | 16,18 | 1,3 | 17,19}.
// Each weight is (q - 8), exact, times d rounded to bf16; the product is
// rounded to bf16 once more.
__device__ __forceinline__ void dequant_pair_bf16(uint32_t d01, uint4 q0, uint4 q1, uint32_t out[32])
{
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>(blk ? d01 >> 16 : d01 & 0xFFFF)));
        const uint32_t h = bf16_rn_bits(d);
        const uint32_t dd = h | (h << 16);
        const uint4 q = blk ? q1 : q0;
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            uint32_t v[4];
            unpack_word_bf16(words[wd], v);
#pragma unroll
            for (int j = 0; j < 4; ++j) out[blk * 16 + wd * 4 + j] = bf16x2_mul(v[j], dd);
        }
    }
}

// SPLIT: the K slices of a tile run as one cluster and meet in its first
// CTA; without it (a.ks == 1) the kernel carries none of that code.
template <bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1) gemm_kernel(const PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // CTA = (128-row tile = packed group, token tile, K slice); the a.ks
    // slices of a tile are one cluster and take consecutive pair ranges
    const int KS = SPLIT ? a.ks : 1;
    const int ksi = static_cast<int>(blockIdx.x) % KS;
    const int tile = static_cast<int>(blockIdx.x) / KS;
    const int rt = tile / a.ts;
    const int jt = tile % a.ts;
    const int T = a.T;
    const int p0 = ksi * ((a.np + KS - 1) / KS);
    const int np = min(a.np, p0 + (a.np + KS - 1) / KS) - p0; // this CTA's pairs (the planner keeps it >= 1)
    const int RB = a.bring, RW = a.wring;
    const int AST = a.astages;
    const uint32_t bstage = static_cast<uint32_t>(T) * 128u;
    const uint32_t acol0 = static_cast<uint32_t>((T + 31) & ~31); // first A column after D
    const TraceRef tr{a.trace_buf, a.trace_cap, a.trace_cta};
    trace_init();
    if (tid == 0) trace(tr, kTrStart, 0);

    Smem sm;
    sm.b = base;
    sm.w = sm.b + static_cast<size_t>(RB) * bstage;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm.w + static_cast<size_t>(RW) * kRecordBytes);
    sm.full_b = bars;
    sm.empty_b = sm.full_b + RB;
    sm.full_w = sm.empty_b + RB;
    sm.empty_w = sm.full_w + RW;
    sm.full_a = sm.empty_w + RW;
    sm.empty_a = sm.full_a + AST;
    sm.done = sm.empty_a + AST;
    sm.tmem_slot = reinterpret_cast<uint32_t *>(sm.done + 1);
    sm.abort = reinterpret_cast<int *>(sm.tmem_slot + 1);

    // Token columns [0, N1) go to the MMA thread of warp 1, [N1, T) to the
    // one of warp 11, in near-equal halves (each a multiple of 16) whenever
    // the tile has two; a 16-token tile has one MMA thread.
    const int N1 = T >= 32 ? ((T / 2 + 15) & ~15) : T;
    const int N2 = T - N1;
    const uint32_t issuers = N2 > 0 ? 2u : 1u;
    if (tid == 0) {
        for (int i = 0; i < RB; ++i) mbar_init(&sm.full_b[i], 1), mbar_init(&sm.empty_b[i], issuers);
        for (int i = 0; i < RW; ++i) mbar_init(&sm.full_w[i], 1), mbar_init(&sm.empty_w[i], kDequantWarps / 2);
        for (int i = 0; i < AST; ++i) mbar_init(&sm.full_a[i], kDequantWarps / 2), mbar_init(&sm.empty_a[i], issuers);
        mbar_init(sm.done, issuers);
        *sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, 512u);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;

    const uint8_t *wsrc = a.W + (static_cast<int64_t>(rt) * a.np + p0) * kRecordBytes;
    const uint8_t *xsrc = a.ximg + (static_cast<size_t>(jt) * a.np + p0) * bstage;
    // One lane streams the X tiles, another (in another warp) the weight
    // records, each in pair order through its own ring (one owner per slot).
    const uint64_t pol = policy_evict_last();

    // The dequantising warps (2-9) also run the epilogue: warp 2 + 4 h + i
    // holds TMEM sub-partition q = warp % 4, i.e. weight rows 32 q .. + 31.
    const int q = warp & 3;
    const int h = ((warp - 2) >> 2) & 1;   // dequantiser set: pairs p % 2 == h
    const int row = q * 32 + lane;         // weight row within the tile
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const bool epi_warp = warp >= 2 && warp < 2 + kDequantWarps;
    bool done_ok = false;

    if (warp == 0) {
        // ---------------------------------------------------- X-tile producer
        // Only the X tiles come from the preceding kernel (the X cast); the
        // dequantisers touch shared and tensor memory only until the
        // epilogue, which follows the last MMA and so this wait.
        pdl_wait();
        if (tid == 0) trace(tr, kTrPdl, 0);
        if (lane == 0) {
            int s = 0, last = -1;
            uint32_t ph = 0;
            for (int p = 0; p < np && !aborted(sm); ++p) {
                if (p >= RB && !mbar_wait(&sm.empty_b[s], ph ^ 1u, a.wait_ns)) { fail(sm, a); break; }
                trace(tr, kTrBIssue, static_cast<unsigned>(p));
                mbar_arrive_expect_tx(&sm.full_b[s], bstage);
                bulk_g2s_hint(sm.b + static_cast<size_t>(s) * bstage, xsrc + static_cast<size_t>(p) * bstage, bstage,
                              &sm.full_b[s], pol);
                last = p;
                if (++s == RB) s = 0, ph ^= 1u;
            }
            // no copy may still be landing when the CTA exits: only the last
            // RB tiles' copies can be (a slot reused later has landed)
            for (int p = last; p >= 0 && p >= np - RB; --p)
                if (!mbar_wait(&sm.full_b[p % RB], (p / RB) & 1, a.wait_ns)) fail(sm, a);
        }
        __syncwarp();
    } else if (warp == kWProducerWarp) {
        // ---------------------------------------------- weight-record producer
        // With the weights declared read-only the records stream before the
        // dependency wait (no kernel in flight writes them); otherwise the
        // preceding kernels must have finished first.
        // The ring is shallow (shared memory goes to the X tiles), so records
        // further ahead are pulled into L2 first: a slot then waits out an L2
        // hit, not an HBM round trip.
        if (!a.prefetch_w) pdl_wait();
        if (lane == 0) {
            int s = 0, last = -1;
            uint32_t ph = 0;
            for (int p = RW; p < np && p < RW + kWPrefetch; ++p)
                bulk_prefetch_l2(wsrc + static_cast<size_t>(p) * kRecordBytes, kRecordBytes);
            for (int p = 0; p < np && !aborted(sm); ++p) {
                if (p >= RW && !mbar_wait(&sm.empty_w[s], ph ^ 1u, a.wait_ns)) { fail(sm, a); break; }
                trace(tr, kTrWIssue, static_cast<unsigned>(p));
                mbar_arrive_expect_tx(&sm.full_w[s], kRecordBytes);
                bulk_g2s_hint(sm.w + static_cast<size_t>(s) * kRecordBytes, wsrc + static_cast<size_t>(p) * kRecordBytes,
                              kRecordBytes, &sm.full_w[s], pol);
                if (p + RW + kWPrefetch < np)
                    bulk_prefetch_l2(wsrc + static_cast<size_t>(p + RW + kWPrefetch) * kRecordBytes, kRecordBytes);
                last = p;
                if (++s == RW) s = 0, ph ^= 1u;
            }
            for (int p = last; p >= 0 && p >= np - RW; --p)
                if (!mbar_wait(&sm.full_w[p % RW], (p / RW) & 1, a.wait_ns)) fail(sm, a);
        }
        __syncwarp();
    } else if (warp == 1 || warp == kMma2Warp) {
        // --------------------------------------------------------------- MMA
        // One thread per token-column range; descriptors are precomputed and
        // the loop body is straight-line so its MMAs issue back to back. Both
        // threads wait for every A stage and X tile and both commit to its
        // release barrier (arrival count 2), so a slot is refilled only after
        // both have finished with it: neither can fall a phase behind.
        const bool second = warp == kMma2Warp;
        if (lane == 0 && (!second || N2 > 0)) {
            const uint32_t ncols = static_cast<uint32_t>(second ? N2 : N1);
            const uint32_t idesc = idesc_bf16_f32(128, ncols);
            const uint32_t d = tmem + (second ? static_cast<uint32_t>(N1) : 0u);
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sm.b)) + (second ? static_cast<uint64_t>((N1 * 128) >> 4) : 0u);
            const uint64_t bstep = static_cast<uint64_t>(bstage >> 4);
            uint64_t bd = bdesc0;
            uint32_t at = tmem + acol0;
            int sa = 0, sb = 0;
            uint32_t pha = 0, phb = 0, acc = 0;
            // The barrier tests for pair p + 1 are issued before pair p's
            // MMAs: their round trip (a few hundred cycles) then overlaps
            // the MMA issue, which blocks while the tensor pipe is busy,
            // instead of sitting between two pairs. A pair whose tests came
            // back negative takes the bounded wait.
            bool ready = mbar_test_wait(&sm.full_a[0], 0u) & mbar_test_wait(&sm.full_b[0], 0u);
            for (int p = 0; p < np; ++p) {
                if (!ready && (!mbar_wait(&sm.full_a[sa], pha, a.wait_ns) || !mbar_wait(&sm.full_b[sb], phb, a.wait_ns))) {
                    fail(sm, a);
                    break;
                }
                trace(tr, kTrMmaIssue, static_cast<unsigned>(p));
                int na = sa + 1, nb = sb + 1;
                uint32_t npha = pha, nphb = phb;
                if (na == AST) na = 0, npha ^= 1u;
                if (nb == RB) nb = 0, nphb ^= 1u;
                bool next = false;
                if (p + 1 < np) next = mbar_test_wait(&sm.full_a[na], npha) & mbar_test_wait(&sm.full_b[nb], nphb);
                tc_fence_after();
                tc_mma_f16_ts(d, at, bd, idesc, acc);
                tc_mma_f16_ts(d, at + 8u, bd + 2u, idesc, 1u);
                tc_mma_f16_ts(d, at + 16u, bd + 4u, idesc, 1u);
                tc_mma_f16_ts(d, at + 24u, bd + 6u, idesc, 1u);
                tc_commit(&sm.empty_a[sa]);
                tc_commit(&sm.empty_b[sb]);
                acc = 1u;
                ready = next;
                sa = na, sb = nb, pha = npha, phb = nphb;
                at = tmem + acol0 + 32u * static_cast<uint32_t>(sa);
                bd = bdesc0 + static_cast<uint64_t>(sb) * bstep;
            }
            tc_commit(sm.done); // also taken on abort: no MMA of ours is in flight past this
        }
        __syncwarp();
    } else {
        // ----------------------------------------------------- dequantise W
        for (int p = h; p < np && !__any_sync(0xFFFFFFFFu, aborted(sm)); p += 2) {
            const int sw = p % RW, sa = p % AST;
            if (!warp_wait(&sm.full_w[sw], (p / RW) & 1, a.wait_ns)) { fail(sm, a); break; }
            if (lane == 0) trace(tr, kTrWFull, static_cast<unsigned>(p));
            if (!warp_wait(&sm.empty_a[sa], ((p / AST) & 1) ^ 1, a.wait_ns)) { fail(sm, a); break; }
            const uint8_t *rec = sm.w + static_cast<size_t>(sw) * kRecordBytes;
            const uint32_t d01 = *reinterpret_cast<const uint32_t *>(rec + kRecScaleOff + 4 * row);
            const uint4 q0 = lds128(rec + kRecQs0Off + 16 * row);
            const uint4 q1 = lds128(rec + kRecQs1Off + 16 * row);
            uint32_t out[32];
            dequant_pair_bf16(d01, q0, q1, out);
            tmem_st_32x32b_x32(tmem + lane_base + acol0 + static_cast<uint32_t>(sa) * 32u, out);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.full_a[sa]);
                mbar_arrive(&sm.empty_w[sw]);
                trace(tr, kTrDeqDone, static_cast<unsigned>(p));
            }
        }

        done_ok = warp_wait(sm.done, 0, a.wait_ns);
        if (!done_ok) fail(sm, a);
        if (lane == 0) trace(tr, kTrDone, 0);
        tc_fence_after();
        pdl_launch_dependents();
    }

    // ----------------------------------------------------------- epilogue
    // Each dequantising warp takes its TMEM sub-partition and half of the
    // token columns.
    const int chunks = T / 16;
    const int c_lo = h * ((chunks + 1) / 2), c_hi = h ? chunks : (chunks + 1) / 2;
    const int64_t grow = static_cast<int64_t>(rt) * 128 + row;
    // Y is row-major by token, so a token's outputs for this tile's rows
    // are contiguous, but a warp's tensor-memory load gives each lane one
    // row for 16 tokens. Written directly that is one 4-byte store per
    // output, and the store instructions bound the epilogue. Staged, each
    // warp puts its 32 rows x 16 tokens in shared memory and reads them back
    // as 4 rows of one token per lane: four 16-byte stores per lane per
    // chunk instead of sixteen 4-byte ones. The rings are idle by now (every
    // X tile and weight record was consumed before the last MMA completed),
    // so the whole tile is staged without reuse, when the staging area and
    // the K slices' partial tiles both fit in them. The direct form is kept
    // for Y whose base or row stride is not a multiple of 16 bytes and for
    // tiles too wide to stage. (Uniform over the cluster: its CTAs agree on
    // where the partial tiles go.)
    const size_t ring_bytes = static_cast<size_t>(RB) * bstage + static_cast<size_t>(RW) * kRecordBytes;
    const bool staged = (a.ldy & 3) == 0 && (reinterpret_cast<uintptr_t>(a.Y) & 15u) == 0 &&
                        static_cast<size_t>(KS) * chunks * kStageChunkBytes <= ring_bytes;
    // Partial tiles of slices 1 .. KS - 1, [slice - 1][token column][row]
    // fp32, in the first CTA's rings: after the staging area when staged,
    // else from the start (the planner keeps them inside the rings).
    const size_t partial_off = staged ? static_cast<size_t>(chunks) * kStageChunkBytes : 0;
    float *partials = reinterpret_cast<float *>(sm.b + partial_off);
    if (SPLIT && !q4_check(partial_off + static_cast<size_t>(KS - 1) * chunks * kStageChunkBytes <= ring_bytes, a.status))
        done_ok = false; // (checked build) no partial tile is written or read
    if constexpr (SPLIT) {
        // Every CTA of the cluster has left its K loop (the first CTA's
        // rings are free); every thread passes both barriers, also after a
        // failed wait, so that none is left at one.
        tc_fence_before();
        cluster_sync();
        tc_fence_after();
        if (epi_warp && ksi > 0 && done_ok) {
            const uint32_t dst0 = mapa_shared(smem_u32(partials), 0u) +
                                  static_cast<uint32_t>((static_cast<size_t>(ksi - 1) * T * 128 + row) * 4);
            for (int cc = c_lo; cc < c_hi; ++cc) {
                const int c0 = cc * 16;
                uint32_t r[16];
                tmem_ld_32x32b_x16(tmem + lane_base + static_cast<uint32_t>(c0), r);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i)
                    st_cluster_f32(dst0 + static_cast<uint32_t>((c0 + i) * 128 * 4), __uint_as_float(r[i]));
            }
        }
        tc_fence_before();
        cluster_sync(); // the partial tiles are in the first CTA's shared memory
        tc_fence_after();
    }
    if (epi_warp && ksi == 0 && done_ok) {
        const int64_t rows_here = min(static_cast<int64_t>(128), a.n - static_cast<int64_t>(rt) * 128);
        for (int cc = c_lo; cc < c_hi; ++cc) {
            const int c0 = cc * 16;
            uint32_t r[16];
            tmem_ld_32x32b_x16(tmem + lane_base + static_cast<uint32_t>(c0), r);
            tmem_wait_ld();
            // the other K slices' partial sums, in slice order
            for (int sl = 0; SPLIT && sl + 1 < KS; ++sl) {
                const float *pt = partials + (static_cast<size_t>(sl) * T + c0) * 128 + row;
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) + pt[i * 128]);
            }
            if (staged) {
                // this warp's 32 rows of the chunk: [16 tokens][32 rows]
                uint8_t *part = sm.b + static_cast<size_t>(cc) * kStageChunkBytes + static_cast<size_t>(q) * 2048;
#pragma unroll
                for (int i = 0; i < 16; ++i) *reinterpret_cast<uint32_t *>(part + i * 128 + lane * 4) = r[i];
                __syncwarp();
                // lane l: rows 4 (l % 8) .. + 3 of token 4 k + l / 8
                const int64_t col = static_cast<int64_t>(rt) * 128 + q * 32 + (lane & 7) * 4;
                const int lrow = q * 32 + (lane & 7) * 4;   // within the 128-row tile
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const int i = 4 * k + (lane >> 3);
                    const int tok = jt * T + c0 + i;
                    const uint4 v = lds128(part + i * 128 + (lane & 7) * 16);
                    if (tok < a.m) {
                        const int64_t yrow = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
                        float *dst = a.Y + yrow * a.ldy + col;
                        if (lrow + 3 < rows_here) {
                            *reinterpret_cast<uint4 *>(dst) = v;
                        } else {
                            const uint32_t e4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                if (lrow + e < rows_here) dst[e] = __uint_as_float(e4[e]);
                        }
                    }
                }
            } else {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const int tok = jt * T + c0 + i;
                    if (tok < a.m && grow < a.n) {
                        const int64_t yrow = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
                        a.Y[yrow * a.ldy + grow] = __uint_as_float(r[i]);
                    }
                }
            }
        }
    }
    if (epi_warp && lane == 0) trace(tr, kTrEpiDone, 0);

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 512u);
    }
    if (tid == 0) trace(tr, kTrEnd, 0);
}

__global__ void wait_selftest_kernel(int *status, uint64_t limit_ns)
{
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    // nothing ever arrives on `bar`: the bounded wait must give up
    if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) record_status(status, kErrTimeout);
    __syncthreads();
}

size_t gemm_smem_bytes(int T, int bring, int wring, int astages)
{
    return 1024 + static_cast<size_t>(bring) * static_cast<size_t>(T) * 128 +
           static_cast<size_t>(wring) * kRecordBytes + static_cast<size_t>(2 * bring + 2 * wring + 2 * astages + 1) * 8 +
           16;
}

// Clusters of ks GEMM CTAs (`threads` each, `smem` bytes of dynamic shared
// memory) that the current device holds at once; 0 when it cannot be asked.
// Cached per (device, ks, smem, threads).
int gemm_max_clusters(int ks, size_t smem, int threads)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, size_t, int>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, ks, smem, threads);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void *fn = reinterpret_cast<const void *>(&gemm_kernel<true>);
    int n = 0;
    if (set_max_smem(fn, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(ks));
        cfg.blockDim = dim3(static_cast<unsigned>(threads));
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(ks);
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess) n = 0;
    }
    cudaGetLastError();
    cache.emplace(key, n);
    return n;
}

} // namespace

namespace {

// Rings and tensor-memory stages for a token tile of T; false when none fits.
bool prefill_rings(int T, PrefillPlan *p)
{
    const int acol0 = (T + 31) & ~31;
    // even, so that each stage always belongs to one of the two dequantiser
    // sets (parity waits need a single waiter per barrier)
    p->astages = std::min(8, (512 - acol0) / 32) & ~1;
    if (p->astages < 2) return false;
    // A weight ring of 8 first (the records come from HBM, the X tiles from
    // L2: for 540x9728x2560 a ring of 8 next to 5 X tiles beats 4 next to 6
    // by 4%), then the deepest X-tile ring that fits next to it.
    p->bring = p->wring = 0;
    for (int wr : {8, 4, 2}) {
        int br = 8;
        while (br > 2 && gemm_smem_bytes(T, br, wr, p->astages) > kSmemOptIn) --br;
        if (gemm_smem_bytes(T, br, wr, p->astages) > kSmemOptIn) continue;
        if (wr > p->wring) p->bring = br, p->wring = wr;
    }
    if (p->bring == 0) return false;
    p->smem = gemm_smem_bytes(T, p->bring, p->wring, p->astages);
    if (p->smem > kSmemOptIn) return false;
    // one CTA per SM: each holds all 512 tensor-memory columns
    p->smem = std::max<size_t>(p->smem, kSmemPerSM / 2 + 1024);
    return true;
}

// Time model of a call, fitted to graph-replay timings on GB300: a CTA's
// 64-deep K step takes about the same whatever the token tile (0.39 us at
// 16 tokens, 0.43 at 144, 0.45 at 272: the dequantisation and the MMA issue
// set it, not the tensor math), plus a fixed 5 us per wave; a K split adds
// its exchange, and the direct epilogue (no room to stage) its stores.
constexpr double kPairUs = 0.42, kWaveUs = 5.0, kSplitUs = 1.0, kDirectUs = 1.3;

bool plan_prefill_search(int64_t m, int64_t k, int64_t n, int sm_count, PrefillPlan *plan)
{
    const int64_t rowtiles = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    PrefillPlan best;
    double best_cost = 1e300;
    for (int64_t ts = ceil_div(m, 448); ts <= std::max<int64_t>(1, ceil_div(m, 16)); ++ts) {
        const int64_t T = round_up(ceil_div(m, ts), 16);
        if (T > 448) continue;
        PrefillPlan c;
        c.T = static_cast<int>(T);
        c.ts = static_cast<int>(ts);
        c.rowtiles = static_cast<int>(rowtiles);
        if (!prefill_rings(c.T, &c)) continue;
        const size_t cap = static_cast<size_t>(c.bring) * c.T * 128 + static_cast<size_t>(c.wring) * kRecordBytes;
        const int threads = c.T >= 32 ? kThreads : kThreads - 32;
        const int64_t tiles = rowtiles * ts;
        // ks K slices: a cluster of ks CTAs per tile; the first CTA sums the
        // others' partial tiles, which must fit in its rings (with the
        // staging area too for the staged epilogue); every slice non-empty
        // and at least 4 pairs long
        for (int ks = 1; ks <= 8; ++ks) {
            int64_t waves = ceil_div(tiles, static_cast<int64_t>(sm_count));
            if (ks > 1) {
                if (np < 8 || ks > np / 4) break;
                if ((ks - 1) * ceil_div(np, ks) >= np) continue;
                if (static_cast<size_t>(ks - 1) * c.T * 512 > cap) continue;
                const int mc = gemm_max_clusters(ks, c.smem, threads);
                if (mc < 1) continue;
                waves = ceil_div(tiles, static_cast<int64_t>(mc));
            }
            const bool staged = static_cast<size_t>(ks) * c.T * 512 <= cap;
            const double cost = static_cast<double>(waves) * (kPairUs * static_cast<double>(ceil_div(np, ks)) + kWaveUs) +
                                (ks > 1 ? kSplitUs : 0.0) + (staged ? 0.0 : kDirectUs * c.T / 272.0);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best = c;
                best.ks = ks;
            }
        }
        if (ts > 4096) break;
    }
    if (best.T == 0) return false;
    best.est_us = best_cost;
    // Two blocks per SM: they run beside the GEMM CTA of the preceding call
    // (launched early, each waiting for that call to end) in one wave
    // whatever registers the GEMM holds; each thread converts several items.
    best.xcast_blocks = static_cast<int>(std::min<int64_t>(
        ceil_div(static_cast<int64_t>(best.ts) * np * best.T * 8, 256), 2 * static_cast<int64_t>(sm_count)));
    best.ws_ximg_off = 0;
    best.ws_bytes = static_cast<size_t>(best.ts) * np * best.T * 128;
    *plan = best;
    return true;
}

} // namespace

// Choose the token tile T (multiple of 16, at most 448 so that tensor memory
// keeps room for two weight stages), the number of token tiles and the K
// slices by the time model above, then the rings that fit in shared memory.
// Computed once per (device, shape, SM count).
bool plan_prefill(int64_t m, int64_t k, int64_t n, int sm_count, PrefillPlan *plan)
{
    if (m < 1 || sm_count < 1) return false;
    static std::mutex mu;
    static std::map<std::tuple<int, int64_t, int64_t, int64_t, int>, PrefillPlan> cache;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        dev = -1;
    }
    const auto key = std::make_tuple(dev, m, k, n, sm_count);
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            if (it->second.T == 0) return false;
            *plan = it->second;
            return true;
        }
    }
    PrefillPlan found;
    const bool ok = plan_prefill_search(m, k, n, sm_count, &found);
    if (dev >= 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache.emplace(key, ok ? found : PrefillPlan{});
    }
    if (!ok) return false;
    *plan = found;
    return true;
}

cudaError_t launch_prefill(const PrefillPlan &plan, const XcastArgs &xa, const PrefillArgs &pa, cudaStream_t s)
{
    {
        XcastArgs a = xa;
        void *kargs[] = {&a};
        const int64_t grid = std::max(1, plan.xcast_blocks);
        cudaError_t e = launch_pdl(reinterpret_cast<const void *>(&xcast_kernel), dim3(static_cast<unsigned>(grid)),
                                   dim3(256), 0, s, kargs);
        if (e != cudaSuccess) return e;
    }
    const void *fn = plan.ks > 1 ? reinterpret_cast<const void *>(&gemm_kernel<true>)
                                 : reinterpret_cast<const void *>(&gemm_kernel<false>);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    PrefillArgs a = pa;
    const TraceSettings tset = trace_settings();
    a.trace_buf = tset.buf;
    a.trace_cap = tset.cap;
    a.trace_cta = tset.cta;
    void *kargs[] = {&a};
    // warp 11 exists only when the tile takes two MMA threads (T >= 32)
    const int threads = plan.T >= 32 ? kThreads : kThreads - 32;
    return launch_pdl(fn, dim3(static_cast<unsigned>(plan.rowtiles * plan.ts * plan.ks)), dim3(threads), plan.smem, s,
                      kargs, plan.ks);
}

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

} // namespace q4
