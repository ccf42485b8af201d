// q4mm_decode.cu -- the memory-bound kernel for m <= 16 token rows: decode
// (m = 1) and continuous batching, where every active slot's token rides the
// same read of the weights (golem, "Several conversations, one pass"; golem-
// server, "Several conversations, in one pass"). The pages bound this case by
// the weight read (golem, "Qwen3.8 drafts its own next token": two columns
// cost what one did on the card) and goinfer ch. 10 ("What the kernels are")
// calls the quantised GEMV the decode workhorse.
//
// Design (GB300): one persistent launch per call and K range.
//   * Work is split into 128-row groups (one packed group each) and S slices
//     of K. The S CTAs of a thread-block cluster hold the S slices and walk
//     the groups c, c + C, c + 2C, ... of their cluster c together, so each
//     CTA stages its slice of X once and streams weight records without a
//     break from one group to the next. Two CTAs fit on an SM.
//   * Warp 0: four producer lanes, each owning every fourth record of the
//     CTA's sequence, stream the 4608-byte packed records through a shared-
//     memory ring with 1-D bulk copies.
//   * Warps 3-10, two sets of four (one warp per TMEM sub-partition): each
//     thread owns one weight row; it turns a pair's 64 split-half nibbles into
//     fp16 (q - 8) * d, rounded once, and stores them straight into tensor
//     memory (tcgen05.st). The sets take alternate records.
//   * Warps 1-2: one thread each issues tcgen05.mma kind::f16 for every other
//     pair of a group into its own accumulator: A = those weights from tensor
//     memory, B = X from shared memory, D = 128 x N fp32 in tensor memory. A
//     single issuing warp can start an MMA only every ~50 cycles, whatever N
//     is; two keep the four MMAs of a pair well inside its HBM time. The
//     accumulators are double-buffered across groups.
//   * Warps 11-14 stage X: every token row is scaled by a power of two (its
//     largest |x| in the slice lands in [2^14, 2^15)) and split into fp16 hi
//     + lo, 22 significant bits, as the N = 16 (m <= 8) or N = 32 rows of the
//     B operand. They then drain each group's accumulators while the next
//     group streams: y = ((D0_hi + D0_lo) + (D1_hi + D1_lo)) / scale.
//   * Slices meet in the first CTA of the cluster: the others store their
//     partial rows into its shared memory (DSMEM) and signal an mbarrier
//     there; it sums them in slice order and writes Y, so results are
//     bitwise reproducible and no global scratch is needed. K ranges too long
//     for one cluster run as further launches that add into Y in order.
//   * Only the X warps wait for the preceding kernel (griddepcontrol.wait);
//     with weights declared read-only the producer streams, and the
//     dequantisers convert, before it has finished, and every CTA lets the
//     next kernel be scheduled as soon as it has started.
#include <algorithm>
#include <cuda_runtime.h>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5; // Q4_ERR_DEVICE_TIMEOUT
constexpr int kIssuers = 2;         // MMA-issuing warps, one accumulator each
constexpr int kXWarps = 4;          // stage X, then the epilogue (one per TMEM sub-partition)
constexpr int kDeqWarp0 = 1 + kIssuers;
constexpr int kXThreads = kXWarps * 32;

// Warp layout for SETS dequantiser sets (records u = set (mod SETS)), four
// warps each, one per TMEM sub-partition.
template <int SETS>
struct Warps {
    static constexpr int kXWarp0 = kDeqWarp0 + 4 * SETS;
    static constexpr int kThreads = (kXWarp0 + kXWarps) * 32;
};
constexpr int kProducerLanes = 4;
constexpr int kMaxRing = 12;        // weight records in flight per CTA (deeper only queues)
constexpr uint32_t kTmemCols = 256;
constexpr int kLoadBatch = 2;       // staging items (two float4 each) a thread keeps in flight
constexpr int kMaxSlices = 8;

// Tensor-memory map for MMA width N: accumulators [group parity][issuer]
// (N columns each), then dequantised weight stages of 32 columns.
template <int N>
struct Tmem {
    static constexpr int kDCols = 2 * kIssuers * N;
    static constexpr int kAcol0 = kDCols;
    static constexpr int kAStages = (static_cast<int>(kTmemCols) - kDCols) / 32;
    static_assert(kAStages >= 2 && kAStages % kIssuers == 0, "tensor memory layout");
};

// X image: per pair, N rows (hi tokens, then lo tokens) x 128 bytes, 128-byte
// swizzle, chunk c = 4 blk + quad holding block elements 4 quad + {0,2,16,18,
// 1,3,17,19}: the order dequant_pair_f16 writes the weights in.
__device__ __forceinline__ uint32_t ximg_off(int N, int q, int row, int c)
{
    return static_cast<uint32_t>(q * N * 128 + row * 128 + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ uint32_t f16_bits(float x)
{
    return static_cast<uint32_t>(__half_as_ushort(__float2half_rn(x)));
}

// hi + lo fp16 split of an already scaled value.
__device__ __forceinline__ void split_f16(float xs, uint32_t &hi, uint32_t &lo)
{
    hi = f16_bits(xs);
    const float r = xs - __half2float(__ushort_as_half(static_cast<unsigned short>(hi)));
    lo = isfinite(r) ? f16_bits(r) : 0u;
}

// One row's block -> 16 fp16x2 columns of tensor memory (same column order
// as the X image): (q - 8) exact, times d, rounded once.
__device__ __forceinline__ void dequant_block_f16(uint32_t dbits, uint4 q, uint32_t out[16])
{
    const uint32_t dd = dbits | (dbits << 16);
    const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t v[4];
        unpack_word_f16(words[wd], v);
#pragma unroll
        for (int j = 0; j < 4; ++j) out[wd * 4 + j] = hmul2_bits(v[j], dd);
    }
}

struct Smem {
    uint8_t *xs, *w;
    float *red;           // [2][S - 1][m][128] partial rows (first CTA of the cluster)
    uint64_t *full_w, *empty_w, *full_a, *empty_a;
    uint64_t *dfull, *dfree;       // [2] accumulators of a group parity ready / drained
    uint64_t *red_full, *red_free; // [2] partials landed (first CTA) / slot free (others)
    uint64_t *x_ready;
    uint32_t *tmem_slot;
    unsigned *maxbits;    // [16] largest |x| bits per token
    float *scale_up;      // [16] 2^e per token
    float *scale_dn;      // [16] 2^-e per token
    int *rowid;           // [16] X / Y row of each token
};

__device__ __forceinline__ void fail(const DecodeArgs &a) { record_status(a.status, kErrTimeout); }

// Bounded wait by every lane of a warp, with one outcome for the whole warp,
// so that a timeout never leaves a warp diverged in front of the .aligned
// tcgen05 instructions that follow.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns)) != 0;
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar, parity, limit_ns)) != 0;
}

__device__ __forceinline__ void xwarps_sync()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kXThreads) : "memory");
}

// Zero the token rows of the X image that no token fills (m < N / 2). Needs
// nothing from the preceding kernel, so it runs before the dependency wait.
template <int N>
__device__ __forceinline__ void zero_x_padding(const Smem &sm, int m, int P, int xt)
{
    constexpr int MP = N / 2;
    const int pad = MP - m;     // padded rows per half
    if (pad <= 0) return;
    const int per_pair = 2 * pad * 8;
    for (int i = xt; i < P * per_pair; i += kXThreads) {
        const int q = i / per_pair, r = i - q * per_pair;
        const int half = r / (pad * 8), rr = r - half * pad * 8;
        const int row = half * MP + m + (rr >> 3);
        sts128(sm.xs + q * N * 128 + row * 128 + (rr & 7) * 16, make_uint4(0u, 0u, 0u, 0u));
    }
}

// Loads of one staging item: token t, pair q, chunk c (block c >> 2, quad
// c & 3) = block elements 4 quad .. 4 quad + 3 and 16 + 4 quad .. + 3.
__device__ __forceinline__ void load_item(const DecodeArgs &a, const Smem &sm, int p0, int it, float4 &xa, float4 &xb)
{
    const int m = a.m;
    const int c = it & 7, t = (it >> 3) % m, q = (it >> 3) / m;
    const int b = 2 * (p0 + q) + (c >> 2);
    xa = make_float4(0.f, 0.f, 0.f, 0.f);
    xb = xa;
    if (b < a.nb) {
        const float *xr = a.X + static_cast<int64_t>(sm.rowid[t]) * a.ldx + 32 * b + 4 * (c & 3);
        xa = __ldg(reinterpret_cast<const float4 *>(xr));
        xb = __ldg(reinterpret_cast<const float4 *>(xr + 16));
    }
}

__device__ __forceinline__ unsigned absmax_bits(const float4 &v)
{
    return max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
               max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu));
}

template <int N>
__device__ __forceinline__ void store_item(const DecodeArgs &a, const Smem &sm, int it, const float4 &xa, const float4 &xb)
{
    constexpr int MP = N / 2;
    const int m = a.m;
    const int c = it & 7, t = (it >> 3) % m, q = (it >> 3) / m;
    const float su = sm.scale_up[t];
    const float v[8] = {xa.x, xa.z, xb.x, xb.z, xa.y, xa.w, xb.y, xb.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t h0, l0, h1, l1;
        split_f16(v[2 * i] * su, h0, l0);
        split_f16(v[2 * i + 1] * su, h1, l1);
        hw[i] = h0 | (h1 << 16);
        lw[i] = l0 | (l1 << 16);
    }
    sts128(sm.xs + ximg_off(N, q, t, c), make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(sm.xs + ximg_off(N, q, MP + t, c), make_uint4(lw[0], lw[1], lw[2], lw[3]));
}

// Stage the slice of X (pairs p0 .. p0+P-1) as the scaled fp16 hi/lo image.
// Run by the kXThreads threads of the X warps after the dependency wait; xt
// is the thread's index among them. The first kLoadBatch items of every
// thread stay in registers between the two passes, so a slice of up to
// kXThreads * kLoadBatch items costs one round trip to memory.
template <int N>
__device__ __forceinline__ void stage_x(const DecodeArgs &a, const Smem &sm, int p0, int P, int xt, const TraceRef &tr)
{
    const int m = a.m;
    if (xt < m) sm.rowid[xt] = a.rows ? a.rows[xt] : xt;
    xwarps_sync();
    const int items = P * m * 8;
    // 1. largest |x| of each token over the slice
    float4 ra[kLoadBatch], rb[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
        const int it = xt + u * kXThreads;
        if (it < items) load_item(a, sm, p0, it, ra[u], rb[u]);
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
        const int it = xt + u * kXThreads;
        if (it < items) atomicMax(&sm.maxbits[(it >> 3) % m], max(absmax_bits(ra[u]), absmax_bits(rb[u])));
    }
    for (int base = xt + kLoadBatch * kXThreads; base < items; base += kLoadBatch * kXThreads) {
        float4 va[kLoadBatch], vb[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int it = base + u * kXThreads;
            if (it < items) load_item(a, sm, p0, it, va[u], vb[u]);
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int it = base + u * kXThreads;
            if (it < items) atomicMax(&sm.maxbits[(it >> 3) % m], max(absmax_bits(va[u]), absmax_bits(vb[u])));
        }
    }
    xwarps_sync();
    if (xt == 0) trace(tr, kTrXLoaded, 0);
    // 2. per-token power of two: largest |x| into [2^14, 2^15)
    if (xt < m) {
        const unsigned mb = sm.maxbits[xt];
        int e = 0;
        if (mb != 0 && mb < 0x7F800000u) {
            const int E = static_cast<int>(mb >> 23) - 126; // |x|max = f * 2^E, f in [0.5, 1) (normal)
            e = (mb >> 23) == 0 ? 100 : 15 - E;
            e = max(-100, min(100, e));
        }
        sm.scale_up[xt] = __uint_as_float(static_cast<unsigned>(e + 127) << 23);
        sm.scale_dn[xt] = __uint_as_float(static_cast<unsigned>(127 - e) << 23);
    }
    xwarps_sync();
    if (xt == 0) trace(tr, kTrXScaled, 0);
    // 3. the split: first batch from registers, the rest reloaded (L1 hits)
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
        const int it = xt + u * kXThreads;
        if (it < items) store_item<N>(a, sm, it, ra[u], rb[u]);
    }
    for (int base = xt + kLoadBatch * kXThreads; base < items; base += kLoadBatch * kXThreads) {
        float4 va[kLoadBatch], vb[kLoadBatch];
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int it = base + u * kXThreads;
            if (it < items) load_item(a, sm, p0, it, va[u], vb[u]);
        }
#pragma unroll
        for (int u = 0; u < kLoadBatch; ++u) {
            const int it = base + u * kXThreads;
            if (it < items) store_item<N>(a, sm, it, va[u], vb[u]);
        }
    }
    // generic-proxy writes -> visible to the tensor core's shared-memory reads
    fence_proxy_async_smem();
    xwarps_sync();
    if (xt == 0) mbar_arrive(sm.x_ready);
}

// Every barrier of the pipeline has a single waiter agent that sees all of
// its phases in order (a parity wait is only sound that way): ring slot s is
// always refilled by producer lane s % 4 and drained by set s % SETS (the
// ring depth is a multiple of both), and stage s is always written by set
// s % SETS and read by issuer s % 2 (the stage count is a multiple of both).
template <int N, int SETS>
__global__ void __launch_bounds__(Warps<SETS>::kThreads, 2) decode_kernel(const DecodeArgs a)
{
    constexpr int MP = N / 2;
    constexpr int AS = Tmem<N>::kAStages;
    constexpr int kAcol0 = Tmem<N>::kAcol0;
    constexpr int kXWarp0 = Warps<SETS>::kXWarp0;
    static_assert(AS % SETS == 0, "a stage must always belong to one dequantiser set");
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int G0 = blockIdx.x / S;                  // first group of this cluster
    const int stride = a.clusters;
    const int ntiles = G0 < a.groups ? (a.groups - 1 - G0) / stride + 1 : 0;
    const int p0 = a.pass_p0 + rank * a.pbase + min(rank, a.prem);
    const int P = a.pbase + (rank < a.prem ? 1 : 0);
    const int total = ntiles * P;                    // records this CTA streams
    const int m = a.m;
    const TraceRef tr{a.trace_buf, a.trace_cap, a.trace_cta};
    trace_init();
    if (tid == 0) trace(tr, kTrStart, 0);

    Smem sm;
    sm.xs = base;
    sm.w = sm.xs + a.xs_bytes;
    const int R = a.ring;
    sm.red = reinterpret_cast<float *>(sm.w + static_cast<size_t>(R) * kRecordBytes);
    const int red_floats = S > 1 ? 2 * (S - 1) * m * 128 : 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm.red + red_floats + (red_floats & 1));
    sm.full_w = bars;
    sm.empty_w = sm.full_w + R;
    sm.full_a = sm.empty_w + R;
    sm.empty_a = sm.full_a + AS;
    sm.dfull = sm.empty_a + AS;
    sm.dfree = sm.dfull + 2;
    sm.red_full = sm.dfree + 2;
    sm.red_free = sm.red_full + 2;
    sm.x_ready = sm.red_free + 2;
    sm.tmem_slot = reinterpret_cast<uint32_t *>(sm.x_ready + 1);
    sm.maxbits = reinterpret_cast<unsigned *>(sm.tmem_slot + 1);
    sm.scale_up = reinterpret_cast<float *>(sm.maxbits + 16);
    sm.scale_dn = sm.scale_up + 16;
    sm.rowid = reinterpret_cast<int *>(sm.scale_dn + 16);

    if (tid == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&sm.full_w[i], 1), mbar_init(&sm.empty_w[i], 4);
        for (int i = 0; i < AS; ++i) mbar_init(&sm.full_a[i], 4), mbar_init(&sm.empty_a[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.dfull[i], kIssuers);
            mbar_init(&sm.dfree[i], kXWarps);
            mbar_init(&sm.red_full[i], S > 1 ? kXWarps * (S - 1) : 1);
            mbar_init(&sm.red_free[i], kXWarps);
        }
        mbar_init(sm.x_ready, 1);
        fence_barrier_init();
    }
    if (tid < 16) sm.maxbits[tid] = 0u;
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, kTmemCols);
        tmem_relinquish();
        if (lane == 0) trace(tr, kTrAlloc, 0);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // The next kernel in the stream may be scheduled now: it waits for this
    // one to complete before it reads anything this one writes.
    pdl_launch_dependents();
    if (tid == 0) trace(tr, kTrSetup, 0);
    if (S > 1) cluster_sync(); // barriers of every CTA initialised before any remote arrive
    const uint32_t tmem = *sm.tmem_slot;
    if (tid == 0) trace(tr, kTrSetup, 1);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // Weights may stream before the preceding kernel has finished only
        // when the caller declared them read-only.
        if (!a.prefetch_w) pdl_wait();
        if (lane < kProducerLanes && total > 0) {
            const uint64_t pol = policy_evict_first();
            // record u = lane, lane + 4, ...: group i, pair j, ring slot s
            int i = 0, j = lane, s = lane, last = -1;
            uint32_t ph = 0;
            while (j >= P) j -= P, ++i;
            for (int u = lane; u < total; u += kProducerLanes) {
                if (u >= R && !mbar_wait(&sm.empty_w[s], ph ^ 1u, a.wait_ns)) { fail(a); break; }
                trace(tr, kTrWIssue, static_cast<unsigned>(u));
                const int64_t rec = static_cast<int64_t>(G0 + i * stride) * a.np + p0 + j;
                mbar_arrive_expect_tx(&sm.full_w[s], kRecordBytes);
                bulk_g2s_hint(sm.w + static_cast<size_t>(s) * kRecordBytes, a.W + rec * kRecordBytes, kRecordBytes,
                              &sm.full_w[s], pol);
                last = u;
                s += kProducerLanes;
                if (s >= R) s -= R, ph ^= 1u;
                j += kProducerLanes;
                while (j >= P) j -= P, ++i;
            }
            // No copy of ours may still be landing when the CTA exits. A record
            // whose slot a later record reused has landed (and been consumed)
            // already; only the last R records of the sequence need a wait.
            for (int u = last; u >= 0 && u >= total - R; u -= kProducerLanes)
                if (!mbar_wait(&sm.full_w[u % R], (u / R) & 1, a.wait_ns)) fail(a);
        }
        __syncwarp();
    } else if (warp < kDeqWarp0) {
        // --------------------------------------------------------------- MMA
        // Issuer e owns the records u = e (mod kIssuers) -- in group i the
        // pairs j = e + i P (mod 2) -- and the accumulator [group parity][e].
        // Descriptor arithmetic is hoisted so the four MMAs of a pair issue
        // back to back.
        const int e = warp - 1;
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, N);
            const uint64_t bdesc0 = smem_desc_sw128(smem_u32(sm.xs));
            constexpr uint64_t kPairStep = static_cast<uint64_t>((N * 128) >> 4);
            bool ok = ntiles == 0 || mbar_wait(sm.x_ready, 0, a.wait_ns);
            for (int i = 0; ok && i < ntiles; ++i) {
                const int tb = i & 1;
                const int j0 = (e + i * P) & 1;
                if (j0 < P) {
                    if (i >= 2 && !mbar_wait(&sm.dfree[tb], ((i >> 1) & 1) ^ 1, a.wait_ns)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem + static_cast<uint32_t>((tb * kIssuers + e) * N);
                    uint64_t bdesc = bdesc0 + kPairStep * static_cast<uint64_t>(j0);
                    uint32_t acc = 0;
                    for (int j = j0; j < P; j += kIssuers) {
                        const int u = i * P + j;
                        const int sa = u % AS;
                        if (!mbar_wait(&sm.full_a[sa], (u / AS) & 1, a.wait_ns)) { ok = false; break; }
                        trace(tr, kTrMmaIssue, static_cast<unsigned>(u));
                        tc_fence_after();
                        const uint32_t at = tmem + static_cast<uint32_t>(kAcol0 + sa * 32);
                        tc_mma_f16_ts(d_tmem, at, bdesc, idesc, acc);
                        tc_mma_f16_ts(d_tmem, at + 8u, bdesc + 2u, idesc, 1u);
                        tc_mma_f16_ts(d_tmem, at + 16u, bdesc + 4u, idesc, 1u);
                        tc_mma_f16_ts(d_tmem, at + 24u, bdesc + 6u, idesc, 1u);
                        tc_commit(&sm.empty_a[sa]);
                        acc = 1u;
                        bdesc += kIssuers * kPairStep;
                    }
                    if (!ok) break;
                }
                tc_commit(&sm.dfull[tb]); // the group's MMAs of this issuer are done (at once if it had none)
            }
            // The tensor core's arrivals on the stage barriers must all have
            // landed before the CTA exits: wait for the last use of each stage.
            if (ok && e == 0)
                for (int st = 0; st < AS && st < total; ++st) {
                    const int u = st + AS * ((total - 1 - st) / AS);
                    if (!mbar_wait(&sm.empty_a[st], (u / AS) & 1, a.wait_ns)) { ok = false; break; }
                }
            if (!ok) fail(a);
        }
        __syncwarp();
    } else if (warp < kXWarp0) {
        // -------------------------------------------------------- dequantise
        // Set h converts records u = h (mod SETS), one block at a time.
        const int dw = warp - kDeqWarp0;
        const int q = warp & 3;              // TMEM sub-partition this warp may access
        const int h = dw >> 2;
        const int row = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        int sw = h, sa = h;                  // ring slot and tensor-memory stage of record u
        uint32_t phw = 0, pha = 0;
        for (int u = h; u < total; u += SETS) {
            if (!warp_wait(&sm.full_w[sw], phw, a.wait_ns)) { fail(a); break; }
            if (lane == 0) trace(tr, kTrWFull, static_cast<unsigned>(u));
            const uint8_t *rec = sm.w + static_cast<size_t>(sw) * kRecordBytes;
            const uint32_t d01 = *reinterpret_cast<const uint32_t *>(rec + kRecScaleOff + 4 * row);
            const uint4 q0 = lds128(rec + kRecQs0Off + 16 * row);
            const uint4 q1 = lds128(rec + kRecQs1Off + 16 * row);
            uint32_t out[16];
            dequant_block_f16(d01 & 0xFFFFu, q0, out);
            if (u >= AS && !warp_wait(&sm.empty_a[sa], pha ^ 1u, a.wait_ns)) { fail(a); break; }
            tc_fence_after();
            const uint32_t ta = tmem + lane_base + static_cast<uint32_t>(kAcol0 + sa * 32);
            tmem_st_32x32b_x16(ta, out);
            dequant_block_f16(d01 >> 16, q1, out);
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty_w[sw]);   // the record has been consumed
            tmem_st_32x32b_x16(ta + 16u, out);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.full_a[sa]);
                trace(tr, kTrDeqDone, static_cast<unsigned>(u));
            }
            sw += SETS;
            if (sw >= R) sw -= R, phw ^= 1u;
            sa += SETS;
            if (sa >= AS) sa -= AS, pha ^= 1u;
        }
    } else {
        // ------------------------------------------------ stage X, epilogue
        const int xt = tid - kXWarp0 * 32;
        zero_x_padding<N>(sm, m, P, xt);
        pdl_wait();
        if (xt == 0) trace(tr, kTrPdl, 0);
        stage_x<N>(a, sm, p0, P, xt, tr);
        if (xt == 0) trace(tr, kTrXStaged, 0);

        // thread = weight row of the group, in this warp's TMEM sub-partition
        const int q = warp & 3;
        const int row = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        const uint32_t red0 = smem_u32(sm.red);
        for (int i = 0; i < ntiles; ++i) {
            const int tb = i & 1;
            const uint32_t par = static_cast<uint32_t>((i >> 1) & 1);
            if (!warp_wait(&sm.dfull[tb], par, a.wait_ns)) { fail(a); break; }
            tc_fence_after();
            // y = (((D0_hi + D0_lo) + D1_hi) + D1_lo) * 2^-e, in this order;
            // 8 columns per load (hi rows 0..MP-1, then lo rows)
            float y[MP];
#pragma unroll
            for (int t = 0; t < MP; ++t) y[t] = 0.f;
#pragma unroll
            for (int e = 0; e < kIssuers; ++e) {
                if (((e + i * P) & 1) >= P) continue;   // issuer e had no pair of this group
#pragma unroll
                for (int c0 = 0; c0 < N; c0 += 8) {
                    uint32_t d[8];
                    tmem_ld_32x32b_x8(tmem + lane_base + static_cast<uint32_t>((tb * kIssuers + e) * N + c0), d);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const int t = (c0 + c) % MP;
                        if (t < m) y[t] += __uint_as_float(d[c]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.dfree[tb]);
#pragma unroll
            for (int t = 0; t < MP; ++t)
                if (t < m) y[t] *= sm.scale_dn[t];

            const int64_t grow = static_cast<int64_t>(G0 + i * stride) * kGroupRows + row;
            if (rank > 0) {
                // partial rows into the first CTA's slot tb, then signal it
                if (i >= 2 && !warp_wait_cluster(&sm.red_free[tb], par ^ 1u, a.wait_ns)) { fail(a); break; }
                const uint32_t dst = mapa_shared(red0, 0u) +
                                     static_cast<uint32_t>((((tb * (S - 1) + rank - 1) * m) * 128 + row) * 4);
#pragma unroll
                for (int t = 0; t < MP; ++t)
                    if (t < m) st_cluster_f32(dst + static_cast<uint32_t>(t * 128 * 4), y[t]);
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_full[tb]), 0u));
            } else {
                if (S > 1 && !warp_wait_cluster(&sm.red_full[tb], par, a.wait_ns)) { fail(a); break; }
                if (grow < a.n) {
#pragma unroll
                    for (int t = 0; t < MP; ++t) {
                        if (t < m) {
                            float v = y[t];
                            for (int r = 1; r < S; ++r) v += sm.red[((tb * (S - 1) + r - 1) * m + t) * 128 + row];
                            float *dst = a.Y + static_cast<int64_t>(sm.rowid[t]) * a.ldy + grow;
                            *dst = a.accumulate ? *dst + v : v;
                        }
                    }
                }
                if (S > 1) {
                    __syncwarp();
                    if (lane == 0)
                        for (int r = 1; r < S; ++r)
                            mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_free[tb]), static_cast<uint32_t>(r)));
                }
            }
            if (lane == 0) trace(tr, kTrTile, static_cast<unsigned>(i));
        }
        if (lane == 0) trace(tr, kTrEpiDone, 0);
    }

    // every CTA of the cluster stays until the others are done with its
    // shared memory and barriers
    if (S > 1) cluster_sync();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0) trace(tr, kTrEnd, 0);
}

size_t decode_smem(int N, int P, int S, int64_t m, int ring)
{
    const int as = N == 16 ? Tmem<16>::kAStages : Tmem<32>::kAStages;
    const size_t xs = static_cast<size_t>(round_up(static_cast<int64_t>(P) * N * 128, 1024));
    const size_t red = S > 1 ? static_cast<size_t>(2 * (S - 1)) * m * 128 * 4 + 8 : 0;
    const size_t bars = static_cast<size_t>(2 * ring + 2 * as + 9) * 8 + 4 + 64 * 4;
    return 1024 + xs + static_cast<size_t>(ring) * kRecordBytes + red + bars;
}

} // namespace

// Choose the cluster size S (K slices per 128-row group, at most 8), the
// number of persistent clusters, the number of launches over K and the ring
// depth. Two CTAs share an SM (shared and tensor memory are sized for that).
// Cost, in record times of one SM's share of HBM: the busiest SM's records,
// or one CTA's records at the rate a single CTA's ring sustains (kCtaRate of
// the share at a ring of 8, in proportion to the ring), whichever is larger,
// plus per-group and per-CTA overheads, plus the start-up time that cannot
// overlap the preceding call when every SM already holds two CTAs.
bool plan_decode(int64_t m, int64_t k, int64_t n, int sm_count, DecodePlan *plan)
{
    if (m < 1 || m > 16 || sm_count < 1) return false;
    constexpr double kCtaRate = 0.6;
    const int N = m <= 8 ? 16 : 32;
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const size_t smem_min = kSmemPerSM / 3 + 1024;          // never three (tensor memory)
    DecodePlan best;
    double best_cost = 1e300;
    // Shared memory for two CTAs per SM, or, for N = 32, all of it for one
    // (wide): the N = 32 image of X and the slices' reduction buffer leave a
    // half-SM CTA only a shallow ring or several K passes (measured: the
    // 151936x2560 m = 16 layer 158 -> 101 us, 9728x2560 m = 16 35.8 -> 26.4
    // us). For N = 16 the wide plans the cost below prefers run slower
    // (2560x9728 m = 4: 15.5 -> 29.4 us). A wide CTA leaves no room for the
    // next call's, but K passes cost more than that overlap does.
    for (int wide = 0; wide <= (N == 32 ? 1 : 0); ++wide)
    for (int S = 1; S <= kMaxSlices && S <= np; ++S) {
        const size_t smem_max = wide ? kSmemOptIn - 1024 : kSmemPerSM / 2 - 1024 - 512;
        for (int64_t passes = 1; passes <= np; ++passes) {
            const int64_t ppp = ceil_div(np, passes);        // pairs per pass
            if (ppp < S) break;
            const int64_t P = ceil_div(ppp, S);
            // ring: a multiple of the four producer lanes and of the sets
            auto fits = [&](int r) { return decode_smem(N, static_cast<int>(P), S, m, r) <= smem_max; };
            int sets = 2, ring = 0;
            if (N == 16 && fits(12)) {
                sets = 3;
                ring = 12;
            } else {
                for (int r = kMaxRing; r >= 4 && ring == 0; r -= 4)
                    if (fits(r)) ring = r;
            }
            if (ring == 0) continue;                          // more passes: smaller slices
            const size_t smem = std::max(decode_smem(N, static_cast<int>(P), S, m, ring), smem_min);
            // a wide CTA holds its SM alone; otherwise one CTA per SM (room
            // for the next call to overlap) or two
            if (wide && smem <= kSmemPerSM / 2 - 1024 - 512) break;      // not wide after all
            for (int per = 1; per <= (wide ? 1 : 2); ++per) {
                const int64_t clusters = std::min<int64_t>(groups, (per * sm_count) / S);
                if (clusters < 1) continue;
                const int64_t tiles_per = ceil_div(groups, clusters);
                const int64_t ctas = clusters * S;
                const double cta_pairs = static_cast<double>(tiles_per * P);
                const double sm_pairs = (ctas > sm_count ? 2.0 : 1.0) * cta_pairs;
                const double rate = std::min(1.0, kCtaRate * ring / 8.0);
                const double stream =
                    std::max({sm_pairs, cta_pairs / rate, static_cast<double>(groups * ppp) / sm_count});
                // A grid of more than one CTA per SM leaves no room for the next
                // call's CTAs to start streaming while this one finishes.
                const double no_overlap = ctas > sm_count ? 12.0 : 0.0;
                const double cost = static_cast<double>(passes) *
                                    (stream + static_cast<double>(tiles_per) * (1.5 + (S > 1 ? 1.0 : 0.0)) + 6.0 +
                                     no_overlap);
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best.N = N;
                    best.S = S;
                    best.passes = static_cast<int>(passes);
                    best.pairs_per_pass = static_cast<int>(ppp);
                    best.clusters = static_cast<int>(clusters);
                    best.ctas = static_cast<int>(ctas);
                    best.ring = ring;
                    best.sets = sets;
                    best.xs_bytes = static_cast<int>(round_up(P * N * 128, 1024));
                    best.smem = smem;
                }
            }
            break;                                            // fewest passes that fit
        }
    }
    if (best.ctas == 0) return false;
    *plan = best;
    return true;
}

cudaError_t launch_decode(const DecodePlan &plan, const DecodeArgs &args, cudaStream_t s)
{
    const void *fn = plan.N == 32  ? reinterpret_cast<const void *>(&decode_kernel<32, 2>)
                     : plan.sets == 3 ? reinterpret_cast<const void *>(&decode_kernel<16, 3>)
                                      : reinterpret_cast<const void *>(&decode_kernel<16, 2>);
    const int threads = plan.sets == 3 ? Warps<3>::kThreads : Warps<2>::kThreads;
    if (plan.N == 32 && plan.sets != 2) return cudaErrorInvalidValue;
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    for (int pass = 0; pass < plan.passes; ++pass) {
        DecodeArgs a = args;
        a.pass_p0 = pass * plan.pairs_per_pass;
        const int pp = std::min(plan.pairs_per_pass, args.np - a.pass_p0);
        a.S = plan.S;
        a.pbase = pp / plan.S;
        a.prem = pp % plan.S;
        a.clusters = plan.clusters;
        a.ring = plan.ring;
        a.accumulate = pass > 0 ? 1 : 0;
        a.xs_bytes = plan.xs_bytes;
        const TraceSettings ts = trace_settings();
        a.trace_buf = ts.buf;
        a.trace_cap = ts.cap;
        a.trace_cta = ts.cta;
        void *kargs[] = {&a};
        e = launch_pdl(fn, dim3(plan.ctas), dim3(threads), plan.smem, s, kargs, plan.S);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace q4
