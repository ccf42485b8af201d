// q4mm_decode.cu -- the memory-bound kernel for m <= 16 token rows: decode
// (m = 1) and continuous batching, where every active slot's token rides the
// same read of the weights (golem, "Several conversations, one pass"; golem-
// server, "Several conversations, in one pass"). The pages bound this case by
// the weight read (golem, "Qwen3.8 drafts its own next token": two columns
// cost what one did on the card) and goinfer ch. 10 ("What the kernels are")
// calls the quantised GEMV the decode workhorse.
//
// Design (GB300, one kernel per call and K range):
//   * A CTA owns 128 weight rows (one packed group) and a slice of K; the
//     slices of a group form one thread-block cluster (up to 8 CTAs).
//   * Warp 0: four producer lanes, each owning every fourth pair, stream the
//     4608-byte packed records through a shared-memory ring with 1-D bulk
//     copies (several independent rings keep tens of KB in flight per SM).
//   * Warps 2-9: each thread owns one weight row; it turns the pair's 64
//     split-half nibbles into fp16 (q - 8) * d, rounded once, and stores them
//     straight into tensor memory (tcgen05.st). No warp waits on a tensor
//     core result, so the CUDA cores only stream.
//   * Warp 1: one thread issues tcgen05.mma kind::f16: A = those weights
//     from tensor memory, B = X from shared memory, D = 128 x N fp32 in
//     tensor memory.
//   * Warps 10-13 stage X once per CTA while the first weights stream and
//     dequantise: every token row is scaled by a power of two (its largest
//     |x| in the slice lands in [2^14, 2^15)) and split into fp16 hi + lo,
//     22 significant bits, as the N = 16 (m <= 8) or N = 32 rows of the B
//     operand. They then run the epilogue.
//   * Epilogue: y = (D_hi + D_lo) / scale. Slices of a cluster add their
//     partial rows into the first CTA's shared memory (DSMEM) and that CTA
//     sums them in slice order, so results are bitwise reproducible and no
//     global scratch is needed. K ranges too long for one cluster run as
//     further launches that add into Y in order.
#include <algorithm>
#include <cuda_runtime.h>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5; // Q4_ERR_DEVICE_TIMEOUT
constexpr int kDequantWarps = 8;
constexpr int kXWarps = 4;          // stage X, then the epilogue (one per TMEM sub-partition)
constexpr int kXWarp0 = 2 + kDequantWarps;
constexpr int kXThreads = kXWarps * 32;
constexpr int kThreads = (2 + kDequantWarps + kXWarps) * 32;
constexpr int kProducerLanes = 4;
constexpr int kAStages = 7;        // weight stages in tensor memory (32 columns each)
constexpr int kAcol0 = 32;         // D uses columns 0..31
constexpr uint32_t kTmemCols = 256;
constexpr int kStageUnroll = 4;
constexpr int kMaxSlices = 8;

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

// One row's pair of blocks -> 32 fp16x2 columns of tensor memory (same
// column order as the X image): (q - 8) exact, times d, rounded once.
__device__ __forceinline__ void dequant_pair_f16(uint32_t d01, uint4 q0, uint4 q1, uint32_t out[32])
{
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const uint32_t h = blk ? (d01 >> 16) : (d01 & 0xFFFFu);
        const uint32_t dd = h | (h << 16);
        const uint4 q = blk ? q1 : q0;
        const uint32_t words[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int wd = 0; wd < 4; ++wd) {
            uint32_t v[4];
            unpack_word_f16(words[wd], v);
#pragma unroll
            for (int j = 0; j < 4; ++j) out[blk * 16 + wd * 4 + j] = hmul2_bits(v[j], dd);
        }
    }
}

struct Smem {
    uint8_t *xs, *w;
    float *red;
    uint64_t *full_w, *empty_w, *full_a, *empty_a, *done, *x_ready;
    uint32_t *tmem_slot;
    int *abort;
    unsigned *maxbits;    // [16] largest |x| bits per token
    float *scale_up;      // [16] 2^e per token
    float *scale_dn;      // [16] 2^-e per token
};

__device__ __forceinline__ bool aborted(const Smem &sm) { return *reinterpret_cast<volatile int *>(sm.abort) != 0; }

__device__ __forceinline__ void fail(const Smem &sm, const DecodeArgs &a)
{
    *reinterpret_cast<volatile int *>(sm.abort) = 1;
    record_status(a.status, kErrTimeout);
}

__device__ __forceinline__ void xwarps_sync()
{
    asm volatile("bar.sync 2, %0;" ::"n"(kXThreads) : "memory");
}

// Stage the slice of X (pairs p0 .. p0+P-1) as the scaled fp16 hi/lo image.
// Run by the kXThreads threads of the X warps; xt is the thread's index among
// them.
template <int N>
__device__ __forceinline__ void stage_x(const DecodeArgs &a, const Smem &sm, int p0, int P, int xt)
{
    constexpr int MP = N / 2;
    const int m = a.m;
    const int lane = xt & 31;
    const int kslice = P * 64;
    const int64_t col0 = static_cast<int64_t>(p0) * 64;
    const int64_t kreal = static_cast<int64_t>(a.nb) * 32;
    // 1. largest |x| of each token over the slice
    for (int t = 0; t < m; ++t) {
        const int64_t row = a.rows ? static_cast<int64_t>(a.rows[t]) : t;
        const float *xr = a.X + row * a.ldx + col0;
        unsigned mx = 0;
        for (int i = xt; i < kslice / 4; i += kXThreads) {
            if (col0 + 4 * i < kreal) {
                const float4 v = __ldg(reinterpret_cast<const float4 *>(xr) + i);
                mx = max(mx, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                                 max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = max(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0) atomicMax(&sm.maxbits[t], mx);
    }
    // zero the image (padded token rows and padded K stay zero)
    if (m < MP) {
        const int vecs = P * N * 8;
        for (int i = xt; i < vecs; i += kXThreads) sts128(sm.xs + i * 16, make_uint4(0u, 0u, 0u, 0u));
    }
    xwarps_sync();
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
    // 3. the split, item = (pair q, token t, chunk c); loads of kStageUnroll
    //    items in flight per thread
    const int items = P * m * 8;
    for (int base = xt; base < items; base += kXThreads * kStageUnroll) {
        float4 xa[kStageUnroll], xb[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int it = base + u * kXThreads;
            xa[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            xb[u] = xa[u];
            if (it < items) {
                const int c = it & 7, t = (it >> 3) % m, q = (it >> 3) / m;
                const int b = 2 * (p0 + q) + (c >> 2);
                if (b < a.nb) {
                    const int64_t row = a.rows ? static_cast<int64_t>(a.rows[t]) : t;
                    const float *xr = a.X + row * a.ldx + 32 * b + 4 * (c & 3);
                    xa[u] = __ldg(reinterpret_cast<const float4 *>(xr));
                    xb[u] = __ldg(reinterpret_cast<const float4 *>(xr + 16));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int it = base + u * kXThreads;
            if (it < items) {
                const int c = it & 7, t = (it >> 3) % m, q = (it >> 3) / m;
                const float su = sm.scale_up[t];
                const float v[8] = {xa[u].x, xa[u].z, xb[u].x, xb[u].z, xa[u].y, xa[u].w, xb[u].y, xb[u].w};
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
        }
    }
    // generic-proxy writes -> visible to the tensor core's shared-memory reads
    fence_proxy_async_smem();
    xwarps_sync();
    if (xt == 0) mbar_arrive(sm.x_ready);
}

template <int N>
__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeArgs a)
{
    constexpr int MP = N / 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int G = blockIdx.x / S;                   // 128-row group
    const int p0 = a.pass_p0 + rank * a.pbase + min(rank, a.prem);
    const int P = a.pbase + (rank < a.prem ? 1 : 0);
    const int R = a.ring;
    const int m = a.m;
    const TraceRef tr{a.trace_buf, a.trace_cap, a.trace_cta};
    trace_init();
    if (tid == 0) trace(tr, kTrStart, 0);

    Smem sm;
    sm.xs = base;
    sm.w = sm.xs + a.xs_bytes;
    sm.red = reinterpret_cast<float *>(sm.w + static_cast<size_t>(R) * kRecordBytes);
    const int red_floats = S > 1 ? (S - 1) * m * 128 : 0;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm.red + red_floats + (red_floats & 1));
    sm.full_w = bars;
    sm.empty_w = sm.full_w + R;
    sm.full_a = sm.empty_w + R;
    sm.empty_a = sm.full_a + kAStages;
    sm.done = sm.empty_a + kAStages;
    sm.x_ready = sm.done + 1;
    sm.tmem_slot = reinterpret_cast<uint32_t *>(sm.x_ready + 1);
    sm.abort = reinterpret_cast<int *>(sm.tmem_slot + 1);
    sm.maxbits = reinterpret_cast<unsigned *>(sm.abort + 1);
    sm.scale_up = reinterpret_cast<float *>(sm.maxbits + 16);
    sm.scale_dn = sm.scale_up + 16;

    if (tid == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&sm.full_w[i], 1), mbar_init(&sm.empty_w[i], kDequantWarps / 2);
        for (int i = 0; i < kAStages; ++i) mbar_init(&sm.full_a[i], kDequantWarps / 2), mbar_init(&sm.empty_a[i], 1);
        mbar_init(sm.done, 1);
        mbar_init(sm.x_ready, 1);
        *sm.abort = 0;
        fence_barrier_init();
    }
    if (tid < 16) sm.maxbits[tid] = 0u;
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (S > 1) cluster_sync(); // every CTA of the cluster is running before any DSMEM traffic
    const uint32_t tmem = *sm.tmem_slot;

    const uint8_t *wsrc = a.W + (static_cast<int64_t>(G) * a.np + p0) * kRecordBytes;
    const bool producer = warp == 0 && lane < kProducerLanes;
    const uint64_t pol = policy_evict_first();
    int w_next = lane; // producer lane: next pair (relative to p0) to issue
    auto issue = [&](int j) {
        const int s = j % R;
        trace(tr, kTrWIssue, static_cast<unsigned>(j));
        mbar_arrive_expect_tx(&sm.full_w[s], kRecordBytes);
        bulk_g2s_hint(sm.w + static_cast<size_t>(s) * kRecordBytes, wsrc + static_cast<size_t>(j) * kRecordBytes,
                      kRecordBytes, &sm.full_w[s], pol);
    };

    // Weights may stream before the preceding kernel has finished only when
    // the caller declared them read-only; X and Y are touched after the wait.
    if (producer && a.prefetch_w)
        for (; w_next < P && w_next < R; w_next += kProducerLanes) issue(w_next);
    pdl_wait();
    if (tid == 0) trace(tr, kTrPdl, 0);
    if (producer)
        for (; w_next < P && w_next < R; w_next += kProducerLanes) issue(w_next);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (producer) {
            int last = w_next - kProducerLanes;
            for (int j = w_next; j < P && !aborted(sm); j += kProducerLanes) {
                if (!mbar_wait(&sm.empty_w[j % R], ((j / R) & 1) ^ 1, a.wait_ns)) { fail(sm, a); break; }
                issue(j);
                last = j;
            }
            for (int j = last; j >= 0 && j > last - R; j -= kProducerLanes)
                if (!mbar_wait(&sm.full_w[j % R], (j / R) & 1, a.wait_ns)) fail(sm, a);
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idesc = idesc_f16_f32(128, N);
            const uint32_t xs0 = smem_u32(sm.xs);
            if (P > 0 && !mbar_wait(sm.x_ready, 0, a.wait_ns)) fail(sm, a);
            for (int j = 0; j < P && !aborted(sm); ++j) {
                const int sa = j % kAStages;
                if (!mbar_wait(&sm.full_a[sa], (j / kAStages) & 1, a.wait_ns)) { fail(sm, a); break; }
                trace(tr, kTrMmaIssue, static_cast<unsigned>(j));
                tc_fence_after();
                const uint32_t at = tmem + kAcol0 + static_cast<uint32_t>(sa) * 32u;
                const uint32_t bs = xs0 + static_cast<uint32_t>(j * N * 128);
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                    tc_mma_f16_ts(tmem, at + 8 * kk, smem_desc_sw128(bs + kk * 32), idesc, (j | kk) != 0);
                tc_commit(&sm.empty_a[sa]);
            }
            tc_commit(sm.done); // also taken on abort: no MMA of ours is in flight past this
        }
        __syncwarp();
    } else if (warp >= kXWarp0) {
        // ------------------------------------------------------------ stage X
        stage_x<N>(a, sm, p0, P, tid - kXWarp0 * 32);
        if (tid == kXWarp0 * 32) trace(tr, kTrXStaged, 0);
    } else {
        // -------------------------------------------------------- dequantise
        const int dw = warp - 2;
        const int q = warp & 3;
        const int h = dw >> 2;
        const int row = q * 32 + lane;
        const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
        for (int j = h; j < P && !aborted(sm); j += 2) {
            const int sw = j % R, sa = j % kAStages;
            if (!mbar_wait(&sm.full_w[sw], (j / R) & 1, a.wait_ns)) { fail(sm, a); break; }
            if (lane == 0) trace(tr, kTrWFull, static_cast<unsigned>(j));
            if (!mbar_wait(&sm.empty_a[sa], ((j / kAStages) & 1) ^ 1, a.wait_ns)) { fail(sm, a); break; }
            const uint8_t *rec = sm.w + static_cast<size_t>(sw) * kRecordBytes;
            const uint32_t d01 = *reinterpret_cast<const uint32_t *>(rec + kRecScaleOff + 4 * row);
            const uint4 q0 = lds128(rec + kRecQs0Off + 16 * row);
            const uint4 q1 = lds128(rec + kRecQs1Off + 16 * row);
            uint32_t out[32];
            dequant_pair_f16(d01, q0, q1, out);
            tmem_st_32x32b_x32(tmem + lane_base + kAcol0 + static_cast<uint32_t>(sa) * 32u, out);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.full_a[sa]);
                mbar_arrive(&sm.empty_w[sw]);
                trace(tr, kTrDeqDone, static_cast<unsigned>(j));
            }
        }
    }

    // ------------------------------------------------------------ epilogue
    // the X warps cover the four TMEM sub-partitions: thread = weight row
    const bool epi = warp >= kXWarp0;
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int64_t grow = static_cast<int64_t>(G) * kGroupRows + row;
    float y[MP];
#pragma unroll
    for (int t = 0; t < MP; ++t) y[t] = 0.f;
    if (epi) {
        if (!mbar_wait(sm.done, 0, a.wait_ns)) fail(sm, a);
        if (lane == 0) trace(tr, kTrDone, 0);
        tc_fence_after();
        uint32_t d[N];
        if constexpr (N == 16) {
            tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(q * 32) << 16), d);
        } else {
            tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(q * 32) << 16), d);
        }
        tmem_wait_ld();
        if (P > 0) {
#pragma unroll
            for (int t = 0; t < MP; ++t)
                if (t < m) y[t] = (__uint_as_float(d[t]) + __uint_as_float(d[MP + t])) * sm.scale_dn[t];
        }
        if (S > 1 && rank > 0) {
            const uint32_t dst = mapa_shared(smem_u32(sm.red), 0u);
#pragma unroll
            for (int t = 0; t < MP; ++t)
                if (t < m) st_cluster_f32(dst + static_cast<uint32_t>((((rank - 1) * m + t) * 128 + row) * 4), y[t]);
        }
    }
    pdl_launch_dependents();
    if (S > 1) cluster_sync(); // partial rows have landed in the first CTA
    if (epi && rank == 0 && grow < a.n) {
#pragma unroll
        for (int t = 0; t < MP; ++t) {
            if (t < m) {
                float v = y[t];
                for (int rr = 1; rr < S; ++rr) v += sm.red[((rr - 1) * m + t) * 128 + row];
                const int64_t yrow = a.rows ? static_cast<int64_t>(a.rows[t]) : t;
                float *dst = a.Y + yrow * a.ldy + grow;
                *dst = a.accumulate ? *dst + v : v;
            }
        }
    }

    if (epi && lane == 0) trace(tr, kTrEpiDone, 0);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
    if (tid == 0) trace(tr, kTrEnd, 0);
}

size_t decode_smem(int N, int P, int ring, int S, int64_t m)
{
    const size_t xs = static_cast<size_t>(round_up(static_cast<int64_t>(P) * N * 128, 1024));
    const size_t red = S > 1 ? static_cast<size_t>(S - 1) * m * 128 * 4 + 8 : 0;
    const size_t bars = static_cast<size_t>(2 * ring + 2 * kAStages + 2) * 8 + 16 + 48 * 4;
    return 1024 + xs + static_cast<size_t>(ring) * kRecordBytes + red + bars;
}

} // namespace

// Choose the cluster size S (K slices per 128-row group, at most 8) and the
// number of launches over K: the busiest SM's pair count plus a per-CTA
// start-up cost, with at most two CTAs per SM (tensor memory: 256 columns each).
bool plan_decode(int64_t m, int64_t k, int64_t n, int sm_count, DecodePlan *plan)
{
    if (m < 1 || m > 16) return false;
    const int N = m <= 8 ? 16 : 32;
    const int64_t tiles = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const int64_t xs_budget = 96 * 1024;
    const int64_t pmax = xs_budget / (N * 128);
    DecodePlan best;
    double best_cost = 1e300;
    for (int S = 1; S <= kMaxSlices; ++S) {
        if (S > np) break;
        const int64_t passes = ceil_div(np, S * pmax);
        const int64_t ppp = ceil_div(np, passes);          // pairs per pass
        if (ppp < S) continue;
        const int64_t P = ceil_div(ppp, S);
        const int ring = 8;
        size_t smem = decode_smem(N, static_cast<int>(P), ring, S, m);
        // at most two resident CTAs per SM, so that tensor memory always suffices
        smem = std::max<size_t>(smem, kSmemPerSM / 3 + 1024);
        if (smem > kSmemOptIn) continue;
        const int64_t units = tiles * S;
        const int64_t per_sm = ceil_div(units, sm_count);
        const double cost = static_cast<double>(passes) * per_sm * (static_cast<double>(P) + 6.0 + (S > 1 ? 2.0 : 0.0));
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best.N = N;
            best.S = S;
            best.passes = static_cast<int>(passes);
            best.pairs_per_pass = static_cast<int>(ppp);
            best.ring = ring;
            best.ctas = static_cast<int>(units);
            best.xs_bytes = static_cast<int>(round_up(P * N * 128, 1024));
            best.smem = smem;
        }
    }
    if (best.ctas == 0) return false;
    *plan = best;
    return true;
}

cudaError_t launch_decode(const DecodePlan &plan, const DecodeArgs &args, cudaStream_t s)
{
    const void *fn = plan.N == 16 ? reinterpret_cast<const void *>(&decode_kernel<16>)
                                  : reinterpret_cast<const void *>(&decode_kernel<32>);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    for (int pass = 0; pass < plan.passes; ++pass) {
        DecodeArgs a = args;
        a.pass_p0 = pass * plan.pairs_per_pass;
        const int pp = std::min(plan.pairs_per_pass, args.np - a.pass_p0);
        a.S = plan.S;
        a.pbase = pp / plan.S;
        a.prem = pp % plan.S;
        a.accumulate = pass > 0 ? 1 : 0;
        a.ring = plan.ring;
        a.xs_bytes = plan.xs_bytes;
        const TraceSettings ts = trace_settings();
        a.trace_buf = ts.buf;
        a.trace_cap = ts.cap;
        a.trace_cta = ts.cta;
        void *kargs[] = {&a};
        e = launch_pdl(fn, dim3(plan.ctas), dim3(kThreads), plan.smem, s, kargs, plan.S);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

} // namespace q4
