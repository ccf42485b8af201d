// q4mm_decode.cu -- the memory-bound kernel for m <= 16 token rows: decode
// (m = 1) and continuous batching, where every active slot's token rides the
// same read of the weights (golem, "Several conversations, one pass"; golem-
// server, "Several conversations, in one pass"). The pages bound this case by
// the weight read (golem, "Qwen3.8 drafts its own next token": two columns
// cost what one did on the card) and goinfer ch. 10 ("What the kernels are")
// calls the quantised GEMV the decode workhorse.
//
// Design (GB300, one kernel per call):
//   * Persistent CTAs of 16 warps (8 when m > 8). CTA c owns a K
//     slice (when one is needed) and a strided set of 64-row groups. Each
//     warp streams its own share of every group's pairs (2304 contiguous
//     bytes per pair) through a private ring of shared-memory stages filled
//     by 1-D bulk async copies (TMA engine, L2 evict-first), so each SM keeps
//     tens of KB of weight reads in flight.
//   * X is staged once per CTA for its K slice: each fp32 value becomes a
//     two-term bf16 split (hi = truncation, lo = rounded remainder, 16
//     significant bits) laid out in mma fragment order. All of a thread's
//     global loads are issued before any is used, so staging costs about one
//     memory latency, and it overlaps the first weight copies.
//   * The split-half nibbles become exact bf16 (q - 8) in registers (mask
//     into a biased exponent, subtract 136); warp-level bf16 MMAs
//     (m16n8k16, fp32 accumulate) form each block's exact integer-weighted
//     partial sum, which is scaled by the block's fp16 d in fp32 and
//     accumulated. Tensor cores here only replace CUDA-core FMAs: the kernel
//     stays bound by the weight bytes.
//   * The warps' partials of a group are added in a fixed order through
//     shared memory. With K slices, each slice writes its partial to the
//     workspace and the last slice to finish (a counter) adds all slices in
//     slice order, so results are bitwise reproducible.
#include <algorithm>
#include <cuda_runtime.h>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5; // Q4_ERR_DEVICE_TIMEOUT
constexpr int kStageUnroll = 4; // X items whose loads are in flight together

// Warps per CTA: 16 (four per SM sub-partition, at most 128 registers) for
// one n-tile; 8 for two n-tiles, whose accumulators need more registers.
__host__ __device__ constexpr int warps_for(int NT) { return NT == 1 ? 16 : 8; }

// Shared-memory bytes of the X region per pair: NT x 2 blocks x (hi, lo) x 512.
__host__ __device__ constexpr int xs_pair_bytes(int NT) { return NT * 2048; }
__host__ __device__ constexpr int red_bytes(int NT) { return warps_for(NT) * NT * 8 * 64 * 4; }

struct Split {
    uint32_t hi, lo; // bf16 bits
};

// x = hi + lo with hi the bf16 truncation of x and lo the remainder rounded to
// bf16: 16 significant bits in all, and no overflow near FLT_MAX.
__device__ __forceinline__ Split split_bf16(float x)
{
    uint32_t u = __float_as_uint(x);
    uint32_t hb = u & 0xFFFF0000u;
    float r = x - __uint_as_float(hb);
    if (!isfinite(x)) {
        r = 0.0f;
        if (isnan(x)) hb = 0x7FC00000u;
    }
    return {hb >> 16, bf16_rn_bits(r)};
}

// Fragment-order X region: [pair q][n-tile][blk][hi | lo][lane][16 B]; lane
// L = 4g + c holds token (8 nt + g), block elements 4c + {0,2,16,18,1,3,17,19}.
__device__ __forceinline__ uint8_t *xs_slot(uint8_t *xs, int NT, int q, int tok, int blk, int c)
{
    const int nt = tok >> 3, L = ((tok & 7) << 2) | c;
    return xs + ((q * NT + nt) * 2 + blk) * 1024 + L * 16;
}

__device__ __forceinline__ void store_split(uint8_t *dst, float4 xa, float4 xb)
{
    const float v[8] = {xa.x, xa.z, xb.x, xb.z, xa.y, xa.w, xb.y, xb.w};
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const Split s0 = split_bf16(v[2 * i]), s1 = split_bf16(v[2 * i + 1]);
        hw[i] = s0.hi | (s1.hi << 16);
        lw[i] = s0.lo | (s1.lo << 16);
    }
    sts128(dst, make_uint4(hw[0], hw[1], hw[2], hw[3]));
    sts128(dst + 512, make_uint4(lw[0], lw[1], lw[2], lw[3]));
}

// Stage the CTA's K slice of X (pairs p0 .. p0+P-1): the region is zeroed
// (padded token lanes and padded K stay zero), then the real tokens are read
// from global memory, item = (q, blk, token, quad), with kStageUnroll items'
// loads in flight per thread.
template <int NT, int THREADS>
__device__ __forceinline__ void stage_x(const DecodeArgs &a, uint8_t *xs, int p0, int P)
{
    const int m = a.m;
    if (m < NT * 8) {
        const int vecs = P * xs_pair_bytes(NT) / 16;
        for (int i = threadIdx.x; i < vecs; i += THREADS) sts128(xs + i * 16, make_uint4(0u, 0u, 0u, 0u));
        __syncthreads();
    }
    const int real = P * 2 * m * 4;
    for (int base = threadIdx.x; base < real; base += THREADS * kStageUnroll) {
        float4 xa[kStageUnroll], xb[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int it = base + u * THREADS;
            xa[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            xb[u] = xa[u];
            if (it < real) {
                const int c = it & 3;
                const int tok = (it >> 2) % m;
                const int qb = (it >> 2) / m; // q * 2 + blk
                const int b = 2 * p0 + qb;
                if (b < a.nb) {
                    const int64_t row = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
                    const float *xr = a.X + row * a.ldx + 32 * b;
                    xa[u] = __ldg(reinterpret_cast<const float4 *>(xr + 4 * c));
                    xb[u] = __ldg(reinterpret_cast<const float4 *>(xr + 16 + 4 * c));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int it = base + u * THREADS;
            if (it < real) {
                const int c = it & 3;
                const int tok = (it >> 2) % m;
                const int qb = (it >> 2) / m;
                store_split(xs_slot(xs, NT, qb >> 1, tok, qb & 1, c), xa[u], xb[u]);
            }
        }
    }
}

__device__ __forceinline__ float half_lo(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFF)));
}
__device__ __forceinline__ float half_hi(uint32_t w)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

// One pair (2 blocks) of one 64-row group for this warp: 4 tiles of 16 rows.
template <int NT>
__device__ __forceinline__ void compute_pair(const uint8_t *st, const uint8_t *xq, int lane, float (&acc)[4][NT][4])
{
    const int g = lane >> 2;
    uint4 xh[2][NT], xl[2][NT];
#pragma unroll
    for (int blk = 0; blk < 2; ++blk)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            const uint8_t *p = xq + (nt * 2 + blk) * 1024 + lane * 16;
            xh[blk][nt] = lds128(p);
            xl[blk][nt] = lds128(p + 512);
        }
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        const uint8_t *rec = st + t * kRecordBytes;
        const uint4 nib = lds128(rec + 64 + lane * 16);
        const uint2 sc = lds64(rec + g * 8);
        const float ds[2][2] = {{half_lo(sc.x), half_hi(sc.x)}, {half_lo(sc.y), half_hi(sc.y)}};
#pragma unroll
        for (int blk = 0; blk < 2; ++blk) {
            uint32_t va[4], vb[4];
            unpack_word_bf16(blk ? nib.z : nib.x, va); // row g
            unpack_word_bf16(blk ? nib.w : nib.y, vb); // row g + 8
            const uint32_t A0[4] = {va[0], vb[0], va[1], vb[1]};
            const uint32_t A1[4] = {va[2], vb[2], va[3], vb[3]};
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                float c[4] = {0.f, 0.f, 0.f, 0.f};
                mma_bf16_16816(c, A0, xh[blk][nt].x, xh[blk][nt].y, c);
                mma_bf16_16816(c, A0, xl[blk][nt].x, xl[blk][nt].y, c);
                mma_bf16_16816(c, A1, xh[blk][nt].z, xh[blk][nt].w, c);
                mma_bf16_16816(c, A1, xl[blk][nt].z, xl[blk][nt].w, c);
                acc[t][nt][0] = fmaf(ds[blk][0], c[0], acc[t][nt][0]);
                acc[t][nt][1] = fmaf(ds[blk][0], c[1], acc[t][nt][1]);
                acc[t][nt][2] = fmaf(ds[blk][1], c[2], acc[t][nt][2]);
                acc[t][nt][3] = fmaf(ds[blk][1], c[3], acc[t][nt][3]);
            }
        }
    }
}

__device__ __forceinline__ void named_barrier_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ float ld_cg(const float *p)
{
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
    return v;
}

template <int NT>
__global__ void __launch_bounds__(warps_for(NT) * 32, 1) decode_kernel(const DecodeArgs a)
{
    constexpr int kWarps = warps_for(NT);
    constexpr int kThreads = kWarps * 32;
    extern __shared__ uint8_t smem_raw[];
    __shared__ int s_last;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int s = blockIdx.x % S;
    const int cps = gridDim.x / S;
    const int cidx = blockIdx.x / S;
    const int p0 = s * a.pbase + min(s, a.prem);
    const int P = a.pbase + (s < a.prem ? 1 : 0);
    const int wq0 = warp * (P / kWarps) + min(warp, P % kWarps);
    const int WQ = P / kWarps + (warp < P % kWarps ? 1 : 0);
    const int ng = cidx < a.groups ? (a.groups - cidx + cps - 1) / cps : 0;
    const int J = ng * WQ;
    const int STG = a.stages;

    uint8_t *xs = smem;
    uint8_t *ring = smem + a.xs_bytes;
    float *red = reinterpret_cast<float *>(ring + kWarps * STG * kPairBytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(red) + red_bytes(NT));
    uint64_t *mybar = bars + warp * STG;
    uint8_t *myring = ring + warp * STG * kPairBytes;

    if (lane == 0)
        for (int i = 0; i < STG; ++i) mbar_init(&mybar[i], 1);
    fence_barrier_init();
    __syncthreads();

    const uint64_t pol = policy_evict_first();
    int issued = 0;
    auto issue = [&](int j) {
        const int gi = j / WQ, q = j % WQ;
        const int64_t G = cidx + static_cast<int64_t>(gi) * cps;
        const int pp = p0 + wq0 + q;
        const uint8_t *src = a.W + (G * a.np + pp) * kPairBytes;
        const int slot = j % STG;
        mbar_arrive_expect_tx(&mybar[slot], kPairBytes);
        bulk_g2s_hint(myring + slot * kPairBytes, src, kPairBytes, &mybar[slot], pol);
    };
    // The weights may be streamed before the preceding kernel in the stream
    // has finished only when the caller declared them read-only; X, Y and the
    // workspace are touched after the wait.
    if (a.prefetch_w && lane == 0)
        for (; issued < min(STG, J); ++issued) issue(issued);
    pdl_wait();
    if (lane == 0)
        for (; issued < min(STG, J); ++issued) issue(issued);

    stage_x<NT, kThreads>(a, xs, p0, P);
    __syncthreads();

    const int m = a.m;
    const int n_pad = a.groups * 64;
    const int per = NT * 8 * 64;
    bool ok = true;
    int j = 0;
    for (int gi = 0; gi < ng; ++gi) {
        float acc[4][NT][4];
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int i = 0; i < 4; ++i) acc[t][nt][i] = 0.f;

        for (int q = 0; q < WQ; ++q, ++j) {
            const int slot = j % STG;
            if (ok && !mbar_wait(&mybar[slot], static_cast<uint32_t>((j / STG) & 1), a.wait_ns)) {
                ok = false;
                record_status(a.status, kErrTimeout);
            }
            compute_pair<NT>(myring + slot * kPairBytes, xs + (wq0 + q) * xs_pair_bytes(NT), lane, acc);
            __syncwarp();
            if (lane == 0 && ok && issued < J) issue(issued++);
        }

        // Fixed-order reduction of the 8 warps' partials of this group.
        {
            const int g = lane >> 2, c4 = lane & 3;
            float *mine = red + warp * per;
#pragma unroll
            for (int t = 0; t < 4; ++t)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int tok = nt * 8 + 2 * c4;
                    const int r0 = t * 16 + g;
                    mine[tok * 64 + r0] = acc[t][nt][0];
                    mine[(tok + 1) * 64 + r0] = acc[t][nt][1];
                    mine[tok * 64 + r0 + 8] = acc[t][nt][2];
                    mine[(tok + 1) * 64 + r0 + 8] = acc[t][nt][3];
                }
        }
        named_barrier_sync(1, kThreads);

        const int64_t G = cidx + static_cast<int64_t>(gi) * cps;
        for (int e = tid; e < m * 64; e += kThreads) {
            const int tok = e >> 6, row = e & 63;
            float v = red[e];
#pragma unroll
            for (int w = 1; w < kWarps; ++w) v += red[w * per + e];
            const int64_t grow = G * 64 + row;
            if (S == 1) {
                if (grow < a.n) {
                    const int64_t yrow = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
                    a.Y[yrow * a.ldy + grow] = v;
                }
            } else {
                a.partials[(static_cast<int64_t>(s) * m + tok) * n_pad + grow] = v;
            }
        }
        if (S > 1) {
            __threadfence();
            named_barrier_sync(1, kThreads);
            if (tid == 0) {
                const unsigned old = atomicAdd(&a.counters[G], 1u);
                s_last = old == static_cast<unsigned>(S - 1);
            }
            named_barrier_sync(1, kThreads);
            if (s_last) {
                __threadfence();
                for (int e = tid; e < m * 64; e += kThreads) {
                    const int tok = e >> 6, row = e & 63;
                    const int64_t grow = G * 64 + row;
                    if (grow < a.n) {
                        float v = 0.f;
                        for (int ss = 0; ss < S; ++ss)
                            v += ld_cg(a.partials + (static_cast<int64_t>(ss) * m + tok) * n_pad + grow);
                        const int64_t yrow = a.rows ? static_cast<int64_t>(a.rows[tok]) : tok;
                        a.Y[yrow * a.ldy + grow] = v;
                    }
                }
                // every slice of this group has arrived: leave its counter at
                // zero for the next call
                if (tid == 0) a.counters[G] = 0u;
            }
        }
        // the partials of this group must be read before the next is written
        named_barrier_sync(1, kThreads);
    }

    pdl_launch_dependents();

    // Drain: no bulk copy of ours may still be landing when the CTA exits.
    if (lane == 0) {
        for (int slot = 0; slot < STG; ++slot) {
            int last = -1;
            for (int jj = issued - 1; jj >= 0 && jj >= issued - STG; --jj)
                if (jj % STG == slot) {
                    last = jj;
                    break;
                }
            if (last >= 0 && !mbar_wait(&mybar[slot], static_cast<uint32_t>((last / STG) & 1), a.wait_ns))
                record_status(a.status, kErrTimeout);
        }
    }
}

} // namespace

size_t decode_smem_bytes(int NT, int P, int stages)
{
    const size_t xs = static_cast<size_t>(round_up(static_cast<int64_t>(P) * xs_pair_bytes(NT), 1024));
    const size_t warps = static_cast<size_t>(warps_for(NT));
    return 1024 /* alignment slack */ + xs + warps * stages * kPairBytes + red_bytes(NT) + warps * stages * 8;
}

// Choose the K split S and the grid. Cost model: the busiest SM's pair loads,
// plus a per-group overhead for the reduction (larger when slices must be
// combined through the workspace).
bool plan_decode(int64_t m, int64_t k, int64_t n, int sm_count, DecodePlan *plan)
{
    DecodePlan best;
    double best_cost = 1e300;
    const int NT = m <= 8 ? 1 : 2;
    const int64_t np = ceil_div(k, kPairK);
    const int64_t groups = ceil_div(n, kGroupRows);
    for (int64_t S = 1; S <= np && S <= 64; ++S) {
        if (S > 1 && groups > kDecodeCounterSlots) break;
        const int64_t P = ceil_div(np, S);
        if (S > 1 && ceil_div(np, S - 1) == P) continue; // same slice width, more slices
        const int64_t WQ = ceil_div(P, warps_for(NT));
        if (decode_smem_bytes(NT, static_cast<int>(P), 1) > kSmemOptIn) continue;
        // deepest ring that fits (at most every job of a warp, at most 8)
        int stages = 1;
        while (stages < 8 && decode_smem_bytes(NT, static_cast<int>(P), stages + 1) <= kSmemOptIn) ++stages;
        size_t smem = decode_smem_bytes(NT, static_cast<int>(P), stages);
        int64_t r = std::min<int64_t>(2048 / (warps_for(NT) * 32), static_cast<int64_t>(kSmemPerSM / (smem + 1024)));
        int64_t cps = std::min<int64_t>(groups, std::max<int64_t>(1, sm_count * r / S));
        int64_t ng = ceil_div(groups, cps);
        const int64_t jobs = ng * WQ;
        if (jobs < stages) {
            stages = static_cast<int>(std::max<int64_t>(1, jobs));
            smem = decode_smem_bytes(NT, static_cast<int>(P), stages);
            r = std::min<int64_t>(2048 / (warps_for(NT) * 32), static_cast<int64_t>(kSmemPerSM / (smem + 1024)));
            cps = std::min<int64_t>(groups, std::max<int64_t>(1, sm_count * r / S));
            ng = ceil_div(groups, cps);
        }
        const int64_t ctas = cps * S;
        const int64_t per_sm = ceil_div(ctas, sm_count);
        const double overhead = 1.0 + (S > 1 ? 2.0 : 0.0);
        // a ring shallower than three stages leaves the memory pipe idle
        const int64_t want = std::min<int64_t>(3, ng * WQ);
        const double shallow = 1.0 + 0.25 * static_cast<double>(std::max<int64_t>(0, want - stages));
        const double cost = static_cast<double>(per_sm) * ng * (static_cast<double>(P) + overhead) * shallow;
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best.NT = NT;
            best.S = static_cast<int>(S);
            best.pbase = static_cast<int>(np / S);
            best.prem = static_cast<int>(np % S);
            best.stages = stages;
            best.ctas = static_cast<int>(ctas);
            best.xs_bytes = static_cast<int>(round_up(P * xs_pair_bytes(NT), 1024));
            best.smem = smem;
        }
    }
    if (best.ctas == 0) return false;
    if (best.S > 1) {
        // counters first, at a fixed place, so they stay zero between calls of
        // any shape; partials after them
        best.ws_counters_off = 0;
        best.ws_partials_off = kWsCounterBytes;
        best.ws_bytes = best.ws_partials_off + static_cast<size_t>(best.S) * m * groups * 64 * sizeof(float);
    }
    *plan = best;
    return true;
}

cudaError_t launch_decode(const DecodePlan &plan, const DecodeArgs &args, cudaStream_t s)
{
    const void *fn = plan.NT == 1 ? reinterpret_cast<const void *>(&decode_kernel<1>)
                                  : reinterpret_cast<const void *>(&decode_kernel<2>);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    DecodeArgs a = args;
    void *kargs[] = {&a};
    return launch_pdl(fn, dim3(plan.ctas), dim3(warps_for(plan.NT) * 32), plan.smem, s, kargs);
}

} // namespace q4
