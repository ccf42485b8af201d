// q4mm_mmv.cu -- the decode kernel for m <= 16 token rows on the warp-level
// tensor-core MMA (mma.sync m16n8k16, fp16 x fp16 -> fp32): the decode step
// (m = 1) and continuous batching, where every active slot's token rides the
// same read of the weights (golem, "Several conversations, one pass"; golem-
// server, "Several conversations, in one pass"). The pages bound this case by
// the weight read (golem, "Qwen3.8 drafts its own next token": two columns
// cost what one did on the card), so the design goal is to consume a packed
// record at the rate one SM's share of HBM delivers it (one 4608-byte record
// every ~214 SM cycles on GB300) with as little issue as possible.
//
// Arithmetic. The CUDA cores only dequantise: one lop3 per two weights puts a
// pair of nibbles into the fp16 pattern of 1024 (1024 + q, or 1024 + 16 q for
// a high nibble) and one exact fp16 FMA turns the pair into (q - 8). Those
// integers are the A operand of the MMA as they are, never multiplied by d
// and never rounded. X is the B operand: each 32-element block of a token row
// is scaled by a power of two (its largest |x| lands in [2^14, 2^15)) and
// split into fp16 hi + lo, two columns of the MMA (22 significant bits
// relative to the block's largest |x|). The tensor core accumulates a block's
// 32 products in fp32; the block sum is then scaled in fp32 by d times the
// block's power of two and added to the row's fp32 total. A weight is never
// rounded, so the error is X's split plus fp32 accumulation.
//
// MMA shape. A 16 x 16 A tile holds 16 rows x 16 k of a record; thread (g,
// t) of a warp (lane = 4 g + t) holds rows g and g + 8. The K index of the
// MMA is a permutation of the block's elements chosen so that thread t's A
// registers come straight from its 4-byte word t of the row's 16 bytes of
// split-half nibbles (elements 4t .. 4t+3 low, 16 + 4t .. 19 + 4t high), in
// the packed layout as it is; the B fragments of X are staged in the same
// permutation. N = 8 columns are (hi, lo) of four tokens, so m <= 4 costs one
// MMA per 16 x 16 weight tile and every further four tokens one more.
//
// Work split (the decode kernels'): 128-row groups and S slices of K; the S
// CTAs of a thread-block cluster hold the S slices of the groups c, c + C,
// ... of their cluster c, and slices meet in the first CTA (DSMEM), summed in
// slice order, so results are bitwise reproducible and no global scratch is
// used.
//
// Warp roles in a CTA (two CTAs fit on an SM):
//   * warp 8, lane 0: streams the CTA's records (its groups x its pairs, in
//     that order) through a ring of R shared-memory slots with 1-D bulk
//     copies;
//   * warps 0-7: first stage the CTA's slice of X as B fragments in shared
//     memory (after the dependency wait), then warp w takes rows 16w .. 16w +
//     15 of every record: no partial sums cross warps, and each warp holds
//     its rows' totals in registers until the group ends.
// Every wait is bounded and warp-uniform; a slot's full barrier is waited on
// by the eight consumer warps, each of which releases the slot (empty
// barrier, eight arrivals) before the producer refills it, so no waiter can
// fall a phase behind.
#include <algorithm>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5;      // Q4_ERR_DEVICE_TIMEOUT
constexpr int kCWarps = 8;          // consumer warps
constexpr int kThreads = (kCWarps + 1) * 32;
constexpr int kMaxSlices = 8;
constexpr int kMaxRing = 32;
constexpr int kMaxTokens = 16;

struct MSmem {
    uint8_t *w;          // [R] records
    uint4 *ximg;         // [P][2][NT][32] B fragments of X
    float *xsc;          // [P][2][16] 2^-e of (pair, block, token)
    float *part;         // [2][16][128] this CTA's row totals of a group (S > 1)
    uint64_t *full, *empty;          // [R]
    uint64_t *red_full, *red_free;   // [2][8] a row tile's other slices landed / slot free
};

__device__ __forceinline__ void fail(const DecodeArgs &a) { record_status(a.status, kErrTimeout); }

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns)) != 0;
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar, parity, limit_ns)) != 0;
}

__device__ __forceinline__ uint32_t lds32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr)
{
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void consumers_sync()
{
    asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory");
}

// D = A * B + C, m16n8k16, fp16 operands, fp32 accumulate.
__device__ __forceinline__ void mma_f16(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1, const float c[4])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]),
                   "f"(c[2]), "f"(c[3]));
}

__device__ __forceinline__ unsigned absmax_bits(const float4 &v)
{
    return max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
               max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu));
}

// The hi (h = 0) or lo (h = 1) fp16 terms of two already scaled values, as
// one packed register (x0 in the low half): hi = fp16(x), lo = fp16(x - hi).
// A block whose largest |x| is not finite gets lo = 0 (its rows' results are
// infinite or NaN whatever lo holds).
__device__ __forceinline__ uint32_t split_pair(float x0, float x1, int h, bool finite)
{
    const __half2 hi = __floats2half2_rn(x0, x1);
    if (h == 0) return *reinterpret_cast<const uint32_t *>(&hi);
    const float2 back = __half22float2(hi);
    const __half2 lo = __floats2half2_rn(x0 - back.x, x1 - back.y);
    return finite ? *reinterpret_cast<const uint32_t *>(&lo) : 0u;
}

// Stage the CTA's slice of X (pairs p0 .. p0 + P - 1) as MMA B fragments.
// Entry (pair p, block b, column tile nt) holds, for lane (g, t), column g =
// (token 4 nt + g / 2, hi or lo by g % 2) at the K positions the A fragments
// use: k-step 0 elements (4t, 4t+2 | 16+4t, 18+4t), k-step 1 (4t+1, 4t+3 |
// 17+4t, 19+4t). Each (block, token) is scaled by its own power of two, whose
// inverse goes to xsc. Run by the consumer warps; warp c takes entries c, c +
// 8, ...
template <int NT>
__device__ __forceinline__ void stage_x(const DecodeArgs &a, const MSmem &sm, int p0, int P, int c, int lane,
                                        const int yrow[kMaxTokens])
{
    constexpr int kBatch = 8;                      // entries whose loads are in flight together
    const int g = lane >> 2, t = lane & 3;
    const int h = g & 1;
    const int E = P * 2 * NT;
    for (int e0 = c; e0 < E; e0 += kBatch * kCWarps) {
        float4 xa[kBatch], xb[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int e = e0 + q * kCWarps;
            const int nt = e % NT, pb = e / NT;
            const int blk = 2 * p0 + pb;           // pb = 2 p + b
            const int j = 4 * nt + (g >> 1);
            xa[q] = make_float4(0.f, 0.f, 0.f, 0.f);
            xb[q] = xa[q];
            if (e < E && blk < a.nb && j < a.m) {
                const float *xr = a.X + static_cast<int64_t>(yrow[j]) * a.ldx + 32 * blk + 4 * t;
                xa[q] = __ldg(reinterpret_cast<const float4 *>(xr));
                xb[q] = __ldg(reinterpret_cast<const float4 *>(xr + 16));
            }
        }
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const int e = e0 + q * kCWarps;
            if (e >= E) break;                     // warp-uniform
            const int nt = e % NT, pb = e / NT;
            const int j = 4 * nt + (g >> 1);
            // largest |x| of the block for token j: lanes 4g .. 4g+3 hold all 32
            unsigned mb = max(absmax_bits(xa[q]), absmax_bits(xb[q]));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            int ex = 0;
            if (mb != 0 && mb < 0x7F800000u) {
                const int E2 = static_cast<int>(mb >> 23) - 126;   // |x|max = f 2^E2, f in [0.5, 1) (normal)
                ex = (mb >> 23) == 0 ? 100 : 15 - E2;
                ex = max(-100, min(100, ex));
            }
            const float su = __uint_as_float(static_cast<unsigned>(ex + 127) << 23);
            const bool fin = mb < 0x7F800000u;
            uint4 f;
            f.x = split_pair(xa[q].x * su, xa[q].z * su, h, fin);
            f.y = split_pair(xb[q].x * su, xb[q].z * su, h, fin);
            f.z = split_pair(xa[q].y * su, xa[q].w * su, h, fin);
            f.w = split_pair(xb[q].y * su, xb[q].w * su, h, fin);
            sm.ximg[e * 32 + lane] = f;
            if (h == 0 && t == 0)
                sm.xsc[pb * kMaxTokens + j] = __uint_as_float(static_cast<unsigned>(127 - ex) << 23);
        }
    }
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 2) mmv_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int G0 = blockIdx.x / S;                  // first group of this cluster
    const int ntiles = G0 < a.groups ? (a.groups - 1 - G0) / a.clusters + 1 : 0;
    const int p0 = rank * a.pbase + min(rank, a.prem);
    const int P = a.pbase + (rank < a.prem ? 1 : 0);
    const int total = ntiles * P;                    // records this CTA streams
    const int R = a.ring;
    // Every CTA of the cluster lays out its shared memory for the largest
    // slice, so that a barrier or partial row sits at the same offset in all
    // of them (remote accesses map this CTA's offsets onto the first CTA's).
    const int Pmax = a.pbase + (a.prem > 0 ? 1 : 0);

    MSmem sm;
    sm.w = smem_raw;
    sm.ximg = reinterpret_cast<uint4 *>(sm.w + static_cast<size_t>(R) * kRecordBytes);
    sm.xsc = reinterpret_cast<float *>(sm.ximg + static_cast<size_t>(Pmax) * 2 * NT * 32);
    sm.part = sm.xsc + static_cast<size_t>(Pmax) * 2 * kMaxTokens;
    const int part_floats = S > 1 ? 2 * kMaxTokens * kGroupRows : 0;
    sm.full = reinterpret_cast<uint64_t *>(sm.part + part_floats);
    sm.empty = sm.full + R;
    sm.red_full = sm.empty + R;
    sm.red_free = sm.red_full + 2 * kCWarps;

    if (tid == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&sm.full[i], 1), mbar_init(&sm.empty[i], kCWarps);
        for (int i = 0; i < 2 * kCWarps; ++i) {
            mbar_init(&sm.red_full[i], S > 1 ? S - 1 : 1);
            mbar_init(&sm.red_free[i], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // The next kernel in the stream may be scheduled now: it waits for this
    // one to complete before it reads anything this one writes.
    pdl_launch_dependents();
    if (S > 1) cluster_sync(); // every CTA's barriers initialised before any remote arrive

    if (warp == kCWarps) {
        // ---------------------------------------------------------- producer
        // Weights may stream before the preceding kernel has finished only
        // when the caller declared them read-only.
        if (!a.prefetch_w) pdl_wait();
        if (lane == 0 && total > 0) {
            const uint64_t pol = policy_evict_first();
            int i = 0, j = 0, s = 0;
            uint32_t ph = 0;
            int issued = 0;
            for (int u = 0; u < total; ++u) {
                if (u >= R && !mbar_wait(&sm.empty[s], ph ^ 1u, a.wait_ns)) { fail(a); break; }
                const int64_t rec = static_cast<int64_t>(G0 + i * a.clusters) * a.np + p0 + j;
                mbar_arrive_expect_tx(&sm.full[s], kRecordBytes);
                bulk_g2s_hint(sm.w + static_cast<size_t>(s) * kRecordBytes, a.W + rec * kRecordBytes, kRecordBytes,
                              &sm.full[s], pol);
                issued = u + 1;
                if (++s == R) s = 0, ph ^= 1u;
                if (++j == P) j = 0, ++i;
            }
            // No copy may still be landing when the CTA exits: a record whose
            // slot a later record reused has landed already, so only the last
            // R issued records need a wait (their phase is final).
            for (int u = issued - 1; u >= 0 && u >= issued - R; --u)
                if (!mbar_wait(&sm.full[u % R], (u / R) & 1, a.wait_ns)) { fail(a); break; }
        }
        __syncwarp();
    } else {
        // --------------------------------------------------------- consumers
        // Warp w: rows 16w + g and 16w + g + 8 of every record (MMA rows g
        // and g + 8).
        const int w = warp;
        const int g = lane >> 2, t = lane & 3;
        const int R0 = 16 * w + g;
        pdl_wait();                                   // X, Y and the slot rows are the preceding kernel's
        int yrow[kMaxTokens];
#pragma unroll
        for (int j = 0; j < kMaxTokens; ++j) yrow[j] = j < a.m ? (a.rows ? __ldg(a.rows + j) : j) : 0;
        stage_x<NT>(a, sm, p0, P, warp, lane, yrow);
        consumers_sync();

        const uint32_t w0 = smem_u32(sm.w);
        const uint32_t off_sc = static_cast<uint32_t>(kRecScaleOff + 4 * R0);
        const uint32_t off_q0 = static_cast<uint32_t>(kRecQs0Off + 16 * R0 + 4 * t);
        const uint32_t off_q1 = static_cast<uint32_t>(kRecQs1Off + 16 * R0 + 4 * t);
        const uint32_t xi0 = smem_u32(sm.ximg) + static_cast<uint32_t>(lane * 16);
        const uint32_t xs0 = smem_u32(sm.xsc) + static_cast<uint32_t>(t * 4);
        const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
        bool ok = true;
        int s = 0;
        uint32_t ph = 0;
        for (int gi = 0; gi < ntiles && ok; ++gi) {
            float y[NT][2];
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) y[nt][0] = y[nt][1] = 0.f;
            for (int j = 0; j < P; ++j) {
                if (!warp_wait(&sm.full[s], ph, a.wait_ns)) { ok = false; break; }
                const uint32_t rec = w0 + static_cast<uint32_t>(s * kRecordBytes);
                const uint32_t sc0 = lds32(rec + off_sc), sc1 = lds32(rec + off_sc + 32);
                const uint32_t q00 = lds32(rec + off_q0), q01 = lds32(rec + off_q0 + 128);
                const uint32_t q10 = lds32(rec + off_q1), q11 = lds32(rec + off_q1 + 128);
                // A fragments [block][k-step]: (q - 8) of rows g, g + 8, exact
                uint32_t v00[4], v01[4], v10[4], v11[4];
                unpack_word_f16(q00, v00);
                unpack_word_f16(q01, v01);
                unpack_word_f16(q10, v10);
                unpack_word_f16(q11, v11);
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.empty[s]);   // the warp's share of the slot has been read
                const uint32_t A[2][2][4] = {{{v00[0], v01[0], v00[1], v01[1]}, {v00[2], v01[2], v00[3], v01[3]}},
                                             {{v10[0], v11[0], v10[1], v11[1]}, {v10[2], v11[2], v10[3], v11[3]}}};
                const float2 d0 = __half22float2(*reinterpret_cast<const __half2 *>(&sc0));   // row g: block 0, 1
                const float2 d1 = __half22float2(*reinterpret_cast<const __half2 *>(&sc1));   // row g + 8
                const uint32_t xi = xi0 + static_cast<uint32_t>(j * 2 * NT * 512);
                const uint32_t xs = xs0 + static_cast<uint32_t>(j * 2 * kMaxTokens * 4);
#pragma unroll
                for (int b = 0; b < 2; ++b) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        uint4 bf;
                        asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                                     : "=r"(bf.x), "=r"(bf.y), "=r"(bf.z), "=r"(bf.w)
                                     : "r"(xi + static_cast<uint32_t>((b * NT + nt) * 512)));
                        float su;
                        asm volatile("ld.shared.f32 %0, [%1];"
                                     : "=f"(su)
                                     : "r"(xs + static_cast<uint32_t>((b * kMaxTokens + 4 * nt) * 4)));
                        float D[4];
                        mma_f16(D, A[b][0], bf.x, bf.y, zero4);
                        mma_f16(D, A[b][1], bf.z, bf.w, D);
                        y[nt][0] = fmaf((b ? d0.y : d0.x) * su, D[0] + D[1], y[nt][0]);
                        y[nt][1] = fmaf((b ? d1.y : d1.x) * su, D[2] + D[3], y[nt][1]);
                    }
                }
                if (++s == R) s = 0, ph ^= 1u;
            }
            if (!ok) break;
            // ------------------------------------------------ group gi done
            const int tb = gi & 1;
            const uint32_t par = static_cast<uint32_t>((gi >> 1) & 1);
            if (rank > 0) {
                // rows into this CTA's part[tb]; the first CTA reads them
                if (gi >= 2 && !warp_wait_cluster(&sm.red_free[tb * kCWarps + w], par ^ 1u, a.wait_ns)) {
                    ok = false;
                    break;
                }
                float *pp = sm.part + tb * kMaxTokens * kGroupRows;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    pp[(4 * nt + t) * kGroupRows + R0] = y[nt][0];
                    pp[(4 * nt + t) * kGroupRows + R0 + 8] = y[nt][1];
                }
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_full[tb * kCWarps + w]), 0u));
                continue;
            }
            if (S > 1) {
                if (!warp_wait_cluster(&sm.red_full[tb * kCWarps + w], par, a.wait_ns)) { ok = false; break; }
                const uint32_t pbase = smem_u32(sm.part + tb * kMaxTokens * kGroupRows);
                for (int rr = 1; rr < S; ++rr) {
                    const uint32_t rp = mapa_shared(pbase, static_cast<uint32_t>(rr));
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint32_t o = static_cast<uint32_t>(((4 * nt + t) * kGroupRows + R0) * 4);
                        y[nt][0] += ld_cluster_f32(rp + o);
                        y[nt][1] += ld_cluster_f32(rp + o + 32);
                    }
                }
                __syncwarp();
                if (lane == 0)
                    for (int rr = 1; rr < S; ++rr)
                        mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_free[tb * kCWarps + w]), static_cast<uint32_t>(rr)));
            }
            const int64_t row0 = static_cast<int64_t>(G0 + gi * a.clusters) * kGroupRows + R0;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int tok = 4 * nt + t;
                if (tok < a.m) {
                    float *yr = a.Y + static_cast<int64_t>(yrow[tok]) * a.ldy + row0;
                    if (row0 < a.n) yr[0] = y[nt][0];
                    if (row0 + 8 < a.n) yr[8] = y[nt][1];
                }
            }
        }
        if (!ok) fail(a);
    }

    // every CTA of the cluster stays until the others are done with its
    // shared memory and barriers
    if (S > 1) cluster_sync();
}

size_t mmv_smem(int NT, int P, int S, int ring)
{
    const size_t ximg = static_cast<size_t>(P) * 2 * NT * 32 * 16;
    const size_t xsc = static_cast<size_t>(P) * 2 * kMaxTokens * 4;
    const size_t part = S > 1 ? static_cast<size_t>(2 * kMaxTokens * kGroupRows * 4) : 0;
    const size_t bars = static_cast<size_t>(2 * ring + 4 * kCWarps) * 8;
    return static_cast<size_t>(ring) * kRecordBytes + ximg + xsc + part + bars;
}

const void *mmv_fn(int NT)
{
    switch (NT) {
    case 1: return reinterpret_cast<const void *>(&mmv_kernel<1>);
    case 2: return reinterpret_cast<const void *>(&mmv_kernel<2>);
    case 3: return reinterpret_cast<const void *>(&mmv_kernel<3>);
    default: return reinterpret_cast<const void *>(&mmv_kernel<4>);
    }
}

// Largest number of clusters of S CTAs of the kernel with `smem` bytes of
// dynamic shared memory that the current device can hold at once (clusters
// live inside one GPC, so this is less than the SM count allows whenever S
// does not divide a GPC's SMs). Cached per (device, NT, S, smem).
int mmv_max_clusters(int NT, int S, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, NT, S, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void *fn = mmv_fn(NT);
    int n = 0;
    if (set_max_smem(fn, smem) == cudaSuccess) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(S));
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cudaLaunchAttribute attr{};
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = static_cast<unsigned>(S);
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

// Choose the cluster size S (K slices per 128-row group), the number of
// persistent clusters and the ring depth. Candidates per S: the deepest ring
// that fits one CTA's shared memory, and the deepest that leaves room for a
// second CTA on the SM (the next call's, or this call's). The number of
// clusters is capped by what the device holds at once (a second wave would
// double the time). Cost, in record times of one SM's share of HBM (about
// 0.1 us on GB300): the busiest SM's records at the rate its CTAs sustain,
// plus the cross-CTA reduction of split K (measured about 1.3 us a call),
// per-group overheads, and the start-up that cannot overlap the preceding
// call when no SM has room left for the next call's CTA.
bool plan_mmv(int64_t m, int64_t k, int64_t n, int sm_count, MmvPlan *plan)
{
    if (m < 1 || m > kMaxTokens || sm_count < 1) return false;
    const int NT = static_cast<int>((m + 3) / 4);
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const double total = static_cast<double>(groups * np);
    const size_t half = kSmemPerSM / 2 - 1024;
    MmvPlan best;
    double best_cost = 1e300;
    for (int S = 1; S <= kMaxSlices && S <= np; ++S) {
        const int64_t P = ceil_div(np, S);
        for (int two = 0; two <= 1; ++two) {
            const size_t limit = two ? half : kSmemOptIn;
            int ring = 0;
            for (int r = kMaxRing; r >= 4 && ring == 0; r -= 2)
                if (mmv_smem(NT, static_cast<int>(P), S, r) <= limit) ring = r;
            if (ring == 0) continue;
            const size_t smem = mmv_smem(NT, static_cast<int>(P), S, ring);
            const bool two_fit = smem <= half;
            if (!two && two_fit) continue;             // the same plan as two = 1
            const int64_t cmax = mmv_max_clusters(NT, S, smem);
            if (cmax < 1) continue;
            const int64_t clusters = std::min<int64_t>(groups, cmax);
            const int64_t tiles = ceil_div(groups, clusters);
            const int64_t ctas = clusters * S;
            const int per_sm = ctas > sm_count ? 2 : 1;
            // records an SM turns over per record time: one CTA of this kernel
            // alone on an SM takes about 2.5 record times per record (issue-
            // bound); two CTAs of the call share an SM at about 0.6 records
            // per record time (measured on GB300)
            const double rate = per_sm == 2 ? 0.6 : 0.4;
            const double recs = static_cast<double>(tiles * P);   // records per CTA
            const double stream = std::max(recs * per_sm / rate, total / sm_count);
            const double no_overlap = (!two_fit || per_sm == 2) ? 15.0 : 0.0;
            // A CTA with several groups reduces each through the cluster
            // handshake at the end of the next one. Measured: about 3 us more
            // than a grid of single-group CTAs (9728 x 2560 at m = 16: 23.8 us
            // with two groups per CTA, 15.9 us with one), and per group about
            // 5 + 6 S record times (151936 x 2560 at m = 16: 132 us at S = 1,
            // 297 us at S = 8 with 33 groups per CTA).
            const double groups_cost =
                tiles > 1 ? 30.0 + static_cast<double>(tiles) * (5.0 + 6.0 * S) : 0.5;
            // a ring of 4 records does not cover the weight stream's latency
            // (14336 x 4096 at m = 9: one group per CTA with a ring of 4,
            // 32.5 us; two groups with a ring of 12, 27.7 us); a ring of 6
            // measured fine (9728 x 2560 at m = 9: 13.2 us)
            const double starve = ring <= 4 ? recs * (8 - ring) * 0.4 / per_sm : 0.0;
            const double cost = stream + (S > 1 ? 12.0 : 0.0) + no_overlap + groups_cost + starve;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.NT = NT;
                best.S = S;
                best.clusters = static_cast<int>(clusters);
                best.ctas = static_cast<int>(ctas);
                best.ring = ring;
                best.smem = smem;
            }
        }
    }
    if (best.ctas == 0) return false;
    *plan = best;
    return true;
}

cudaError_t launch_mmv(const MmvPlan &plan, const DecodeArgs &args, cudaStream_t s)
{
    const void *fn = mmv_fn(plan.NT);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    DecodeArgs a = args;
    a.pass_p0 = 0;
    a.S = plan.S;
    a.pbase = args.np / plan.S;
    a.prem = args.np % plan.S;
    a.clusters = plan.clusters;
    a.ring = plan.ring;
    a.accumulate = 0;
    a.xs_bytes = 0;
    void *kargs[] = {&a};
    return launch_pdl(fn, dim3(plan.ctas), dim3(kThreads), plan.smem, s, kargs, plan.S);
}

} // namespace q4
