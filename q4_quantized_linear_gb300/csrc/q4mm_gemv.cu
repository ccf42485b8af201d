// q4mm_gemv.cu -- the decode kernel in which each warp takes whole packed
// records, for the decode step (m = 1) and small continuous batches (golem,
// "Several conversations, one pass"; golem-server, "Several conversations, in
// one pass"). The pages bound this case by the weight read (golem: two
// columns cost what one did; goinfer ch. 10, "What the kernels are": the
// quantised mat-vec is the decode workhorse), so the design goal is to
// consume a packed record at the rate one SM's share of HBM delivers it with
// as few instructions as possible. Three modes share the warps, ring and
// reductions: fp32 FMAs on the CUDA cores (m <= 4, below), the record-MMA
// mode on the warp-level tensor core (m <= 16, further down) and its W4A8
// form (X coded to int8 per block, integer block dots; q4_0_matmul_w4a8).
//
// CUDA-core arithmetic. A weight is (q - 8) * d. One lop3 per weight ORs the nibble,
// left where it lies in its 32-bit word (bit offset s <= 16), into the fp32
// pattern of 2^23, giving exactly 2^23 + q * 2^s. One fp32 FMA per weight,
// v * 2^-s - (2^(23-s) + 8), gives (q - 8) exactly. A second FMA per weight
// and token multiplies by x, read as fp32 and never rounded, and accumulates
// in fp32 over the block's 32 elements; the block sum is then scaled by d
// (fp16, exact in fp32) into the row's fp32 partial. The FMAs are scalar: on
// GB300 the packed two-lane form holds one of the sub-partition's two FMA
// pipes for twice as long, and the scalar form runs faster (measured: 152k x
// 2560 rows, m = 1: 55.7 -> 51.3 us).
//
// Work split (the decode kernel's): 128-row groups and S slices of K; the S
// CTAs of a thread-block cluster hold the S slices of the groups c, c + C, ...
// of their cluster c, and slices meet in the first CTA's shared memory
// (DSMEM), summed in slice order, so results are bitwise reproducible and no
// global scratch is used.
//
// Warp roles: eight warps per CTA, all alike (two CTAs fit on an SM up to
// m = 8). Warp c owns the records u = c (mod 8) of the CTA's sequence (its
// groups x its pairs, in that order) and the ring slots they pass through,
// R / 8 of them: lane 0 refills a slot with a 1-D bulk copy of the record R
// places ahead as soon as the warp has read it, so every barrier has one
// waiter and no copy is in flight when the CTA exits. In the CUDA-core mode
// lane l owns rows l, l + 32, l + 64 and l + 96 of a record: every
// shared-memory load is 512 contiguous bytes per warp (conflict-free) and
// every X value a thread loads (a broadcast, L1-resident) serves four rows.
// At the end of a group each warp leaves its partial rows in shared memory;
// one group later (so that no warp waits for the slowest), warp c sums the
// eight partials of rows 16c .. 16c + 15 in order, and then the cluster's
// slices of those rows, and writes Y. When every CTA has a single group, the
// slices meet through the kernel's closing cluster barrier instead. Every
// wait is bounded and warp-uniform.
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
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSliceRows = kGroupRows / kWarps;   // rows of a group each warp reduces
constexpr int kMaxSlices = 8;
constexpr int kMaxRing = 32;

struct GSmem {
    uint8_t *w;          // [R] records
    float *part;         // [2][kWarps][M][128] warps' partial rows of a group
    float *red;          // [2][S - 1][M][128] other slices' rows (first CTA of the cluster)
    uint64_t *full_w;    // [R]
    uint64_t *gfull, *gfree;        // [2] partials of a group parity written / summed
    uint64_t *red_full, *red_free;  // [2][kWarps] a row slice's other slices landed / slot free
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

// (w & mask) | bits of 2^23: the nibble under `mask` (at bit s <= 16) read as
// the fp32 value 2^23 + q * 2^s, exactly.
__device__ __forceinline__ float nib_f32(uint32_t w, uint32_t mask)
{
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(0x4B000000u));
    return __uint_as_float(r);
}

// The eight weights of one word of split-half nibbles (bytes 4c..4c+3 of a
// block's qs, element base e = 4c; byte i holds element i low, i + 16 high)
// as exact fp32 (q - 8), paired like the X values they multiply:
//   f[0] = (e, e+1)  f[1] = (e+2, e+3)  f[2] = (e+16, e+17)  f[3] = (e+18, e+19).
// Bit offsets in w: e 0, e+16 4, e+1 8, e+17 12, e+2 16, e+18 20, e+3 24,
// e+19 28; the last three are read from w >> 12 at 8, 12, 16.
// Two scalar fp32 FMAs, lane by lane.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    return make_float2(fmaf(a.x, b.x, c.x), fmaf(a.y, b.y, c.y));
}

// Multipliers and addends of the conversion, one pair per f[] entry, held in
// registers for the whole kernel.
struct Conv {
    float2 m[4], c[4];
};

// A float pair the compiler must keep in registers as it is (no constant
// folding or rematerialisation).
__device__ __forceinline__ float2 reg_pair(float a, float b)
{
    float x, y;
    asm volatile("mov.b32 %0, %2;\n\tmov.b32 %1, %3;" : "=f"(x), "=f"(y) : "f"(a), "f"(b));
    return make_float2(x, y);
}

__device__ __forceinline__ Conv make_conv()
{
    Conv k;
    k.m[0] = reg_pair(1.0f, 0x1p-8f);
    k.c[0] = reg_pair(-(0x1p23f + 8.0f), -(0x1p15f + 8.0f));
    k.m[1] = reg_pair(0x1p-16f, 0x1p-12f);
    k.c[1] = reg_pair(-(0x1p7f + 8.0f), -(0x1p11f + 8.0f));
    k.m[2] = reg_pair(0x1p-4f, 0x1p-12f);
    k.c[2] = reg_pair(-(0x1p19f + 8.0f), -(0x1p11f + 8.0f));
    k.m[3] = reg_pair(0x1p-8f, 0x1p-16f);
    k.c[3] = reg_pair(-(0x1p15f + 8.0f), -(0x1p7f + 8.0f));
    return k;
}

__device__ __forceinline__ void unpack_word_f32(uint32_t w, const Conv &k, float2 f[4])
{
    const uint32_t w2 = w >> 12;
    const float2 a = make_float2(nib_f32(w, 0x0000Fu), nib_f32(w, 0x00F00u));    // e   (s 0),  e+1  (s 8)
    const float2 b = make_float2(nib_f32(w, 0xF0000u), nib_f32(w2, 0x0F000u));   // e+2 (s 16), e+3  (s 12)
    const float2 c = make_float2(nib_f32(w, 0x000F0u), nib_f32(w, 0x0F000u));    // e+16 (s 4), e+17 (s 12)
    const float2 d = make_float2(nib_f32(w2, 0x00F00u), nib_f32(w2, 0xF0000u));  // e+18 (s 8), e+19 (s 16)
    f[0] = fma2(a, k.m[0], k.c[0]);
    f[1] = fma2(b, k.m[1], k.c[1]);
    f[2] = fma2(c, k.m[2], k.c[2]);
    f[3] = fma2(d, k.m[3], k.c[3]);
}

__device__ __forceinline__ uint32_t lds32(const void *p)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(smem_u32(p)));
    return v;
}

// One block (32 elements) of the record for the thread's four rows: adds
// d * sum_i (q_i - 8) x[t][kb + i] into yp[r][t]. A row's 16 bytes of
// nibbles are one 16-byte load (lanes 16 bytes apart: conflict-free). M == 1
// keeps two accumulator pairs per row for a shorter dependency chain.
template <int M>
__device__ __forceinline__ void gemv_block(const uint8_t *qs, uint32_t dsh, const uint32_t sc[4],
                                           const float *const xr[M], int kb, int lane, const Conv &kc,
                                           float yp[4][M])
{
    constexpr int A = M == 1 ? 2 : 1;
    float2 acc[4][M][A];
#pragma unroll
    for (int r = 0; r < 4; ++r)
#pragma unroll
        for (int t = 0; t < M; ++t)
#pragma unroll
            for (int z = 0; z < A; ++z) acc[r][t][z] = make_float2(0.0f, 0.0f);
    uint4 q[4];
#pragma unroll
    for (int r = 0; r < 4; ++r) q[r] = lds128(qs + 16 * (lane + 32 * r));
#pragma unroll
    for (int wd = 0; wd < 4; ++wd) {
        uint32_t qw[4];
#pragma unroll
        for (int r = 0; r < 4; ++r) qw[r] = wd == 0 ? q[r].x : wd == 1 ? q[r].y : wd == 2 ? q[r].z : q[r].w;
        float4 xl[M], xh[M];
#pragma unroll
        for (int t = 0; t < M; ++t) {
            xl[t] = __ldg(reinterpret_cast<const float4 *>(xr[t] + kb + 4 * wd));
            xh[t] = __ldg(reinterpret_cast<const float4 *>(xr[t] + kb + 16 + 4 * wd));
        }
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            float2 f[4];
            unpack_word_f32(qw[r], kc, f);
#pragma unroll
            for (int t = 0; t < M; ++t) {
                acc[r][t][0] = fma2(f[0], make_float2(xl[t].x, xl[t].y), acc[r][t][0]);
                acc[r][t][A - 1] = fma2(f[1], make_float2(xl[t].z, xl[t].w), acc[r][t][A - 1]);
                acc[r][t][0] = fma2(f[2], make_float2(xh[t].x, xh[t].y), acc[r][t][0]);
                acc[r][t][A - 1] = fma2(f[3], make_float2(xh[t].z, xh[t].w), acc[r][t][A - 1]);
            }
        }
    }
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const float d = __half2float(__ushort_as_half(static_cast<unsigned short>((sc[r] >> dsh) & 0xFFFFu)));
#pragma unroll
        for (int t = 0; t < M; ++t) {
            float s = acc[r][t][0].x + acc[r][t][0].y;
            if (A == 2) s += acc[r][t][A - 1].x + acc[r][t][A - 1].y;
            yp[r][t] = fmaf(d, s, yp[r][t]);
        }
    }
}

// ------------------------------------------------------------------------
// Record-MMA mode (m <= 16): the same warps, ring and reductions, but a warp
// turns its record's nibbles into exact fp16 (q - 8) (lop3 magic and one fp16
// FMA per two weights) and multiplies them by X on the tensor core with
// mma.sync m16n8k16, 16 rows at a time, in (m + 3) / 4 column tiles of four
// tokens. The MMA's K index is a permutation of
// a block's elements chosen so that thread (g, t) of the warp (lane 4g + t)
// takes its A registers straight from word t of its rows' 16 nibble bytes;
// X's B fragments use the same permutation. Column g of the 8 is token g / 2,
// its hi (g even) or lo (g odd) fp16 term after the block is scaled by a power
// of two (largest |x| into [2^14, 2^15)): 22 significant bits relative to the
// block's largest |x|. d is applied in fp32 per block.

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

// The hi (h = 0) or lo (h = 1) fp16 terms of two scaled values, packed (x0 in
// the low half). A block whose largest |x| is not finite gets lo = 0 (its
// rows' results are infinite or NaN whatever lo holds).
__device__ __forceinline__ uint32_t split_pair(float x0, float x1, int h, bool finite)
{
    const __half2 hi = __floats2half2_rn(x0, x1);
    if (h == 0) return *reinterpret_cast<const uint32_t *>(&hi);
    const float2 back = __half22float2(hi);
    const __half2 lo = __floats2half2_rn(x0 - back.x, x1 - back.y);
    return finite ? *reinterpret_cast<const uint32_t *>(&lo) : 0u;
}

// This lane's 8 X values of block blk for its column's token (token g / 2):
// elements 4t .. 4t + 3 and 16 + 4t .. 19 + 4t; lanes 4g .. 4g + 3 together
// hold the block. Zero when the column or the block is not live.
__device__ __forceinline__ void x_load(const float *xrow, int blk, bool live, int lane, float4 &xa, float4 &xb)
{
    const int t = lane & 3;
    xa = make_float4(0.f, 0.f, 0.f, 0.f);
    xb = xa;
    if (live) {
        const float *xr = xrow + 32 * blk + 4 * t;
        xa = __ldg(reinterpret_cast<const float4 *>(xr));
        xb = __ldg(reinterpret_cast<const float4 *>(xr + 16));
    }
}

// B fragments of one block from this lane's X values (column g: token g / 2,
// term g % 2), and the inverse of the scale this lane's column took. Lanes
// 4g .. 4g + 3 (of `lane`, which may be a lane index within a half warp)
// agree on the scale.
__device__ __forceinline__ void x_fragments(const float4 &xa, const float4 &xb, int lane, uint4 &bf, float &inv)
{
    const int h = (lane >> 2) & 1;
    unsigned mb = max(absmax_bits(xa), absmax_bits(xb));
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
    bf.x = split_pair(xa.x * su, xa.z * su, h, fin);   // k-step 0: elements 4t, 4t+2
    bf.y = split_pair(xb.x * su, xb.z * su, h, fin);   //           16+4t, 18+4t
    bf.z = split_pair(xa.y * su, xa.w * su, h, fin);   // k-step 1: 4t+1, 4t+3
    bf.w = split_pair(xb.y * su, xb.w * su, h, fin);   //           17+4t, 19+4t
    inv = __uint_as_float(static_cast<unsigned>(127 - ex) << 23);
}

// One record through the tensor core: y[nt][rt][0 / 1] += rows 16 rt + g
// and 16 rt + g + 8, token 4 nt + t (lane 4g + t). The weights of a row tile
// are turned into fp16 once for all NT column tiles.
template <int NT>
__device__ __forceinline__ void mma_record(const uint8_t *rec, const uint4 bf[NT][2], const float su[NT][2],
                                           int lane, float y[NT][8][2])
{
    const int g = lane >> 2, t = lane & 3;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t base = smem_u32(rec);
#pragma unroll
    for (int rt = 0; rt < 8; ++rt) {
        const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
        uint32_t sc0, sc1, q00, q01, q10, q11;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc0) : "r"(base + kRecScaleOff + 4 * r0));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc1) : "r"(base + kRecScaleOff + 4 * r0 + 32));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q00) : "r"(base + kRecQs0Off + 16 * r0 + 4 * t));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q01) : "r"(base + kRecQs0Off + 16 * r0 + 4 * t + 128));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q10) : "r"(base + kRecQs1Off + 16 * r0 + 4 * t));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q11) : "r"(base + kRecQs1Off + 16 * r0 + 4 * t + 128));
        uint32_t v00[4], v01[4], v10[4], v11[4];
        unpack_word_f16(q00, v00);
        unpack_word_f16(q01, v01);
        unpack_word_f16(q10, v10);
        unpack_word_f16(q11, v11);
        const uint32_t A[2][2][4] = {{{v00[0], v01[0], v00[1], v01[1]}, {v00[2], v01[2], v00[3], v01[3]}},
                                     {{v10[0], v11[0], v10[1], v11[1]}, {v10[2], v11[2], v10[3], v11[3]}}};
        const float2 d0 = __half22float2(*reinterpret_cast<const __half2 *>(&sc0));   // row g: block 0, 1
        const float2 d1 = __half22float2(*reinterpret_cast<const __half2 *>(&sc1));   // row g + 8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float D[4];
                mma_f16(D, A[b][0], bf[nt][b].x, bf[nt][b].y, zero4);
                mma_f16(D, A[b][1], bf[nt][b].z, bf[nt][b].w, D);
                y[nt][rt][0] = fmaf((b ? d0.y : d0.x) * su[nt][b], D[0] + D[1], y[nt][rt][0]);
                y[nt][rt][1] = fmaf((b ? d1.y : d1.x) * su[nt][b], D[2] + D[3], y[nt][rt][1]);
            }
    }
}

// ------------------------------------------------------------------------
// W4A8 mode (the integer-dot variant, q4_0_matmul_w4a8): X is coded per
// 32-element block to int8, c = round-half-even(x * (127 / amax)), scale
// s = amax / 127, both in fp32 exactly as written (IEEE quotient and
// product); a block with amax = 0 has codes 0 and scale 0, and a block holding
// a NaN or an infinity gets a NaN scale, which makes every output of its row
// NaN. The codes and (q - 8) are exact in fp16 and a block's integer dot
// product (at most 32 * 8 * 127 in size) is exact in the MMA's fp32
// accumulator, so each block's dot is the integer one; d * s is applied to it
// in fp32. Column g of the eight MMA columns is token g of the column tile.

// This lane's B fragment of one block (the codes of its column's token,
// elements 4t .. 4t + 3 and 16 + 4t .. 19 + 4t, in the K permutation of the
// hi/lo mode) and the block's scale s for that token. Lanes 4g .. 4g + 3
// agree on amax.
__device__ __forceinline__ void x_codes(const float4 &xa, const float4 &xb, uint4 &bf, float &scale)
{
    unsigned mb = max(absmax_bits(xa), absmax_bits(xb));
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
    mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
    const float amax = __uint_as_float(mb);
    const bool finite = mb < 0x7F800000u;
    const float inv = (finite && mb != 0u) ? __fdiv_rn(127.0f, amax) : 0.0f;
    scale = finite ? __fdiv_rn(amax, 127.0f) : __uint_as_float(0x7FC00000u);
    auto code2 = [inv](float lo, float hi) {
        const __half2 h = __halves2half2(__int2half_rn(__float2int_rn(__fmul_rn(lo, inv))),
                                         __int2half_rn(__float2int_rn(__fmul_rn(hi, inv))));
        return *reinterpret_cast<const uint32_t *>(&h);
    };
    bf.x = code2(xa.x, xa.z);   // k-step 0: elements 4t, 4t+2
    bf.y = code2(xb.x, xb.z);   //           16+4t, 18+4t
    bf.z = code2(xa.y, xa.w);   // k-step 1: 4t+1, 4t+3
    bf.w = code2(xb.y, xb.w);   //           17+4t, 19+4t
}

// One record through the tensor core in W4A8 mode: y[nt][rt][0..3] += rows
// 16 rt + g (0, 1) and 16 rt + g + 8 (2, 3), tokens 8 nt + 2t (0, 2) and
// 8 nt + 2t + 1 (1, 3). sc[nt][b][0 / 1]: the block's scales of those two
// tokens.
template <int NT>
__device__ __forceinline__ void mma_record_a8(const uint8_t *rec, const uint4 bf[NT][2], const float sc[NT][2][2],
                                              int lane, float y[NT][8][4])
{
    const int g = lane >> 2, t = lane & 3;
    const float zero4[4] = {0.f, 0.f, 0.f, 0.f};
    const uint32_t base = smem_u32(rec);
#pragma unroll
    for (int rt = 0; rt < 8; ++rt) {
        const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
        uint32_t sc0, sc1, q00, q01, q10, q11;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc0) : "r"(base + kRecScaleOff + 4 * r0));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(sc1) : "r"(base + kRecScaleOff + 4 * r0 + 32));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q00) : "r"(base + kRecQs0Off + 16 * r0 + 4 * t));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q01) : "r"(base + kRecQs0Off + 16 * r0 + 4 * t + 128));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q10) : "r"(base + kRecQs1Off + 16 * r0 + 4 * t));
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(q11) : "r"(base + kRecQs1Off + 16 * r0 + 4 * t + 128));
        uint32_t v00[4], v01[4], v10[4], v11[4];
        unpack_word_f16(q00, v00);
        unpack_word_f16(q01, v01);
        unpack_word_f16(q10, v10);
        unpack_word_f16(q11, v11);
        const uint32_t A[2][2][4] = {{{v00[0], v01[0], v00[1], v01[1]}, {v00[2], v01[2], v00[3], v01[3]}},
                                     {{v10[0], v11[0], v10[1], v11[1]}, {v10[2], v11[2], v10[3], v11[3]}}};
        const float2 d0 = __half22float2(*reinterpret_cast<const __half2 *>(&sc0));   // row g: block 0, 1
        const float2 d1 = __half22float2(*reinterpret_cast<const __half2 *>(&sc1));   // row g + 8
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                float D[4];
                mma_f16(D, A[b][0], bf[nt][b].x, bf[nt][b].y, zero4);
                mma_f16(D, A[b][1], bf[nt][b].z, bf[nt][b].w, D);
                const float dg = b ? d0.y : d0.x, dg8 = b ? d1.y : d1.x;
                y[nt][rt][0] = fmaf(__fmul_rn(dg, sc[nt][b][0]), D[0], y[nt][rt][0]);
                y[nt][rt][1] = fmaf(__fmul_rn(dg, sc[nt][b][1]), D[1], y[nt][rt][1]);
                y[nt][rt][2] = fmaf(__fmul_rn(dg8, sc[nt][b][0]), D[2], y[nt][rt][2]);
                y[nt][rt][3] = fmaf(__fmul_rn(dg8, sc[nt][b][1]), D[3], y[nt][rt][3]);
            }
    }
}

// Issue the bulk copy of the CTA's record (group i of its cluster, pair j of
// its slice) into ring slot s. Lane 0 of the slot's warp only.
__device__ __forceinline__ void load_record(const DecodeArgs &a, const GSmem &sm, int i, int j, int s, int G0,
                                            int p0, uint64_t pol)
{
    const int64_t rec = static_cast<int64_t>(G0 + i * a.clusters) * a.np + p0 + j;
    mbar_arrive_expect_tx(&sm.full_w[s], kRecordBytes);
    bulk_g2s_hint(sm.w + static_cast<size_t>(s) * kRecordBytes, a.W + rec * kRecordBytes, kRecordBytes,
                  &sm.full_w[s], pol);
}

// Advance a (group, pair) position of the CTA's record sequence by one step
// of a warp (kWarps records).
__device__ __forceinline__ void step_pos(int &i, int &j, int P)
{
    j += kWarps;
    while (j >= P) j -= P, ++i;
}

// First CTA of the cluster: add the other slices of group g's rows (landed
// in its shared memory) to this warp's sums y and write them to Y.
template <int M>
__device__ __forceinline__ void write_rows(const DecodeArgs &a, const GSmem &sm, int g, int c, int lane, int G0,
                                           const int yrow[M], const float y[(M + 1) / 2])
{
    const int S = a.S;
    const int tb = g & 1;
    const int row = c * kSliceRows + (lane & (kSliceRows - 1));
    const int t0 = lane >> 4;
    const int64_t grow = static_cast<int64_t>(G0 + g * a.clusters) * kGroupRows + row;
    if (grow >= a.n) return;
#pragma unroll
    for (int h = 0; h < (M + 1) / 2; ++h) {
        const int t = t0 + 2 * h;
        if (t < M && t < a.m) {
            float v = y[h];
            for (int r = 1; r < S; ++r) v += sm.red[((tb * (S - 1) + r - 1) * M + t) * kGroupRows + row];
            a.Y[static_cast<int64_t>(yrow[t]) * a.ldy + grow] = v;
        }
    }
}

// Sum the eight warps' partials of group g for this warp's rows (into y),
// then meet the cluster's other slices of them and write Y (first CTA) or
// send them there. Lane l handles row 16 c + (l & 15) and tokens t = l / 16,
// + 2, ... With `merged` (the group is the CTA's only one) the slices meet
// through the cluster barrier that ends the kernel instead: no barrier
// handshake, and the first CTA writes Y after that barrier.
template <int M>
__device__ __forceinline__ bool reduce_group(const DecodeArgs &a, const GSmem &sm, int g, int c, int lane, int rank,
                                             int G0, const int yrow[M], bool merged, float y[(M + 1) / 2])
{
    const int S = a.S;
    const int tb = g & 1;
    const uint32_t par = static_cast<uint32_t>((g >> 1) & 1);
    if (!warp_wait(&sm.gfull[tb], par, a.wait_ns)) return false;
    const int row = c * kSliceRows + (lane & (kSliceRows - 1));
    const int t0 = lane >> 4;
#pragma unroll
    for (int h = 0; h < (M + 1) / 2; ++h) {
        const int t = t0 + 2 * h;
        float v = 0.0f;
        if (t < M)
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v += sm.part[((tb * kWarps + w) * M + t) * kGroupRows + row];
        y[h] = v;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.gfree[tb]);
    if (rank > 0) {
        // this slice's rows into the first CTA's slot tb, then signal it
        if (g >= 2 && !warp_wait_cluster(&sm.red_free[tb * kWarps + c], par ^ 1u, a.wait_ns)) return false;
        const uint32_t dst = mapa_shared(smem_u32(sm.red), 0u) +
                             static_cast<uint32_t>(((((tb * (S - 1) + rank - 1) * M) * kGroupRows) + row) * 4);
#pragma unroll
        for (int h = 0; h < (M + 1) / 2; ++h) {
            const int t = t0 + 2 * h;
            if (t < M) st_cluster_f32(dst + static_cast<uint32_t>(t * kGroupRows * 4), y[h]);
        }
        if (!merged) {
            __syncwarp();
            if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_full[tb * kWarps + c]), 0u));
        }
    } else if (!merged) {
        if (S > 1 && !warp_wait_cluster(&sm.red_full[tb * kWarps + c], par, a.wait_ns)) return false;
        write_rows<M>(a, sm, g, c, lane, G0, yrow, y);
        if (S > 1) {
            __syncwarp();
            if (lane == 0)
                for (int r = 1; r < S; ++r)
                    mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_free[tb * kWarps + c]), static_cast<uint32_t>(r)));
        }
    }
    return true;
}

template <int M, bool MMA, bool A8>
__global__ void __launch_bounds__(kThreads, M > 8 ? 1 : 2) gemv_kernel(const DecodeArgs a)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int tid = threadIdx.x, c = tid >> 5, lane = tid & 31;
    const int S = a.S;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    const int G0 = blockIdx.x / S;                  // first group of this cluster
    const int ntiles = G0 < a.groups ? (a.groups - 1 - G0) / a.clusters + 1 : 0;
    const int p0 = rank * a.pbase + min(rank, a.prem);
    const int P = a.pbase + (rank < a.prem ? 1 : 0);
    const int total = ntiles * P;                    // records this CTA streams
    const int R = a.ring;

    GSmem sm;
    sm.w = smem_raw;
    sm.part = reinterpret_cast<float *>(sm.w + static_cast<size_t>(R) * kRecordBytes);
    sm.red = sm.part + 2 * kWarps * M * kGroupRows;
    const int red_floats = S > 1 ? 2 * (S - 1) * M * kGroupRows : 0;
    sm.full_w = reinterpret_cast<uint64_t *>(sm.red + red_floats);
    sm.gfull = sm.full_w + R;
    sm.gfree = sm.gfull + 2;
    sm.red_full = sm.gfree + 2;
    sm.red_free = sm.red_full + 2 * kWarps;

    if (tid == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&sm.full_w[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.gfull[i], kWarps);
            mbar_init(&sm.gfree[i], kWarps);
        }
        for (int i = 0; i < 2 * kWarps; ++i) {
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

    // Warp c reads the records u = c, c + 8, ... of the sequence (group u / P,
    // pair u % P), record u through slot u % R. Positions advance by steps,
    // without divisions: (ci, cj) the next record to read, in slot s of
    // phase ph; (fi, fj) the next record to fetch, R places ahead.
    const Conv kc = make_conv();
    const uint64_t pol = policy_evict_first();
    // Weights may stream before the preceding kernel has finished only when
    // the caller declared them read-only.
    if (!a.prefetch_w) pdl_wait();
    int ci = c / max(P, 1), cj = c - ci * max(P, 1);
    int fi = ci, fj = cj;
    for (int u = c; u < R; u += kWarps) {
        if (lane == 0 && fi < ntiles) load_record(a, sm, fi, fj, u, G0, p0, pol);
        step_pos(fi, fj, P);
    }
    __syncwarp();
    pdl_wait();                                       // X, Y and the slot rows are the preceding kernel's
    const float *xr[M];
    int yrow[M];
#pragma unroll
    for (int t = 0; t < M; ++t) {
        yrow[t] = t < a.m ? (a.rows ? __ldg(a.rows + t) : t) : 0;
        xr[t] = a.X + static_cast<int64_t>(yrow[t]) * a.ldx;
    }
    // Record-MMA mode: in column tile nt, this lane's B column is token
    // 4 nt + lane / 8. For m <= 2 the live columns are lanes 0-15 only, so X
    // is built in one pass: lanes 0-15 build block 2p of a pair p and lanes
    // 16-31 block 2p + 1 for the same columns, handed to lanes 0-15 by
    // shuffles. With one column tile a warp's X values are loaded one record
    // ahead; with more (m = 5..16) they are loaded where they are used (L1).
    // (W4A8 mode: column tile nt holds tokens 8 nt .. 8 nt + 7, one per column)
    constexpr int NT = A8 ? (M + 7) / 8 : (MMA ? (M + 3) / 4 : 1);
    constexpr bool kOnePass = MMA && !A8 && M <= 2;
    const int xb1 = kOnePass ? (lane >> 4) : 0;       // block of the pair this lane builds
    const int col_tok = kOnePass ? ((lane & 15) >> 3) : (lane >> 3);
    const bool col_live = col_tok < M && col_tok < a.m;
    const float *xcol = a.X + (col_live ? static_cast<int64_t>(a.rows ? __ldg(a.rows + col_tok) : col_tok) * a.ldx : 0);
    // further column tiles (NT > 1): token 4 nt + lane / 8
    const float *xcolt[NT];
    bool livet[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int tok = A8 ? 8 * nt + (lane >> 2) : 4 * nt + (lane >> 3);
        const bool own = A8 || nt > 0;
        livet[nt] = own ? (tok < M && tok < a.m) : col_live;
        xcolt[nt] = own ? a.X + (livet[nt] ? static_cast<int64_t>(a.rows ? __ldg(a.rows + tok) : tok) * a.ldx : 0)
                        : xcol;
    }

    bool ok = true;
    int s = c;
    uint32_t ph = 0;
    int pending = c;                                  // first of this warp's records not yet read
    // record-MMA mode: X values of the warp's next record, loaded one record
    // ahead so that their latency hides behind the current record's work
    float4 xn[2][2];
    if (MMA && !A8 && NT == 1 && ci < ntiles) {
        const int b0 = 2 * (p0 + cj);
        if (kOnePass) {
            x_load(xcol, b0 + xb1, col_live && b0 + xb1 < a.nb, lane, xn[0][0], xn[0][1]);
        } else {
            x_load(xcol, b0, col_live, lane, xn[0][0], xn[0][1]);
            x_load(xcol, b0 + 1, col_live && b0 + 1 < a.nb, lane, xn[1][0], xn[1][1]);
        }
    }
    for (int g = 0; g < ntiles && ok; ++g) {
        const int tb = g & 1;
        float yp[4][M];
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int t = 0; t < M; ++t) yp[r][t] = 0.0f;
        float yq[NT][8][2];
        float y8[NT][8][4];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                yq[nt][r][0] = yq[nt][r][1] = 0.0f;
                y8[nt][r][0] = y8[nt][r][1] = y8[nt][r][2] = y8[nt][r][3] = 0.0f;
            }
        for (; ci == g; step_pos(ci, cj, P)) {
            if (!warp_wait(&sm.full_w[s], ph, a.wait_ns)) { ok = false; break; }
            const uint8_t *rec = sm.w + static_cast<size_t>(s) * kRecordBytes;
            const int b0 = 2 * (p0 + cj);
            if constexpr (A8) {
                // a missing second block is padding (weights exactly 0) against X = 0
                uint4 bf[NT][2];
                float sc[NT][2][2];
                const int tq = lane & 3;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        float4 xa, xb;
                        x_load(xcolt[nt], b0 + b, livet[nt] && b0 + b < a.nb, lane, xa, xb);
                        float scale;
                        x_codes(xa, xb, bf[nt][b], scale);
                        sc[nt][b][0] = __shfl_sync(0xFFFFFFFFu, scale, 8 * tq);       // token 2 tq's column
                        sc[nt][b][1] = __shfl_sync(0xFFFFFFFFu, scale, 8 * tq + 4);   // token 2 tq + 1
                    }
                mma_record_a8<NT>(rec, bf, sc, lane, y8);
            } else if (MMA) {
                // a missing second block is padding (weights exactly 0) against X = 0
                uint4 bf[NT][2];
                float su[NT][2];
                const int tq = lane & 3;                  // token of this lane's accumulators, per tile
                if (NT > 1) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int b = 0; b < 2; ++b) {
                            float4 xa, xb;
                            x_load(xcolt[nt], b0 + b, livet[nt] && b0 + b < a.nb, lane, xa, xb);
                            float inv;
                            x_fragments(xa, xb, lane, bf[nt][b], inv);
                            su[nt][b] = __shfl_sync(0xFFFFFFFFu, inv, 8 * tq);
                        }
                } else if (kOnePass) {
                    uint4 v;
                    float inv;
                    x_fragments(xn[0][0], xn[0][1], lane & 15, v, inv);
                    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
                    uint4 hi;
                    hi.x = __shfl_down_sync(0xFFFFFFFFu, v.x, 16);
                    hi.y = __shfl_down_sync(0xFFFFFFFFu, v.y, 16);
                    hi.z = __shfl_down_sync(0xFFFFFFFFu, v.z, 16);
                    hi.w = __shfl_down_sync(0xFFFFFFFFu, v.w, 16);
                    bf[0][0] = lane < 16 ? v : zero;      // columns 4-7 (tokens 2, 3) are zero
                    bf[0][1] = lane < 16 ? hi : zero;
                    su[0][0] = __shfl_sync(0xFFFFFFFFu, inv, 8 * tq);     // token tq's hi column
                    su[0][1] = __shfl_sync(0xFFFFFFFFu, inv, 16 + 8 * tq);
                } else {
                    float inv0, inv1;
                    x_fragments(xn[0][0], xn[0][1], lane, bf[0][0], inv0);
                    x_fragments(xn[1][0], xn[1][1], lane, bf[0][1], inv1);
                    su[0][0] = __shfl_sync(0xFFFFFFFFu, inv0, 8 * tq);
                    su[0][1] = __shfl_sync(0xFFFFFFFFu, inv1, 8 * tq);
                }
                int ni = ci, nj = cj;
                step_pos(ni, nj, P);
                if (NT == 1 && ni < ntiles) {
                    const int nb0 = 2 * (p0 + nj);
                    if (kOnePass) {
                        x_load(xcol, nb0 + xb1, col_live && nb0 + xb1 < a.nb, lane, xn[0][0], xn[0][1]);
                    } else {
                        x_load(xcol, nb0, col_live, lane, xn[0][0], xn[0][1]);
                        x_load(xcol, nb0 + 1, col_live && nb0 + 1 < a.nb, lane, xn[1][0], xn[1][1]);
                    }
                }
                mma_record<NT>(rec, bf, su, lane, yq);
            } else {
                uint32_t sc[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) sc[r] = lds32(rec + kRecScaleOff + 4 * (lane + 32 * r));
                gemv_block<M>(rec + kRecQs0Off, 0, sc, xr, 32 * b0, lane, kc, yp);
                if (b0 + 1 < a.nb) gemv_block<M>(rec + kRecQs1Off, 16, sc, xr, 32 * (b0 + 1), lane, kc, yp);
            }
            // Every lane has its values of the slot in registers: refill it
            // with the record R places ahead (same warp, same slot).
            __syncwarp();
            if (lane == 0 && fi < ntiles) load_record(a, sm, fi, fj, s, G0, p0, pol);
            step_pos(fi, fj, P);
            pending += kWarps;
            s += kWarps;
            if (s >= R) s -= R, ph ^= 1u;
        }
        if (!ok) break;
        if (g >= 2 && !warp_wait(&sm.gfree[tb], ((g >> 1) & 1) ^ 1u, a.wait_ns)) { ok = false; break; }
        float *pp = sm.part + (tb * kWarps + c) * M * kGroupRows;
        if constexpr (A8) {
            const int g = lane >> 2, t = lane & 3;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int c2 = 0; c2 < 2; ++c2) {
                    const int tok = 8 * nt + 2 * t + c2;
                    if (tok < M)
#pragma unroll
                        for (int r = 0; r < 8; ++r) {
                            pp[tok * kGroupRows + 16 * r + g] = y8[nt][r][c2];
                            pp[tok * kGroupRows + 16 * r + g + 8] = y8[nt][r][2 + c2];
                        }
                }
        } else if (MMA) {
            const int g = lane >> 2;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int t = 4 * nt + (lane & 3);
                if (t < M)
#pragma unroll
                    for (int r = 0; r < 8; ++r) {
                        pp[t * kGroupRows + 16 * r + g] = yq[nt][r][0];
                        pp[t * kGroupRows + 16 * r + g + 8] = yq[nt][r][1];
                    }
            }
        } else {
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int t = 0; t < M; ++t) pp[t * kGroupRows + lane + 32 * r] = yp[r][t];
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.gfull[tb]);
        float yg[(M + 1) / 2];
        if (g >= 1 && !reduce_group<M>(a, sm, g - 1, c, lane, rank, G0, yrow, false, yg)) { ok = false; break; }
    }
    // When every CTA of the grid has a single group, its slices meet through
    // the closing cluster barrier (measured faster there; with two groups per
    // CTA, on 14336 x 4096 at m = 3 and 4, slower than the handshake).
    const bool merged = S > 1 && a.groups <= a.clusters;
    float ylast[(M + 1) / 2];
    const bool fin = ok && ntiles > 0;
    if (fin) ok = reduce_group<M>(a, sm, ntiles - 1, c, lane, rank, G0, yrow, merged, ylast);
    if (!ok) {
        fail(a);
        // A warp that gave up may still have copies landing in its slots
        // (the records after the last one it read): wait for them, bounded,
        // so that none lands after the CTA has exited.
        for (int u = pending; u < total && u < pending + R; u += kWarps)
            if (!mbar_wait(&sm.full_w[u % R], (u / R) & 1, a.wait_ns)) break;
        __syncwarp();
    }

    // Every CTA of the cluster stays until the others are done with its
    // shared memory and barriers; the barrier also makes the other slices'
    // rows of the last group, stored before it, visible to the first CTA.
    if (S > 1) {
        cluster_sync();
        if (merged && fin && ok && rank == 0) write_rows<M>(a, sm, ntiles - 1, c, lane, G0, yrow, ylast);
    }
}

size_t gemv_smem(int M, int S, int ring)
{
    const size_t part = static_cast<size_t>(2 * kWarps) * M * kGroupRows * 4;
    const size_t red = S > 1 ? static_cast<size_t>(2 * (S - 1)) * M * kGroupRows * 4 : 0;
    const size_t bars = static_cast<size_t>(ring + 4 + 4 * kWarps) * 8;
    return static_cast<size_t>(ring) * kRecordBytes + part + red + bars;
}

#define Q4_GEMV_CASES(MMA, A8)                                                                  \
    switch (M) {                                                                               \
    case 1: return reinterpret_cast<const void *>(&gemv_kernel<1, MMA, A8>);                   \
    case 2: return reinterpret_cast<const void *>(&gemv_kernel<2, MMA, A8>);                   \
    case 3: return reinterpret_cast<const void *>(&gemv_kernel<3, MMA, A8>);                   \
    case 4: return reinterpret_cast<const void *>(&gemv_kernel<4, MMA, A8>);                   \
    case 5: return reinterpret_cast<const void *>(&gemv_kernel<5, MMA, A8>);                   \
    case 6: return reinterpret_cast<const void *>(&gemv_kernel<6, MMA, A8>);                   \
    case 7: return reinterpret_cast<const void *>(&gemv_kernel<7, MMA, A8>);                   \
    case 8: return reinterpret_cast<const void *>(&gemv_kernel<8, MMA, A8>);                   \
    case 9: return reinterpret_cast<const void *>(&gemv_kernel<9, MMA, A8>);                   \
    case 10: return reinterpret_cast<const void *>(&gemv_kernel<10, MMA, A8>);                 \
    case 11: return reinterpret_cast<const void *>(&gemv_kernel<11, MMA, A8>);                 \
    case 12: return reinterpret_cast<const void *>(&gemv_kernel<12, MMA, A8>);                 \
    case 13: return reinterpret_cast<const void *>(&gemv_kernel<13, MMA, A8>);                 \
    case 14: return reinterpret_cast<const void *>(&gemv_kernel<14, MMA, A8>);                 \
    case 15: return reinterpret_cast<const void *>(&gemv_kernel<15, MMA, A8>);                 \
    default: return reinterpret_cast<const void *>(&gemv_kernel<16, MMA, A8>);                 \
    }

// The kernel instance for M tokens in a mode (the CUDA-core mode is built for
// M <= 4 only).
const void *gemv_fn(int M, int mode)
{
    if (mode == kGemvModeW4A8) Q4_GEMV_CASES(true, true)
    if (mode == kGemvModeRecordMma) Q4_GEMV_CASES(true, false)
    switch (M) {
    case 1: return reinterpret_cast<const void *>(&gemv_kernel<1, false, false>);
    case 2: return reinterpret_cast<const void *>(&gemv_kernel<2, false, false>);
    case 3: return reinterpret_cast<const void *>(&gemv_kernel<3, false, false>);
    default: return reinterpret_cast<const void *>(&gemv_kernel<4, false, false>);
    }
}
#undef Q4_GEMV_CASES

// Largest number of clusters of S CTAs of the M-token kernel with `smem`
// bytes of dynamic shared memory that the current device can hold at once
// (clusters live inside one GPC, so this is less than the SM count allows
// whenever S does not divide a GPC's SMs). Cached per (device, M, S, smem).
int max_active_clusters(int M, int S, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, M, S, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void *fn = gemv_fn(M, M > kGemvMaxM ? kGemvModeRecordMma : kGemvModeFma);
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
// that fits one CTA's shared memory and the deepest that leaves room for a
// second CTA on the SM, neither deeper than the CTA's records need. The
// number of clusters is capped by what the device holds at once (a second
// wave would double the time).
//
// Costs are in record times of one SM's share of HBM (about 0.1 us on
// GB300), fitted to graph-replay timings of the record-MMA mode:
// - Single-group plans (one 128-row group per cluster) come first: their
//   slices meet through the closing cluster barrier, and on every layer
//   measured the best plan was one of them. Their cost is the busiest SM's
//   records (1.5 each with one CTA on the SM, 1.1 each with two), plus the
//   records a CTA must wait for beyond its ring (three times as dear with a
//   ring of one record per warp), plus per-slice cluster overheads, plus
//   the start-up that cannot overlap the preceding call when no SM has room
//   for the next call's CTA.
// - Grids with more groups than resident clusters pay the busiest SM's
//   records at the rate its CTAs sustain and the per-group overheads.
bool plan_gemv(int64_t m, int64_t k, int64_t n, int sm_count, GemvPlan *plan)
{
    if (m < 1 || m > kRecordMmaMaxM || sm_count < 1) return false;
    const int M = static_cast<int>(m);
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const double total = static_cast<double>(groups * np);
    const size_t half = kSmemPerSM / 2 - 1024;
    GemvPlan best;
    double best_cost = 1e300;
    for (int S = 1; S <= kMaxSlices && S <= np; ++S) {
        const int64_t P = ceil_div(np, S);
        const int need = static_cast<int>(std::min<int64_t>(kMaxRing, std::max<int64_t>(kWarps, ceil_div(P, kWarps) * kWarps)));
        for (int cand = 0; cand < 4; ++cand) {
            const int two = cand & 1;
            const int top = cand < 2 ? need : kMaxRing;    // a ring deeper than the records only helps
            if (cand >= 2 && top == need) continue;          // a CTA with several groups
            const size_t limit = two ? half : kSmemOptIn;
            int ring = 0;
            for (int r = top; r >= kWarps && ring == 0; r -= kWarps)
                if (gemv_smem(M, S, r) <= limit) ring = r;
            if (ring == 0) continue;
            const size_t smem = gemv_smem(M, S, ring);
            const bool two_fit = smem <= half;
            if (!two && two_fit) continue;             // the same plan as two = 1
            const int64_t cmax = max_active_clusters(M, S, smem);
            if (cmax < 1) continue;
            const int64_t clusters = std::min<int64_t>(groups, cmax);
            const int64_t tiles = ceil_div(groups, clusters);
            const int64_t ctas = clusters * S;
            const int per_sm = ctas > sm_count ? 2 : 1;
            const double no_overlap = (!two_fit || per_sm == 2) ? 10.0 : 0.0;
            double cost;
            if (tiles == 1) {
                const double Pd = static_cast<double>(P);
                const double work = per_sm == 2 ? 2.0 * Pd * 1.1 : Pd * 1.5;
                const double starve =
                    per_sm == 1 && P > ring ? static_cast<double>(P - ring) * (ring <= kWarps ? 3.0 : 1.0) : 0.0;
                const double slices = S > 1 ? 3.0 + 2.0 * (S - 2) : 0.0;
                cost = work + starve + slices + no_overlap;
            } else {
                const double rate = per_sm == 2 ? 1.0 : (two_fit ? 0.9 : 0.8);
                const double stream = std::max(static_cast<double>(tiles * P * per_sm) / rate, total / sm_count);
                cost = 1000.0 + stream + 0.5 * static_cast<double>(tiles) + (S > 1 ? 2.0 : 0.0) + 1.5 * no_overlap;
            }
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.M = M;
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

cudaError_t launch_gemv(const GemvPlan &plan, const DecodeArgs &args, int mode, cudaStream_t s)
{
    const void *fn = gemv_fn(plan.M, mode);
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
