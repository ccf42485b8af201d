// q4mm_matvec.cu -- the decode mat-vec for m <= 16 token rows (the decode step
// and continuous batching: golem, "Several conversations, one pass"; golem-
// server, "Several conversations, in one pass"; goinfer ch. 10, "What the
// kernels are": the quantised mat-vec is the decode workhorse, bound by the
// weight read). The design goal is to turn a packed record over in fewer
// issue slots than one SM's share of HBM takes to deliver it, and to keep the
// work after the dependency wait (X, the products, the K-slice reduction)
// short, because in a stream of calls that work is what one call adds to the
// next.
//
// Arithmetic, exact up to the final scaling. X is the B operand of the warp-
// level MMA (mma.sync m16n8k16, bf16 x bf16 -> fp32). Each 32-element block of
// a token row is scaled by a power of two 2^-e (its largest |x| lands in
// [1, 2)) and split into two fixed-point terms: hi, a multiple of 2^-7, and
// lo, a multiple of 2^-15 (x - hi rounded to that grid): 16 bits relative to
// the block's largest |x|. Both are exact in bf16. The A operand is a nibble
// OR'ed into the bf16 pattern of 128: exactly 128 + q, one lop3 for two
// weights and no subtraction. The accumulator of a column starts at
// -136 * (sum of that column's terms over the block), so it ends at
// sum (q - 8) * term. Every partial sum on the way is a multiple of 2^-7 (hi)
// or 2^-15 (lo) below 2^15 (2^5), at most 22 significant bits, so fp32 holds
// each one exactly and the tensor core's summation order cannot change the
// block's two dot products. They are then added and scaled by d * 2^e in fp32
// (one rounding each) into the row's fp32 total. All-eights weights give 0
// exactly, and integer inputs stay integer-exact.
// A block of X that holds a NaN or an infinity switches the CTA to exact
// weights (bf16 q - 8, one subtraction more per two weights) with a zero
// starting accumulator, so that infinities meet (q - 8) and d as IEEE
// arithmetic says; the finite blocks' results are the same bits either way.
//
// MMA columns. For m <= 4 the hi and lo terms of a (token, block) are two
// columns of the 8, and the 8 columns hold up to four (token, block) pairs:
// m = 1 puts a record's two blocks side by side in one accumulator tile
// (thread t of a quad holds block t), m = 2 the two blocks of two tokens, m = 4
// one block of four tokens. The weights of a 16 x 16 tile are dequantised once
// for all of them. For m = 5..16 the columns are tokens and the hi and lo
// terms are two MMAs into the same accumulator (exact weights, zero start:
// the partial sums, below 2^9 on a 2^-15 grid, stay exact too).
//
// K permutation. Thread (g, t) of a warp (lane 4g + t) holds A rows g and
// g + 8. Its A registers come straight from word t of the rows' 16 nibble
// bytes (elements 4t .. 4t+3 low, 16 + 4t .. 19 + 4t high) in the packed
// layout as it is; the B fragments of X are staged in the same permutation.
//
// Work split: 128-row groups and S slices of K; the S CTAs of a thread-block
// cluster hold the S slices of the groups c, c + C, ... of cluster c, and the
// slices of a row meet in the first CTA (DSMEM), summed in slice order, so
// results are bitwise reproducible and no global scratch is used.
//
// Warps (eight per CTA, all alike; two CTAs fit on an SM: one call's and the
// next's). After the dependency wait the warps stage the CTA's slice of X
// once as B fragments in shared memory. Warp c owns the records
// u = c (mod 8) of the CTA's sequence (its groups x its pairs, in that
// order) and the ring slots they pass through: lane 0 refills a slot with a
// 1-D bulk copy of the record R places ahead as soon as the warp has read it,
// so every barrier has one waiter and no copy is in flight when the CTA
// exits; with weights declared read-only the first R records stream before
// the dependency wait. A warp takes a record's eight row tiles at once, which
// gives the scheduler eight independent streams of loads, dequantisation and
// MMAs. At the end of a group each warp leaves its partial rows in shared
// memory; one group later warp c sums rows 16c .. 16c + 15 of the eight
// partials in order, then the cluster's slices of them, and writes Y. Every
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

constexpr int kErrTimeout = 5;                   // Q4_ERR_DEVICE_TIMEOUT
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSliceRows = kGroupRows / kWarps;  // rows of a group each warp finishes
constexpr int kMaxSlices = 8;
constexpr int kMaxRing = 32;                     // records; a multiple of kWarps when slots are refilled

// B entries per (record, block): one for m <= 4 (hi and lo are columns), a hi
// and a lo entry per eight tokens otherwise.
__host__ __device__ constexpr int entries_per_block(int M) { return M <= 4 ? 1 : 2 * (M / 8); }
// Lanes of an entry that hold X: for m <= 2 only the lanes of the block's own
// columns (8 for m = 1, 16 for m = 2; the others read zeros and are not
// stored), all 32 otherwise.
__host__ __device__ constexpr int entry_lanes(int M) { return M == 1 ? 8 : M == 2 ? 16 : 32; }
__host__ __device__ constexpr int entry_bytes(int M) { return entry_lanes(M) * 16; }

// Weight formats the kernel streams: Q4_0 records (4608 bytes: 128 rows x 2
// blocks, scales and nibbles) or per-output-channel int8 records (8192 bytes:
// 128 rows x 64 codes, the rows' scales applied when Y is written).
constexpr int kFmtQ4 = 0;
constexpr int kFmtW8 = 1;
__host__ __device__ constexpr int rec_bytes(int F) { return F == kFmtW8 ? kW8RecordBytes : kRecordBytes; }
// int8 records: B entries per record (hi and lo columns for m <= 4; a hi and a
// lo entry per eight tokens otherwise), each 32 lanes x 32 bytes (four k-steps)
__host__ __device__ constexpr int w8_entries(int M) { return M <= 4 ? 1 : 2 * (M / 8); }
// Shared-memory bytes per record of the CTA's slice: X fragments, parameters.
__host__ __device__ constexpr int xfrag_bytes(int M, int F)
{
    return F == kFmtW8 ? w8_entries(M) * 1024 : 2 * entries_per_block(M) * entry_bytes(M);
}
__host__ __device__ constexpr int xparam_bytes(int M, int F) { return F == kFmtW8 ? M * 4 : 2 * M * (M <= 4 ? 32 : 4); }
// The parameter region of a slice, rounded up so that what follows it (row
// buffers, barriers) stays 16-byte aligned.
__host__ __device__ constexpr int xparam_region(int M, int F, int Pmax) { return (Pmax * xparam_bytes(M, F) + 15) / 16 * 16; }
// Accumulators per row of a thread: one (m <= 4), or two tokens per eight.
__host__ __device__ constexpr int acc_width(int M) { return M <= 4 ? 1 : M / 4; }

struct VSmem {
    uint8_t *ring;        // [R] records
    uint4 *bimg;          // [Pmax] x xfrag_bytes: B fragments of X (Q4_0: [2][NQ][entry_lanes];
                          // int8: [entries][32 lanes][2])
    float4 *xp;           // Q4_0, M <= 4: [Pmax][2][M][2] {the four columns' corrections}, {2^e, 0, 0, 0}
    float *xs;            // Q4_0, M >= 8: [Pmax][2][M] 2^e; int8: [Pmax][M] 2^e
    float *part;          // [NB][8][M][128] the warps' partial rows of a group (single-group
                          // grids with the whole slice in the ring: warp c's first ring slot)
    int part_stride;      // floats from one warp's partial rows to the next's
    float *red;           // [NR][S - 1][M][128] other slices' rows of a group (first CTA)
    int *flag;            // a staged block of X was not finite
    uint64_t *full;                   // [R]
    uint64_t *gfull, *gfree;          // [2] partials of a group parity written / summed
    uint64_t *red_full, *red_free;    // [2][8] a row slice's other slices landed / slot free
    uint64_t *red_tx;                 // single-group grids: the other slices' rows landed
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

__device__ __forceinline__ uint32_t ld32(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint4 ld128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 ld128f(uint32_t addr)
{
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0,%1,%2,%3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 ld64f(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// D += A * B, m16n8k16, bf16 operands, fp32 accumulate in place. Volatile, so
// that a record's MMAs, which consume its shared-memory loads, are issued
// before the record's slot is refilled.
__device__ __forceinline__ void mma_acc(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulate in place (exact fp16
// weights times X's fp16 terms).
__device__ __forceinline__ void mma_acc_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Asynchronous store of one fp32 value into another CTA's shared memory
// (cluster address), counted in bytes on that CTA's barrier `bar` (cluster
// address).
__device__ __forceinline__ void st_async_f32(uint32_t dst, float v, uint32_t bar)
{
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.b32 [%0], %1, [%2];" ::"r"(dst),
                 "r"(__float_as_uint(v)), "r"(bar)
                 : "memory");
}

// The closing cluster barrier in two halves: arrive without ordering any
// memory access, and wait.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

__device__ __forceinline__ unsigned absmax_bits(const float4 &v)
{
    return max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
               max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu));
}

__device__ __forceinline__ uint32_t pack_half2_rn(float a, float b)
{
    const __half2 h = __floats2half2_rn(a, b);   // a in the low half
    return *reinterpret_cast<const uint32_t *>(&h);
}

// Fp16 scale of a row's block from the record's scale word (block 0 in the
// low half, block 1 in the high half).
__device__ __forceinline__ float half_of(uint32_t w, int hi)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(hi ? (w >> 16) : (w & 0xFFFFu))));
}

// The eight weights of one word of split-half nibbles (bytes 4t .. 4t+3 of a
// block's qs) as bf16 pairs in the K permutation: v[0] = (e, e+2),
// v[1] = (e+16, e+18), v[2] = (e+1, e+3), v[3] = (e+17, e+19), e = 4t.
// Biased: 128 + q. Exact: q - 8.
template <bool EXACT>
__device__ __forceinline__ void weights_of(uint32_t w, uint32_t v[4])
{
    v[0] = nib2_bf16_biased(w);
    v[1] = nib2_bf16_biased(w >> 4);
    v[2] = nib2_bf16_biased(w >> 8);
    v[3] = nib2_bf16_biased(w >> 12);
    if (EXACT) {
        const uint32_t k136 = 0x43084308u;   // bf16 (136, 136)
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = bf16x2_sub(v[i], k136);
    }
}

// m <= 4: the eight weights of one word of split-half nibbles (bytes
// 4t .. 4t+3 of a block's qs) as fp16 pairs, the low nibbles for k-step 0
// and the high ones, in place at bits 4-7, for k-step 1:
//   k0a = (e, e+2), k0b = (e+1, e+3): 1024 + q;
//   k1a = (e+16, e+18), k1b = (e+17, e+19): 1024 + 16q;   e = 4t.
// Exact: q - 8 and 16 (q - 8). One shift and four lop3 for eight weights.
template <bool EXACT>
__device__ __forceinline__ void weights_f16(uint32_t w, uint32_t &k0a, uint32_t &k0b, uint32_t &k1a, uint32_t &k1b)
{
    const uint32_t w8 = w >> 8;
    k0a = lop3_and_or(w, 0x000F000Fu, 0x64006400u);
    k0b = lop3_and_or(w8, 0x000F000Fu, 0x64006400u);
    k1a = lop3_and_or(w, 0x00F000F0u, 0x64006400u);
    k1b = lop3_and_or(w8, 0x00F000F0u, 0x64006400u);
    if (EXACT) {
        k0a = hsub2_bits(k0a, 0x64086408u);   // fp16 (1032, 1032)
        k0b = hsub2_bits(k0b, 0x64086408u);
        k1a = hsub2_bits(k1a, 0x64806480u);   // fp16 (1152, 1152)
        k1b = hsub2_bits(k1b, 0x64806480u);
    }
}

// Stage the CTA's slice of X (pairs p0 .. p0 + P - 1) as B fragments. A task
// is one (pair, block, token): four lanes of a warp (t = 0..3) hold its 32
// values, eight each (elements 4t .. 4t+3 and 16 + 4t .. 19 + 4t), agree on
// its scale by two shuffles, split them into hi and lo and store them where
// the consumer lanes read them:
//   m <= 4: entry (p, b), column pair c (c = b for m = 1, 2b + token for
//           m = 2, token for m = 4): hi at lane 4 (2c) + t, lo at
//           lane 4 (2c + 1) + t (for m <= 2 the entry stores only the
//           block's own lanes);
//   m >= 8: entries (p, b, 2h) (hi) and (p, b, 2h + 1) (lo) of tokens
//           8h .. 8h + 7: lane 4 (token - 8h) + t.
// A fragment register holds, for k-step 0, elements (4t, 4t+2) and
// (16+4t, 18+4t); for k-step 1, (4t+1, 4t+3) and (17+4t, 19+4t).
template <int M>
__device__ __forceinline__ void stage_x(const DecodeArgs &a, const VSmem &sm, int p0, int P, int w, int lane)
{
    constexpr int kNQ = entries_per_block(M);
    constexpr int kBatch = 4;                       // tasks per lane whose loads are in flight together
    const int q = lane >> 2, t = lane & 3;
    const int E = P * 2 * M;
    for (int e0 = 8 * w; e0 < E; e0 += 8 * kWarps * kBatch) {
        float4 xa[kBatch], xb[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = e0 + 8 * kWarps * i + q;
            const int tok = e % M, pb = e / M;
            const int blk = 2 * p0 + pb;            // pb = 2p + b
            xa[i] = make_float4(0.f, 0.f, 0.f, 0.f);
            xb[i] = xa[i];
            if (e < E && blk < a.nb && tok < a.m) {
                const int xrow = a.rows ? __ldg(a.rows + tok) : tok;
                const float *xr = a.X + static_cast<int64_t>(xrow) * a.ldx + 32 * blk + 4 * t;
                xa[i] = __ldg(reinterpret_cast<const float4 *>(xr));
                xb[i] = __ldg(reinterpret_cast<const float4 *>(xr + 16));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (e0 + 8 * kWarps * i >= E) break;    // warp-uniform: none of the warp's tasks is left
            const int e = e0 + 8 * kWarps * i + q;
            const int tok = e % M, pb = e / M, b = pb & 1;
            unsigned mb = max(absmax_bits(xa[i]), absmax_bits(xb[i]));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            const bool fin = mb < 0x7F800000u;
            int ex = 0;                             // largest |x| in [2^ex, 2^(ex + 1))
            if (fin && mb >= 0x00800000u) ex = min(static_cast<int>(mb >> 23) - 127, 126);
            else if (fin && mb != 0u) ex = -126;    // subnormal: scaled below 1
            const float sd = __uint_as_float(static_cast<unsigned>(127 - ex) << 23);   // 2^-ex
            const float v[8] = {xa[i].x, xa[i].y, xa[i].z, xa[i].w, xb[i].x, xb[i].y, xb[i].z, xb[i].w};
            float hi[8], lo[8];
            // m <= 4 keeps lo scaled by 2^8 (on the same 2^-7 grid as hi); the
            // high-nibble half of the block (elements 16..31, k-step 1) is
            // divided by 16 to meet weights of 1024 + 16q
            constexpr float kLoScale = M <= 4 ? 256.0f : 1.0f;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                if (fin) {
                    // |s| < 2: adding 1.5 * 2^16 rounds to a multiple of 2^-7 (nearest,
                    // ties to even), adding 1.5 * 2^8 to a multiple of 2^-15
                    const float s = v[j] * sd;
                    hi[j] = __fsub_rn(__fadd_rn(s, 0x1.8p16f), 0x1.8p16f);
                    lo[j] = __fsub_rn(__fadd_rn(__fsub_rn(s, hi[j]), 0x1.8p8f), 0x1.8p8f) * kLoScale;
                } else {
                    hi[j] = v[j];
                    lo[j] = 0.f;
                }
                if (M <= 4 && j >= 4) hi[j] *= 0.0625f, lo[j] *= 0.0625f;
            }
            uint4 *ent = sm.bimg + static_cast<size_t>(pb * kNQ) * entry_lanes(M);
            const float su = __uint_as_float(static_cast<unsigned>(127 + ex) << 23);   // 2^ex
            if constexpr (M <= 4) {
                // the four columns' sums (k-step 0 and 1, hi and lo), exact:
                // multiples of 2^-7 or 2^-11 far below 2^24 of them
                float s0h = hi[0] + hi[1] + hi[2] + hi[3], s0l = lo[0] + lo[1] + lo[2] + lo[3];
                float s1h = hi[4] + hi[5] + hi[6] + hi[7], s1l = lo[4] + lo[5] + lo[6] + lo[7];
#pragma unroll
                for (int o = 1; o <= 2; o <<= 1) {
                    s0h += __shfl_xor_sync(0xFFFFFFFFu, s0h, o);
                    s0l += __shfl_xor_sync(0xFFFFFFFFu, s0l, o);
                    s1h += __shfl_xor_sync(0xFFFFFFFFu, s1h, o);
                    s1l += __shfl_xor_sync(0xFFFFFFFFu, s1l, o);
                }
                if (e >= E) continue;
                uint4 fh, fl;
                fh.x = pack_half2_rn(hi[0], hi[2]);     // k-step 0, b0: elements 4t, 4t+2
                fh.y = pack_half2_rn(hi[1], hi[3]);     //           b1: 4t+1, 4t+3
                fh.z = pack_half2_rn(hi[4], hi[6]);     // k-step 1, b0: 16+4t, 18+4t (/16)
                fh.w = pack_half2_rn(hi[5], hi[7]);     //           b1: 17+4t, 19+4t (/16)
                fl.x = pack_half2_rn(lo[0], lo[2]);
                fl.y = pack_half2_rn(lo[1], lo[3]);
                fl.z = pack_half2_rn(lo[4], lo[6]);
                fl.w = pack_half2_rn(lo[5], lo[7]);
                // column pair c = b (m = 1), 2b + token (m = 2), token (m = 4):
                // lanes 4 (2c) + t and 4 (2c + 1) + t, stored from the entry's
                // first live lane
                const int c = M == 1 ? 0 : tok;
                ent[4 * (2 * c) + t] = fh;
                ent[4 * (2 * c + 1) + t] = fl;
                if (t == 0) {
                    // a weight of 1024 + q (k-step 0) or 1024 + 16q against x / 16
                    // (k-step 1) carries 1032 x or 72 x = 1152 (x / 16) beyond (q - 8) x
                    float4 *pp = sm.xp + (pb * M + tok) * 2;
                    pp[0] = fin ? make_float4(-1032.0f * s0h, -1032.0f * s0l, -1152.0f * s1h, -1152.0f * s1l)
                                : make_float4(0.f, 0.f, 0.f, 0.f);
                    pp[1] = make_float4(su, 0.f, 0.f, 0.f);
                }
            } else {
                if (e >= E) continue;
                uint4 fh, fl;
                fh.x = pack_bf16x2_rn(hi[0], hi[2]);
                fh.y = pack_bf16x2_rn(hi[4], hi[6]);
                fh.z = pack_bf16x2_rn(hi[1], hi[3]);
                fh.w = pack_bf16x2_rn(hi[5], hi[7]);
                fl.x = pack_bf16x2_rn(lo[0], lo[2]);
                fl.y = pack_bf16x2_rn(lo[4], lo[6]);
                fl.z = pack_bf16x2_rn(lo[1], lo[3]);
                fl.w = pack_bf16x2_rn(lo[5], lo[7]);
                const int h = tok >> 3;
                ent[(2 * h) * 32 + 4 * (tok & 7) + t] = fh;
                ent[(2 * h + 1) * 32 + 4 * (tok & 7) + t] = fl;
                if (t == 0) sm.xs[pb * M + tok] = su;
            }
            if (!fin && t == 0) *reinterpret_cast<volatile int *>(sm.flag) = 1;
        }
    }
}


// int8 weights: stage the CTA's slice of X (pairs p0 .. p0 + P - 1, 64
// columns each) as fp16 B fragments. A task is one (pair, token): four lanes
// (t = 0..3) hold its 64 values, sixteen each (columns 16t .. 16t + 15 of the
// pair), agree on a power-of-two scale that puts the largest |x| into
// [2^14, 2^15), and split each value into fp16 hi + lo (22 significant bits
// relative to that largest |x|); a pair holding a NaN or an infinity is taken
// unscaled, hi = x, lo = 0. Lane (g, t) of an entry holds column g and, in
// its two 16-byte halves, k-steps 0-1 and 2-3: k-step s reads columns
// (16t + 4s, 16t + 4s + 2) and (16t + 4s + 1, 16t + 4s + 3), the order in
// which the record's bytes 16t .. 16t + 15 of a row become A fragments.
//   m <= 4: one entry, column g = 2 token + (0 hi, 1 lo);
//   m >= 8: entries 2h (hi) and 2h + 1 (lo), column g = token - 8h.
template <int M>
__device__ __forceinline__ void stage_x_w8(const DecodeArgs &a, const VSmem &sm, int p0, int P, int w, int lane)
{
    constexpr int kNE = w8_entries(M);
    constexpr int kBatch = 2;
    const int q = lane >> 2, t = lane & 3;
    const int E = P * M;
    for (int e0 = 8 * w; e0 < E; e0 += 8 * kWarps * kBatch) {
        float4 xv[kBatch][4];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int e = e0 + 8 * kWarps * i + q;
            const int tok = e % M, p = e / M;
            const int col = (p0 + p) * kPairK + 16 * t;
#pragma unroll
            for (int j = 0; j < 4; ++j) xv[i][j] = make_float4(0.f, 0.f, 0.f, 0.f);
            // (a pair's second block is absent when k is an odd number of
            // blocks: its lanes t = 2, 3 read zeros)
            if (e < E && col < 32 * a.nb && tok < a.m) {
                const int xrow = a.rows ? __ldg(a.rows + tok) : tok;
                const float *xr = a.X + static_cast<int64_t>(xrow) * a.ldx + col;
#pragma unroll
                for (int j = 0; j < 4; ++j) xv[i][j] = __ldg(reinterpret_cast<const float4 *>(xr + 4 * j));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (e0 + 8 * kWarps * i >= E) break;    // warp-uniform
            const int e = e0 + 8 * kWarps * i + q;
            const int tok = e % M, p = e / M;
            unsigned mb = 0u;
#pragma unroll
            for (int j = 0; j < 4; ++j) mb = max(mb, absmax_bits(xv[i][j]));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 1));
            mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, 2));
            const bool fin = mb < 0x7F800000u;
            int ex = 0;                             // scale 2^ex puts the largest |x| in [2^14, 2^15)
            if (fin && mb != 0u) ex = max(-100, min(100, 14 - (static_cast<int>(mb >> 23) - 127)));
            if (fin && mb != 0u && mb < 0x00800000u) ex = 100;
            const float sd = __uint_as_float(static_cast<unsigned>(127 + ex) << 23);
            const float v[16] = {xv[i][0].x, xv[i][0].y, xv[i][0].z, xv[i][0].w, xv[i][1].x, xv[i][1].y,
                                 xv[i][1].z, xv[i][1].w, xv[i][2].x, xv[i][2].y, xv[i][2].z, xv[i][2].w,
                                 xv[i][3].x, xv[i][3].y, xv[i][3].z, xv[i][3].w};
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2)
#pragma unroll
                for (int o = 0; o < 2; ++o) {
                    // k-step s2, b0 (o = 0): columns 4 s2, 4 s2 + 2; b1: 4 s2 + 1, 4 s2 + 3
                    const float x0 = fin ? v[4 * s2 + o] * sd : v[4 * s2 + o];
                    const float x1 = fin ? v[4 * s2 + o + 2] * sd : v[4 * s2 + o + 2];
                    const __half2 h = __floats2half2_rn(x0, x1);
                    const float2 back = __half22float2(h);
                    const __half2 l = __floats2half2_rn(x0 - back.x, x1 - back.y);
                    hi[2 * s2 + o] = *reinterpret_cast<const uint32_t *>(&h);
                    lo[2 * s2 + o] = fin ? *reinterpret_cast<const uint32_t *>(&l) : 0u;
                }
            if (e >= E) continue;
            uint4 *ent = reinterpret_cast<uint4 *>(reinterpret_cast<uint8_t *>(sm.bimg) +
                                                   static_cast<size_t>(p) * xfrag_bytes(M, kFmtW8));
            const int eh = M <= 4 ? 0 : 2 * (tok >> 3);
            const int el = M <= 4 ? 0 : eh + 1;
            const int lh = M <= 4 ? 4 * (2 * tok) + t : 4 * (tok & 7) + t;
            const int ll = M <= 4 ? 4 * (2 * tok + 1) + t : lh;
            ent[(eh * 32 + lh) * 2] = make_uint4(hi[0], hi[1], hi[2], hi[3]);
            ent[(eh * 32 + lh) * 2 + 1] = make_uint4(hi[4], hi[5], hi[6], hi[7]);
            ent[(el * 32 + ll) * 2] = make_uint4(lo[0], lo[1], lo[2], lo[3]);
            ent[(el * 32 + ll) * 2 + 1] = make_uint4(lo[4], lo[5], lo[6], lo[7]);
            if (t == 0) sm.xs[p * M + tok] = __uint_as_float(static_cast<unsigned>(127 - ex) << 23);   // 2^-ex
        }
    }
}

// One record for all eight row tiles: y[rt][r][i] += row 16 rt + g + 8r's
// part, for the token (and block, m <= 2) thread t holds:
//   m = 1:  token 0, block t of the record (t < 2; summed over t at the end);
//   m = 2:  token t & 1, block t >> 1 (summed over t, t ^ 2 at the end);
//   m = 4:  token t;
//   m = 8:  token 2t + i;
//   m = 16: token 8 (i >> 1) + 2t + (i & 1).
// `p` is the record's pair within the slice (its X entries).
template <int M, bool EXACT>
__device__ __forceinline__ void record_mma(const VSmem &sm, uint32_t rec, int p, int lane,
                                           float (&y)[8][2][acc_width(M)])
{
    constexpr int kNQ = entries_per_block(M);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bimg = smem_u32(sm.bimg) + static_cast<uint32_t>(p * 2 * kNQ * entry_bytes(M) + lane * 16);
    if constexpr (M <= 2) {
        // one accumulator tile for both blocks: lanes outside a block's own
        // columns take zeros for its MMAs
        constexpr int SH = M == 1 ? 3 : 4;          // block of the columns of lane (g, t)
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t bl = smem_u32(sm.bimg) +
                            static_cast<uint32_t>((p * 2 + (lane >> SH)) * entry_bytes(M) + (lane & (entry_lanes(M) - 1)) * 16);
        const uint4 B0 = (lane >> SH) == 0 ? ld128(bl) : zero;
        const uint4 B1 = (lane >> SH) == 1 ? ld128(bl) : zero;
        // this thread's (block, token) column pair: corrections and 2^e
        const int bt = M == 1 ? t : (t >> 1);
        const bool live = M == 2 || t < 2;
        const float4 *pp = sm.xp + ((p * 2 + (live ? bt : 0)) * M + (M == 1 ? 0 : (t & 1))) * 2;
        const float4 cr = live ? ld128f(smem_u32(pp)) : make_float4(0.f, 0.f, 0.f, 0.f);
        const float su = live ? ld128f(smem_u32(pp + 1)).x : 0.f;
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
            const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
            const uint32_t w00 = ld32(rec + kRecQs0Off + 16 * r0 + 4 * t);
            const uint32_t w01 = ld32(rec + kRecQs0Off + 16 * r0 + 128 + 4 * t);
            const uint32_t w10 = ld32(rec + kRecQs1Off + 16 * r0 + 4 * t);
            const uint32_t w11 = ld32(rec + kRecQs1Off + 16 * r0 + 128 + 4 * t);
            const uint32_t s0 = ld32(rec + kRecScaleOff + 4 * r0), s1 = ld32(rec + kRecScaleOff + 4 * r0 + 32);
            uint32_t a[2][2][4];                    // [block][k-step][fragment]
            weights_f16<EXACT>(w00, a[0][0][0], a[0][0][2], a[0][1][0], a[0][1][2]);
            weights_f16<EXACT>(w01, a[0][0][1], a[0][0][3], a[0][1][1], a[0][1][3]);
            weights_f16<EXACT>(w10, a[1][0][0], a[1][0][2], a[1][1][0], a[1][1][2]);
            weights_f16<EXACT>(w11, a[1][0][1], a[1][0][3], a[1][1][1], a[1][1][3]);
            // k-step 0 (low nibbles) and k-step 1 (high nibbles) accumulate
            // apart, each from its columns' corrections
            float D[4] = {EXACT ? 0.f : cr.x, EXACT ? 0.f : cr.y, EXACT ? 0.f : cr.x, EXACT ? 0.f : cr.y};
            float E[4] = {EXACT ? 0.f : cr.z, EXACT ? 0.f : cr.w, EXACT ? 0.f : cr.z, EXACT ? 0.f : cr.w};
            mma_acc_f16(D, a[0][0], B0.x, B0.y);
            mma_acc_f16(E, a[0][1], B0.z, B0.w);
            mma_acc_f16(D, a[1][0], B1.x, B1.y);
            mma_acc_f16(E, a[1][1], B1.z, B1.w);
            const float d0 = live ? half_of(s0, bt) : 0.f;
            const float d1 = live ? half_of(s1, bt) : 0.f;
            // hi column + lo column (kept 2^8 larger)
            y[rt][0][0] = fmaf(d0 * su, fmaf(D[1] + E[1], 0x1p-8f, D[0] + E[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(d1 * su, fmaf(D[3] + E[3], 0x1p-8f, D[2] + E[2]), y[rt][1][0]);
        }
    } else if constexpr (M == 4) {
        // a tile per block: thread t holds token t
        const uint4 B0 = ld128(bimg), B1 = ld128(bimg + 512);
        const float4 c0 = ld128f(smem_u32(sm.xp + (p * 2 * 4 + t) * 2));
        const float4 c1 = ld128f(smem_u32(sm.xp + ((p * 2 + 1) * 4 + t) * 2));
        const float su0 = ld128f(smem_u32(sm.xp + (p * 2 * 4 + t) * 2 + 1)).x;
        const float su1 = ld128f(smem_u32(sm.xp + ((p * 2 + 1) * 4 + t) * 2 + 1)).x;
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
            const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
            const uint32_t w00 = ld32(rec + kRecQs0Off + 16 * r0 + 4 * t);
            const uint32_t w01 = ld32(rec + kRecQs0Off + 16 * r0 + 128 + 4 * t);
            const uint32_t w10 = ld32(rec + kRecQs1Off + 16 * r0 + 4 * t);
            const uint32_t w11 = ld32(rec + kRecQs1Off + 16 * r0 + 128 + 4 * t);
            const uint32_t s0 = ld32(rec + kRecScaleOff + 4 * r0), s1 = ld32(rec + kRecScaleOff + 4 * r0 + 32);
            uint32_t a[2][2][4];
            weights_f16<EXACT>(w00, a[0][0][0], a[0][0][2], a[0][1][0], a[0][1][2]);
            weights_f16<EXACT>(w01, a[0][0][1], a[0][0][3], a[0][1][1], a[0][1][3]);
            weights_f16<EXACT>(w10, a[1][0][0], a[1][0][2], a[1][1][0], a[1][1][2]);
            weights_f16<EXACT>(w11, a[1][0][1], a[1][0][3], a[1][1][1], a[1][1][3]);
            float D0[4] = {EXACT ? 0.f : c0.x, EXACT ? 0.f : c0.y, EXACT ? 0.f : c0.x, EXACT ? 0.f : c0.y};
            float E0[4] = {EXACT ? 0.f : c0.z, EXACT ? 0.f : c0.w, EXACT ? 0.f : c0.z, EXACT ? 0.f : c0.w};
            float D1[4] = {EXACT ? 0.f : c1.x, EXACT ? 0.f : c1.y, EXACT ? 0.f : c1.x, EXACT ? 0.f : c1.y};
            float E1[4] = {EXACT ? 0.f : c1.z, EXACT ? 0.f : c1.w, EXACT ? 0.f : c1.z, EXACT ? 0.f : c1.w};
            mma_acc_f16(D0, a[0][0], B0.x, B0.y);
            mma_acc_f16(D1, a[1][0], B1.x, B1.y);
            mma_acc_f16(E0, a[0][1], B0.z, B0.w);
            mma_acc_f16(E1, a[1][1], B1.z, B1.w);
            y[rt][0][0] = fmaf(half_of(s0, 0) * su0, fmaf(D0[1] + E0[1], 0x1p-8f, D0[0] + E0[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(half_of(s1, 0) * su0, fmaf(D0[3] + E0[3], 0x1p-8f, D0[2] + E0[2]), y[rt][1][0]);
            y[rt][0][0] = fmaf(half_of(s0, 1) * su1, fmaf(D1[1] + E1[1], 0x1p-8f, D1[0] + E1[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(half_of(s1, 1) * su1, fmaf(D1[3] + E1[3], 0x1p-8f, D1[2] + E1[2]), y[rt][1][0]);
        }
    } else {
        // tiles (block b, half h): tokens 8h .. 8h + 7; hi and lo are two MMAs
        constexpr int H = M / 8;
        float2 su[2][H];
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int h = 0; h < H; ++h) su[b][h] = ld64f(smem_u32(sm.xs + (p * 2 + b) * M + 8 * h + 2 * t));
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
            const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
            const uint32_t s0 = ld32(rec + kRecScaleOff + 4 * r0), s1 = ld32(rec + kRecScaleOff + 4 * r0 + 32);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const uint32_t qo = b ? kRecQs1Off : kRecQs0Off;
                const uint32_t w0 = ld32(rec + qo + 16 * r0 + 4 * t), w1 = ld32(rec + qo + 16 * r0 + 128 + 4 * t);
                uint32_t v0[4], v1[4];
                weights_of<true>(w0, v0);
                weights_of<true>(w1, v1);
                const uint32_t A0[4] = {v0[0], v1[0], v0[1], v1[1]}, A1[4] = {v0[2], v1[2], v0[3], v1[3]};
                const float dg = half_of(s0, b), dg8 = half_of(s1, b);
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    const uint4 Bh = ld128(bimg + static_cast<uint32_t>((b * kNQ + 2 * h) * 512));
                    const uint4 Bl = ld128(bimg + static_cast<uint32_t>((b * kNQ + 2 * h + 1) * 512));
                    float D[4] = {0.f, 0.f, 0.f, 0.f};
                    mma_acc(D, A0, Bh.x, Bh.y);
                    mma_acc(D, A1, Bh.z, Bh.w);
                    mma_acc(D, A0, Bl.x, Bl.y);
                    mma_acc(D, A1, Bl.z, Bl.w);
                    y[rt][0][2 * h] = fmaf(dg * su[b][h].x, D[0], y[rt][0][2 * h]);
                    y[rt][0][2 * h + 1] = fmaf(dg * su[b][h].y, D[1], y[rt][0][2 * h + 1]);
                    y[rt][1][2 * h] = fmaf(dg8 * su[b][h].x, D[2], y[rt][1][2 * h]);
                    y[rt][1][2 * h + 1] = fmaf(dg8 * su[b][h].y, D[3], y[rt][1][2 * h + 1]);
                }
            }
        }
    }
}


// Four int8 codes (stored as 128 + c) into two fp16 pairs of c, exact: the
// bytes go under the fp16 pattern of 1024 (prmt), 1152 comes off.
__device__ __forceinline__ void codes_f16(uint32_t w, uint32_t &even, uint32_t &odd)
{
    uint32_t e, o;
    asm("prmt.b32 %0, %1, %2, 0x4240;" : "=r"(e) : "r"(w), "r"(0x64646464u));   // bytes 0, 2
    asm("prmt.b32 %0, %1, %2, 0x4341;" : "=r"(o) : "r"(w), "r"(0x64646464u));   // bytes 1, 3
    even = hsub2_bits(e, 0x64806480u);
    odd = hsub2_bits(o, 0x64806480u);
}

// One int8 record for all eight row tiles: y[rt][r][i] += 2^-e * (row's
// codes . X's pair), for the token thread t holds (m <= 4: token t; m = 8:
// 2t + i; m = 16: 8 (i >> 1) + 2t + (i & 1)); the row's scale comes when Y is
// written.
template <int M>
__device__ __forceinline__ void record_mma_w8(const VSmem &sm, uint32_t rec, int p, int lane,
                                              float (&y)[8][2][acc_width(M)])
{
    constexpr int kNE = w8_entries(M);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bimg = smem_u32(sm.bimg) + static_cast<uint32_t>(p * xfrag_bytes(M, kFmtW8) + lane * 32);
    if constexpr (M <= 4) {
        const uint4 e0 = ld128(bimg), e1 = ld128(bimg + 16);
        const float su = t < M ? sm.xs[p * M + t] : 0.f;
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
            const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
            const uint4 qa = ld128(rec + r0 * kPairK + 16 * t), qb = ld128(rec + (r0 + 8) * kPairK + 16 * t);
            const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
            float D[4] = {0.f, 0.f, 0.f, 0.f}, E[4] = {0.f, 0.f, 0.f, 0.f};
            const uint32_t bx[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                uint32_t ae, ao, be, bo;
                codes_f16(wa[s2], ae, ao);
                codes_f16(wb[s2], be, bo);
                const uint32_t A[4] = {ae, be, ao, bo};
                if (s2 & 1) mma_acc_f16(E, A, bx[2 * s2], bx[2 * s2 + 1]);
                else mma_acc_f16(D, A, bx[2 * s2], bx[2 * s2 + 1]);
            }
            y[rt][0][0] = fmaf(su, (D[0] + E[0]) + (D[1] + E[1]), y[rt][0][0]);
            y[rt][1][0] = fmaf(su, (D[2] + E[2]) + (D[3] + E[3]), y[rt][1][0]);
        }
    } else {
        constexpr int H = M / 8;
        float2 su[H];
#pragma unroll
        for (int h = 0; h < H; ++h) su[h] = ld64f(smem_u32(sm.xs + p * M + 8 * h + 2 * t));
#pragma unroll
        for (int rt = 0; rt < 8; ++rt) {
            const uint32_t r0 = static_cast<uint32_t>(16 * rt + g);
            const uint4 qa = ld128(rec + r0 * kPairK + 16 * t), qb = ld128(rec + (r0 + 8) * kPairK + 16 * t);
            const uint32_t wa[4] = {qa.x, qa.y, qa.z, qa.w}, wb[4] = {qb.x, qb.y, qb.z, qb.w};
            uint32_t A[4][4];
#pragma unroll
            for (int s2 = 0; s2 < 4; ++s2) {
                uint32_t ae, ao, be, bo;
                codes_f16(wa[s2], ae, ao);
                codes_f16(wb[s2], be, bo);
                A[s2][0] = ae, A[s2][1] = be, A[s2][2] = ao, A[s2][3] = bo;
            }
#pragma unroll
            for (int h = 0; h < H; ++h) {
                float D[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
                    const uint32_t eb = bimg + static_cast<uint32_t>((2 * h + hl) * 1024);
                    const uint4 e0 = ld128(eb), e1 = ld128(eb + 16);
                    mma_acc_f16(D, A[0], e0.x, e0.y);
                    mma_acc_f16(D, A[1], e0.z, e0.w);
                    mma_acc_f16(D, A[2], e1.x, e1.y);
                    mma_acc_f16(D, A[3], e1.z, e1.w);
                }
                y[rt][0][2 * h] = fmaf(su[h].x, D[0], y[rt][0][2 * h]);
                y[rt][0][2 * h + 1] = fmaf(su[h].y, D[1], y[rt][0][2 * h + 1]);
                y[rt][1][2 * h] = fmaf(su[h].x, D[2], y[rt][1][2 * h]);
                y[rt][1][2 * h + 1] = fmaf(su[h].y, D[3], y[rt][1][2 * h + 1]);
            }
        }
    }
    (void)kNE;
}

// Token of accumulator i of thread t.
template <int M>
__device__ __forceinline__ int acc_token(int t, int i)
{
    if constexpr (M <= 2) return M == 1 ? 0 : (t & 1);
    else if constexpr (M == 4) return t;
    else if constexpr (M == 8) return 2 * t + i;
    else return 8 * (i >> 1) + 2 * t + (i & 1);
}

// Store this warp's partial rows of a group (all 128 rows) into part[tb][c]
// ([M][128] floats).
template <int M>
__device__ __forceinline__ void store_partials(const VSmem &sm, int tb, int c, int lane, float (&y)[8][2][acc_width(M)])
{
    constexpr int NY = acc_width(M);
    const int g = lane >> 2, t = lane & 3;
    // m = 1: blocks 0 and 1 of a row sit in threads t = 0, 1; m = 2: blocks
    // 0 and 1 of a token in threads t and t ^ 2
#pragma unroll
    for (int rt = 0; rt < 8; ++rt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if constexpr (M == 1) y[rt][r][0] += __shfl_xor_sync(0xFFFFFFFFu, y[rt][r][0], 1);
            if constexpr (M == 2) y[rt][r][0] += __shfl_xor_sync(0xFFFFFFFFu, y[rt][r][0], 2);
        }
    const bool writes = M == 1 ? t == 0 : (M == 2 ? t < 2 : true);
    float *pp = sm.part + static_cast<size_t>(tb * kWarps + c) * sm.part_stride;
    if (writes)
#pragma unroll
        for (int rt = 0; rt < 8; ++rt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < NY; ++i) pp[acc_token<M>(t, i) * kGroupRows + 16 * rt + g + 8 * r] = y[rt][r][i];
}

// Rows of a warp's slice in the reduction: lane l handles row 16c + (l & 15)
// and tokens l / 16, + 2, ...
template <int M>
struct SliceRows {
    static constexpr int NT = (M + 1) / 2;
    float v[NT];
};

// Sum the eight warps' partials of a group (buffer tb) for this warp's rows,
// in warp order.
template <int M>
__device__ __forceinline__ void sum_partials(const VSmem &sm, int tb, int c, int lane, SliceRows<M> &s)
{
    const int row = c * kSliceRows + (lane & (kSliceRows - 1));
    const int t0 = lane >> 4;
#pragma unroll
    for (int h = 0; h < SliceRows<M>::NT; ++h) {
        const int tok = t0 + 2 * h;
        float v = 0.0f;
        if (tok < M)
#pragma unroll
            for (int w = 0; w < kWarps; ++w) v += sm.part[static_cast<size_t>(tb * kWarps + w) * sm.part_stride + tok * kGroupRows + row];
        s.v[h] = v;
    }
}

// Write this warp's rows of group g to Y after adding the other slices'
// (red buffer rb of this CTA's shared memory).
template <int M>
__device__ __forceinline__ void write_rows(const DecodeArgs &a, const VSmem &sm, int g, int G0, int c, int lane, int S,
                                           int rb, const SliceRows<M> &s)
{
    const int row = c * kSliceRows + (lane & (kSliceRows - 1));
    const int t0 = lane >> 4;
    const int64_t grow = static_cast<int64_t>(G0 + g * a.clusters) * kGroupRows + row;
    if (grow >= a.n) return;
#pragma unroll
    for (int h = 0; h < SliceRows<M>::NT; ++h) {
        const int tok = t0 + 2 * h;
        if (tok < M && tok < a.m) {
            float v = s.v[h];
            for (int r = 1; r < S; ++r) v += sm.red[((rb * (S - 1) + r - 1) * M + tok) * kGroupRows + row];
            if (a.row_scale) v *= __ldg(a.row_scale + grow);   // int8 weights: the channel's scale
            const int yr = a.rows ? __ldg(a.rows + tok) : tok;
            a.Y[static_cast<int64_t>(yr) * a.ldy + grow] = v;
        }
    }
}

// Reduce group g (partials in buffer g & 1) for this warp's rows and meet
// the cluster's other slices through the per-group handshake (grids whose
// CTAs have several groups), or keep them for the closing exchange (`keep`,
// single-group grids).
template <int M>
__device__ __forceinline__ bool reduce_group(const DecodeArgs &a, const VSmem &sm, int g, int c, int lane, int rank,
                                             int G0, bool merged, SliceRows<M> &keep)
{
    const int S = a.S;
    const int tb = g & 1;
    const uint32_t par = static_cast<uint32_t>((g >> 1) & 1);
    if (!warp_wait(&sm.gfull[tb], par, a.wait_ns)) return false;
    SliceRows<M> s;
    sum_partials<M>(sm, tb, c, lane, s);
    __syncwarp();
    if (lane == 0) mbar_arrive(&sm.gfree[tb]);
    if (merged) {
        keep = s;
        return true;
    }
    if (rank > 0) {
        // this slice's rows into the first CTA's buffer tb, then signal it
        if (g >= 2 && !warp_wait_cluster(&sm.red_free[tb * kWarps + c], par ^ 1u, a.wait_ns)) return false;
        const int row = c * kSliceRows + (lane & (kSliceRows - 1));
        const uint32_t dst = mapa_shared(smem_u32(sm.red), 0u) +
                             static_cast<uint32_t>((((tb * (S - 1) + rank - 1) * M) * kGroupRows + row) * 4);
#pragma unroll
        for (int h = 0; h < SliceRows<M>::NT; ++h) {
            const int tok = (lane >> 4) + 2 * h;
            if (tok < M) st_cluster_f32(dst + static_cast<uint32_t>(tok * kGroupRows * 4), s.v[h]);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_full[tb * kWarps + c]), 0u));
        return true;
    }
    if (S > 1 && !warp_wait_cluster(&sm.red_full[tb * kWarps + c], par, a.wait_ns)) return false;
    write_rows<M>(a, sm, g, G0, c, lane, S, tb, s);
    if (S > 1) {
        __syncwarp();
        if (lane == 0)
            for (int r = 1; r < S; ++r)
                mbar_arrive_remote(mapa_shared(smem_u32(&sm.red_free[tb * kWarps + c]), static_cast<uint32_t>(r)));
    }
    return true;
}

// Issue the bulk copy of the CTA's record n (group n / P, pair n % P of its
// slice) into ring slot s. Lane 0 of the slot's warp only.
template <int F>
__device__ __forceinline__ void load_record(const DecodeArgs &a, const VSmem &sm, int n, int P, int s, int G0, int p0,
                                            uint64_t pol)
{
    constexpr int kRB = rec_bytes(F);
    const int gi = n / P, j = n - gi * P;
    const int64_t rec = static_cast<int64_t>(G0 + gi * a.clusters) * a.np + p0 + j;
    mbar_arrive_expect_tx(&sm.full[s], kRB);
    bulk_g2s_hint(sm.ring + static_cast<size_t>(s) * kRB, a.W + rec * kRB, kRB, &sm.full[s], pol);
}

// The warp's records, group by group: products into registers, partial rows
// into shared memory at each group's end, the previous group's reduction.
// `pending` tracks the warp's first record not yet read (for the drain after
// a failure).
template <int M, bool EXACT, int F>
__device__ __forceinline__ bool consume(const DecodeArgs &a, const VSmem &sm, int c, int lane, int rank, int G0, int p0,
                                        int P, int ntiles, bool merged, uint64_t pol, int &pending,
                                        SliceRows<M> &keep)
{
    constexpr int NY = acc_width(M);
    const int R = a.ring;
    const int total = ntiles * P;
    const uint32_t ring0 = smem_u32(sm.ring);
    int n = c;                                        // the warp's next record
    for (int g = 0; g < ntiles; ++g) {
        float y[8][2][NY];
#pragma unroll
        for (int rt = 0; rt < 8; ++rt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < NY; ++i) y[rt][r][i] = 0.f;
        for (; n < (g + 1) * P; n += kWarps) {
            const int s = n % R;
            if (!warp_wait(&sm.full[s], static_cast<uint32_t>((n / R) & 1), a.wait_ns)) return false;
            const uint32_t rec = ring0 + static_cast<uint32_t>(s * rec_bytes(F));
            if constexpr (F == kFmtW8) record_mma_w8<M>(sm, rec, n - g * P, lane, y);
            else record_mma<M, EXACT>(sm, rec, n - g * P, lane, y);
            // the record's MMAs, which consume its loads, are issued: refill
            // the slot with the record R places ahead (same warp)
            __syncwarp();
            if (lane == 0 && n + R < total) load_record<F>(a, sm, n + R, P, s, G0, p0, pol);
            pending = n + kWarps;
        }
        const int tb = g & 1;
        if (g >= 2 && !warp_wait(&sm.gfree[tb], static_cast<uint32_t>(((g >> 1) & 1) ^ 1), a.wait_ns)) return false;
        store_partials<M>(sm, tb, c, lane, y);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.gfull[tb]);
        if (g >= 1 && !reduce_group<M>(a, sm, g - 1, c, lane, rank, G0, false, keep)) return false;
    }
    return ntiles == 0 || reduce_group<M>(a, sm, ntiles - 1, c, lane, rank, G0, merged, keep);
}

template <int M, int F>
__global__ void __launch_bounds__(kThreads, M >= 16 ? 1 : 2) matvec_kernel(const DecodeArgs call, const ExpertSet set)
{
    constexpr int kRB = rec_bytes(F);
    extern __shared__ __align__(128) uint8_t smem_raw[];
    constexpr int kNQ = entries_per_block(M);
    const int tid = threadIdx.x, c = tid >> 5, lane = tid & 31;
    const int S = call.S;
    const int rank = S > 1 ? static_cast<int>(cluster_ctarank()) : 0;
    // A plain call: cluster c holds groups c, c + clusters, ... An expert
    // set: cluster c holds group c % groups of expert c / groups, whose
    // weights, rows of X and rows of Y the set names.
    DecodeArgs a = call;
    int G0 = static_cast<int>(blockIdx.x) / S;
    if (set.count > 0) {
        const int e = G0 / call.groups;
        G0 -= e * call.groups;
        a.W = set.W[e];
        a.m = set.m[e];
        a.X = call.X + static_cast<int64_t>(set.row0[e]) * call.ldx;
        a.Y = call.Y + static_cast<int64_t>(set.row0[e]) * call.ldy;
        a.clusters = call.groups;
    }
    const int ntiles = G0 < a.groups ? (a.groups - 1 - G0) / a.clusters + 1 : 0;
    const int p0 = rank * a.pbase + min(rank, a.prem);
    const int P = a.pbase + (rank < a.prem ? 1 : 0);
    const int total = ntiles * P;                   // records this CTA streams
    const int R = a.ring;
    // Every CTA of the cluster lays out its shared memory for the largest
    // slice, so that a barrier or a row buffer sits at the same offset in all
    // of them (remote accesses map this CTA's offsets onto another CTA's).
    const int Pmax = a.pbase + (a.prem > 0 ? 1 : 0);
    const bool merged = S > 1 && a.groups <= a.clusters;   // every CTA has a single group
    const int NB = a.groups > a.clusters ? 2 : 1;          // partial-row buffers

    VSmem sm;
    sm.ring = smem_raw;
    sm.bimg = reinterpret_cast<uint4 *>(sm.ring + static_cast<size_t>(R) * kRB);
    uint8_t *after_b = sm.ring + static_cast<size_t>(R) * kRB + static_cast<size_t>(Pmax) * xfrag_bytes(M, F);
    sm.xp = reinterpret_cast<float4 *>(after_b);
    sm.xs = reinterpret_cast<float *>(after_b);
    float *after_x = reinterpret_cast<float *>(after_b + xparam_region(M, F, Pmax));
    // With a single group per CTA and the whole slice in the ring (no slot is
    // refilled), warp c's partial rows go into its first ring slot, which it
    // has read by then.
    const bool part_in_ring = a.groups <= a.clusters && R >= Pmax && R >= kWarps && M * kGroupRows * 4 <= kRB;
    sm.part = part_in_ring ? reinterpret_cast<float *>(sm.ring) : after_x;
    sm.red = after_x + (part_in_ring ? 0 : static_cast<size_t>(NB) * kWarps * M * kGroupRows);
    sm.part_stride = part_in_ring ? kRB / 4 : M * kGroupRows;
    const int red_floats = S > 1 ? (merged ? 1 : 2) * (S - 1) * M * kGroupRows : 0;
    sm.flag = reinterpret_cast<int *>(sm.red + red_floats);
    sm.full = reinterpret_cast<uint64_t *>(sm.flag + 4);
    sm.gfull = sm.full + R;
    sm.gfree = sm.gfull + 2;
    sm.red_full = sm.gfree + 2;
    sm.red_free = sm.red_full + 2 * kWarps;
    sm.red_tx = sm.red_free + 2 * kWarps;

    if (tid == 0) {
        for (int i = 0; i < R; ++i) mbar_init(&sm.full[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.gfull[i], kWarps);
            mbar_init(&sm.gfree[i], kWarps);
        }
        for (int i = 0; i < 2 * kWarps; ++i) {
            mbar_init(&sm.red_full[i], S > 1 ? S - 1 : 1);
            mbar_init(&sm.red_free[i], 1);
        }
        mbar_init(sm.red_tx, 1);
        // single-group grids: the other slices each send all 128 rows x M
        // tokens of the group as asynchronous stores counted on red_tx
        if (merged && rank == 0)
            mbar_arrive_expect_tx(sm.red_tx, static_cast<uint32_t>((S - 1) * kGroupRows * M * 4));
        *sm.flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // The next kernel in the stream may be scheduled now: it waits for this
    // one to complete before it reads anything this one writes.
    pdl_launch_dependents();
    if (S > 1) cluster_sync(); // every CTA's barriers initialised before any remote access

    // Weights may stream before the preceding kernel has finished only when
    // the caller declared them read-only.
    const uint64_t pol = policy_evict_first();
    if (!a.prefetch_w) pdl_wait();
    if (lane == 0)
        for (int n = c; n < R && n < total; n += kWarps) load_record<F>(a, sm, n, P, n, G0, p0, pol);
    __syncwarp();
    pdl_wait();                                       // X, Y and the slot rows are the preceding kernel's
    if constexpr (F == kFmtW8) stage_x_w8<M>(a, sm, p0, P, c, lane);
    else stage_x<M>(a, sm, p0, P, c, lane);
    __syncthreads();

    int pending = c;                                  // the warp's first record not yet read
    SliceRows<M> keep;
#pragma unroll
    for (int h = 0; h < SliceRows<M>::NT; ++h) keep.v[h] = 0.f;
    // (int8 weights are exact codes: no biased form)
    const bool ok = (F == kFmtW8 || M >= 8 || *reinterpret_cast<volatile int *>(sm.flag) != 0)
                        ? consume<M, true, F>(a, sm, c, lane, rank, G0, p0, P, ntiles, merged, pol, pending, keep)
                        : consume<M, (M >= 8 || F == kFmtW8), F>(a, sm, c, lane, rank, G0, p0, P, ntiles, merged, pol,
                                                                 pending, keep);
    if (!ok) {
        fail(a);
        // A warp that gave up may still have copies landing in its slots
        // (the records after the last one it read): wait for them, bounded,
        // so that none lands after the CTA has exited.
        for (int n = pending; n < total && n < pending + R; n += kWarps)
            if (!warp_wait(&sm.full[n % R], static_cast<uint32_t>((n / R) & 1), a.wait_ns)) break;
    }

    if (merged) {
        // The other slices' rows of the group travel as asynchronous stores
        // counted on the first CTA's red_tx, sent on every path (zeros after
        // a failure) so that the count always completes. The closing cluster
        // barrier only keeps every CTA alive until all have arrived; the
        // first CTA arrives first and waits for it last.
        const int row = c * kSliceRows + (lane & (kSliceRows - 1));
        if (rank > 0) {
            const uint32_t dst = mapa_shared(smem_u32(sm.red), 0u) +
                                 static_cast<uint32_t>(((rank - 1) * M * kGroupRows + row) * 4);
            const uint32_t bar = mapa_shared(smem_u32(sm.red_tx), 0u);
#pragma unroll
            for (int h = 0; h < SliceRows<M>::NT; ++h) {
                const int tok = (lane >> 4) + 2 * h;
                if (tok < M)
                    st_async_f32(dst + static_cast<uint32_t>(tok * kGroupRows * 4), ok && ntiles > 0 ? keep.v[h] : 0.f,
                                 bar);
            }
            cluster_arrive_relaxed();
            cluster_wait();
        } else {
            cluster_arrive_relaxed();
            const bool got = warp_wait_cluster(sm.red_tx, 0u, a.wait_ns);
            if (got && ok && ntiles > 0) write_rows<M>(a, sm, 0, G0, c, lane, S, 0, keep);
            if (!got) fail(a);
            cluster_wait();
            // every other CTA has sent before arriving: after a wait that gave
            // up, let those stores land before this CTA exits
            if (!got) warp_wait_cluster(sm.red_tx, 0u, a.wait_ns);
        }
    } else if (S > 1) {
        // Every CTA of the cluster stays until the others are done with its
        // shared memory and barriers.
        cluster_sync();
    }
}

// Shared memory of a plan; `parts` = 2 when CTAs hold several groups (the
// partial rows and the slices' rows are then double-buffered).
size_t matvec_smem(int M, int F, int Pmax, int S, int ring, int parts)
{
    const bool part_in_ring = parts == 1 && ring >= Pmax && ring >= kWarps && M * kGroupRows * 4 <= rec_bytes(F);
    size_t b = static_cast<size_t>(ring) * rec_bytes(F);
    b += static_cast<size_t>(Pmax) * xfrag_bytes(M, F);
    b += static_cast<size_t>(xparam_region(M, F, Pmax));
    b += part_in_ring ? 0 : static_cast<size_t>(parts) * kWarps * M * kGroupRows * 4;
    b += S > 1 ? static_cast<size_t>(parts * (S - 1)) * M * kGroupRows * 4 : 0;
    b += 16;                                                  // flag
    b += static_cast<size_t>(ring + 4 + 4 * kWarps + 1) * 8;  // barriers
    return b;
}

// The instance for m token rows: 1, 2, 4, 8 or 16.
int instance_of(int64_t m) { return m <= 1 ? 1 : m <= 2 ? 2 : m <= 4 ? 4 : m <= 8 ? 8 : 16; }

template <int F>
const void *matvec_fn_f(int M)
{
    switch (M) {
    case 1: return reinterpret_cast<const void *>(&matvec_kernel<1, F>);
    case 2: return reinterpret_cast<const void *>(&matvec_kernel<2, F>);
    case 4: return reinterpret_cast<const void *>(&matvec_kernel<4, F>);
    case 8: return reinterpret_cast<const void *>(&matvec_kernel<8, F>);
    default: return reinterpret_cast<const void *>(&matvec_kernel<16, F>);
    }
}

const void *matvec_fn(int M, int F) { return F == kFmtW8 ? matvec_fn_f<kFmtW8>(M) : matvec_fn_f<kFmtQ4>(M); }

// Largest number of clusters of S CTAs with `smem` bytes of dynamic shared
// memory that the current device holds at once (clusters live inside one
// GPC). Cached per (device, instance, S, smem).
int matvec_max_clusters(int M, int F, int S, size_t smem)
{
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, size_t>, int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const auto key = std::make_tuple(dev, M, F, S, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    const void *fn = matvec_fn(M, F);
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

// Issue cost of a record relative to one SM's share of HBM time for it
// (first estimates from the source's instruction counts; the planner only
// compares plans).
double record_cost(int M) { return M <= 2 ? 0.5 : M == 4 ? 0.6 : M == 8 ? 0.9 : 1.6; }

} // namespace

// Choose the cluster size S (K slices per 128-row group), the number of
// persistent clusters and the ring depth (records, a multiple of 8). For each
// S: the deepest ring that fits one CTA's shared memory and the deepest that
// leaves room for a second CTA on the SM (the next call's), neither deeper
// than the CTA's records. The number of clusters is capped by what the
// device holds at once (a second wave would double the time). Cost, in
// record times of one SM's share of HBM: the busiest warp's records (the
// CTA's records are dealt to its eight warps in turn) at the kernel's issue
// cost, or the whole layer's stream if that is longer; the records a CTA
// must wait for beyond its ring; the slices' reduction; per-group handshakes
// of CTAs with several groups; and the start-up that cannot overlap the
// preceding call when no SM has room for the next call's CTA.
bool plan_matvec(int64_t m, int64_t k, int64_t n, int sm_count, MatvecPlan *plan, int fmt)
{
    if (m < 1 || m > 16 || sm_count < 1) return false;
    const int F = fmt == kMatvecInt8 ? kFmtW8 : kFmtQ4;
    // int8 weights stage all four token columns of a tile (m <= 4 share the
    // four-token instance)
    const int M = F == kFmtW8 ? std::max(4, instance_of(m)) : instance_of(m);
    // a record's weight bytes in units of a Q4_0 record
    const double rw = static_cast<double>(rec_bytes(F)) / kRecordBytes;
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const double total = static_cast<double>(groups * np);
    const size_t half = kSmemPerSM / 2 - 1024;
    const double rc = record_cost(M);
    MatvecPlan best;
    double best_cost = 1e300;
    for (int S = 1; S <= kMaxSlices && S <= np; ++S) {
        const int64_t P = ceil_div(np, S);
        for (int two = 0; two <= 1; ++two) {
            const size_t limit = two ? half : kSmemOptIn;
            // the cluster count decides the partial-row buffers: ask with one
            const size_t probe = matvec_smem(M, F, static_cast<int>(P), S, kWarps, 1);
            if (probe > limit) continue;
            const int64_t cmax = matvec_max_clusters(M, F, S, probe);
            if (cmax < 1) continue;
            const int64_t clusters = std::min<int64_t>(groups, cmax);
            const int64_t tiles = ceil_div(groups, clusters);
            const int parts = tiles > 1 ? 2 : 1;
            // the whole slice in the ring when it fits (no slot is refilled;
            // any depth from 8), else the deepest multiple of 8 that fits
            const int64_t recs_cta = tiles * P;
            int ring = 0;
            if (recs_cta <= kMaxRing) {
                const int r = static_cast<int>(std::max<int64_t>(kWarps, recs_cta));
                if (matvec_smem(M, F, static_cast<int>(P), S, r, parts) <= limit) ring = r;
            }
            for (int64_t r = std::min<int64_t>(kMaxRing, recs_cta / kWarps * kWarps); r >= kWarps && ring == 0; r -= kWarps)
                if (matvec_smem(M, F, static_cast<int>(P), S, static_cast<int>(r), parts) <= limit)
                    ring = static_cast<int>(r);
            if (ring == 0) continue;
            const size_t smem = matvec_smem(M, F, static_cast<int>(P), S, ring, parts);
            if (matvec_max_clusters(M, F, S, smem) < clusters) continue;
            const bool two_fit = smem <= half;
            if (!two && two_fit) continue;             // the same plan as two = 1
            const int64_t ctas = clusters * S;
            const int per_sm = static_cast<int>(ceil_div(ctas, sm_count));
            const double recs = static_cast<double>(tiles * P);
            const double warp = static_cast<double>(ceil_div(tiles * P, kWarps)) * rc * 8.0 * per_sm / 4.0;
            const double work = std::max(warp, rw * total / sm_count);
            const double starve = recs > ring ? (recs - ring) * 0.5 : 0.0;
            const double slices = S > 1 ? 3.0 + 1.0 * (S - 2) : 0.0;
            const double groups_cost = tiles > 1 ? static_cast<double>(tiles) * (2.0 + 1.5 * S) : 0.0;
            const double no_overlap = (!two_fit || per_sm > 1) ? 30.0 : 0.0;
            const double cost = work + starve + slices + groups_cost + no_overlap;
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.M = M;
                best.fmt = fmt;
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

cudaError_t launch_matvec(const MatvecPlan &plan, const DecodeArgs &args, cudaStream_t s)
{
    const void *fn = matvec_fn(plan.M, plan.fmt == kMatvecInt8 ? kFmtW8 : kFmtQ4);
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
    ExpertSet none;
    void *kargs[] = {&a, &none};
    return launch_pdl(fn, dim3(plan.ctas), dim3(kThreads), plan.smem, s, kargs, plan.S);
}

// An expert set runs one group per cluster (a CTA stages one expert's rows
// of X), as many clusters as the set has groups; the hardware runs them in
// waves. Per S: the deepest ring that fits beside a second CTA (else one CTA
// per SM), no deeper than a slice. Cost: the waves of clusters the device
// holds at once times a slice's records, plus the slices' reduction.
bool plan_matvec_experts(int64_t m, int64_t k, int64_t n, int experts, int sm_count, MatvecPlan *plan)
{
    if (m < 1 || m > 16 || experts < 1 || experts > kMaxExpertSet || sm_count < 1) return false;
    const int M = instance_of(m);
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const size_t half = kSmemPerSM / 2 - 1024;
    MatvecPlan best;
    double best_cost = 1e300;
    for (int S = 1; S <= kMaxSlices && S <= np; ++S) {
        const int64_t P = ceil_div(np, S);
        for (int two = 1; two >= 0; --two) {
            const size_t limit = two ? half : kSmemOptIn;
            int ring = 0;
            const int exact = static_cast<int>(std::min<int64_t>(kMaxRing, std::max<int64_t>(kWarps, P)));
            if (P <= kMaxRing && matvec_smem(M, kFmtQ4, static_cast<int>(P), S, exact, 1) <= limit) ring = exact;
            for (int64_t r = std::min<int64_t>(kMaxRing, P / kWarps * kWarps); r >= kWarps && ring == 0; r -= kWarps)
                if (matvec_smem(M, kFmtQ4, static_cast<int>(P), S, static_cast<int>(r), 1) <= limit)
                    ring = static_cast<int>(r);
            if (ring == 0) continue;
            const size_t smem = matvec_smem(M, kFmtQ4, static_cast<int>(P), S, ring, 1);
            const int64_t cmax = matvec_max_clusters(M, kFmtQ4, S, smem);
            if (cmax < 1) continue;
            const int64_t clusters = groups * experts;
            const double waves = static_cast<double>(ceil_div(clusters, cmax));
            const double cost = waves * (static_cast<double>(P) + 4.0) + (S > 1 ? 2.0 : 0.0) +
                                (P > ring ? static_cast<double>(P - ring) : 0.0);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.M = M;
                best.fmt = kMatvecQ4;
                best.S = S;
                best.clusters = static_cast<int>(clusters);
                best.ctas = static_cast<int>(clusters * S);
                best.ring = ring;
                best.smem = smem;
            }
        }
    }
    if (best.ctas == 0) return false;
    *plan = best;
    return true;
}

cudaError_t launch_matvec_experts(const MatvecPlan &plan, const DecodeArgs &args, const ExpertSet &set,
                                  cudaStream_t s)
{
    const void *fn = matvec_fn(plan.M, kFmtQ4);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    DecodeArgs a = args;
    a.pass_p0 = 0;
    a.S = plan.S;
    a.pbase = args.np / plan.S;
    a.prem = args.np % plan.S;
    a.clusters = args.groups;
    a.ring = plan.ring;
    a.accumulate = 0;
    a.xs_bytes = 0;
    ExpertSet es = set;
    void *kargs[] = {&a, &es};
    return launch_pdl(fn, dim3(plan.ctas), dim3(kThreads), plan.smem, s, kargs, plan.S);
}

} // namespace q4
