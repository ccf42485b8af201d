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
// Arithmetic (m <= 4), exact up to the final scaling. X is the B operand of
// the warp-level MMA (mma.sync m16n8k16, fp16 x fp16 -> fp32). Each 32-element
// block of a token row is scaled by a power of two 2^-e (its largest |x|
// lands in [1, 2)) and split into two fixed-point terms: hi, a multiple of
// 2^-7, and lo, a multiple of 2^-15 (x - hi rounded to that grid, kept 2^8
// larger): 16 bits relative to the block's largest |x|. The A operand is a
// nibble OR'ed into the fp16 pattern of 1024: exactly 1024 + q for the low
// nibbles (k-step 0) and, left in place, 1024 + 16q for the high ones
// (k-step 1, whose X terms are divided by 16): one lop3 for two weights and
// no subtraction. The accumulator of a column starts at the correction
// -1032 (sum of its k-step-0 terms) - 1152 (sum of its k-step-1 terms), so it
// ends at sum (q - 8) * term. Every partial sum on the way is a multiple of
// 2^-7 below 2^16, so fp32 holds each one exactly and the tensor core's
// summation order cannot change the block's dot products. They are then added
// and scaled by d * 2^e in fp32 (one rounding each) into the row's fp32 total.
// All-eights weights give 0 exactly, and integer inputs stay integer-exact.
// A block of X that holds a NaN or an infinity switches the CTA to exact
// weights (q - 8, one subtraction more per two weights) with a zero starting
// accumulator, so that infinities meet (q - 8) and d as IEEE arithmetic says;
// the finite blocks' results are the same bits either way.
//
// Arithmetic (m >= 8), where the MMA count per weight grows with the tokens:
// one fp16 term per element, x 2^-e with the block's 2^e taken over all the
// CTA's tokens (relative error at most 2^-11, half the decode bound of 1e-3
// of sum |x w|), against exact weights q - 8 and 16 (q - 8) with a zero
// start; the products are exact and the block's sums are fp32 sums.
//
// MMA columns. For m <= 4 the hi and lo terms of a (token, block) are two
// columns of the 8, and the 8 columns hold up to four (token, block) pairs:
// m = 1 puts a record's two blocks side by side in one accumulator tile
// (thread t of a quad holds block t), m = 2 the two blocks of two tokens, m = 4
// one block of four tokens. The weights of a 16 x 16 tile are dequantised once
// for all of them. For m = 5..16 the columns are tokens, eight per tile.
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
// order) and the ring slots they pass through: lane 0 refills a slot with
// 1-D bulk copies of the record R places ahead as soon as the warp has read
// it, so every barrier has one waiter and no copy is in flight when the CTA
// exits; with weights declared read-only the first R records stream before
// the dependency wait. A warp takes a record's eight row tiles at once, which
// gives the scheduler eight independent streams of loads, dequantisation and
// MMAs. For m >= 8 the items are half records instead (rows 0-63 for warps
// 0-3, rows 64-127 for warps 4-7, each half its own sequence dealt to its
// four warps), which halves the registers and shared memory a warp's partial
// rows take. At the end of a group each warp leaves its partial rows in
// shared memory; one group later warp c sums rows 16c .. 16c + 15 of the
// partials in order, then the cluster's slices of them, and writes Y. Every
// wait is bounded and warp-uniform.
#include <algorithm>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5;                   // Q4_ERR_DEVICE_TIMEOUT
// After a wait gave up, the waits for what is still landing in this CTA's
// shared memory (its bulk copies, the other slices' stores) are bounded by
// at least this, whatever the caller's limit: those transfers are already
// issued and end in microseconds, and the CTA must not exit before them.
constexpr uint64_t kDrainNs = 200000000ull;
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kSliceRows = kGroupRows / kWarps;  // rows of a group each warp finishes
constexpr int kMaxSlices = 8;
constexpr int kMaxRing = 32;                     // records; a multiple of kWarps when slots are refilled

// m >= 8 streams half records: a warp takes rows 0-63 or 64-127 of its
// records (warps 0-3 and 4-7), so that its partial rows cover 64 rows.
__host__ __device__ constexpr int halves(int M) { return M >= 8 ? 2 : 1; }
__host__ __device__ constexpr int item_tiles(int M) { return 8 / halves(M); }   // 16-row tiles of an item
__host__ __device__ constexpr int item_rows(int M) { return kGroupRows / halves(M); }
// B entries per (record, block): one for m <= 4 (hi and lo are columns), one
// per eight tokens otherwise (a single fp16 term).
__host__ __device__ constexpr int entries_per_block(int M) { return M <= 4 ? 1 : M / 8; }
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
// A ring slot holds one item: a record, or half of one (Q4_0: the half's
// scales, block-0 and block-1 nibbles at 0, 256 and 1280; int8: its 64 rows).
__host__ __device__ constexpr int slot_bytes(int M, int F) { return rec_bytes(F) / halves(M); }
constexpr int kHalfQs0Off = 256;
constexpr int kHalfQs1Off = 1280;
__host__ __device__ constexpr int max_ring(int M) { return kMaxRing * halves(M); }
// int8 records: B entries per record (hi and lo columns for m <= 4; a hi and a
// lo entry per eight tokens otherwise), each 32 lanes x 32 bytes (four k-steps)
__host__ __device__ constexpr int w8_entries(int M) { return M <= 4 ? 1 : 2 * (M / 8); }
// Shared-memory bytes per record of the CTA's slice: X fragments, parameters.
__host__ __device__ constexpr int xfrag_bytes(int M, int F)
{
    return F == kFmtW8 ? w8_entries(M) * 1024 : 2 * entries_per_block(M) * entry_bytes(M);
}
__host__ __device__ constexpr int xparam_bytes(int M, int F) { return F == kFmtW8 ? M * 4 : M <= 4 ? 2 * M * 16 : 8; }
// The parameter region of a slice, rounded up so that what follows it (row
// buffers, barriers) stays 16-byte aligned.
__host__ __device__ constexpr int xparam_region(int M, int F, int Pmax) { return (Pmax * xparam_bytes(M, F) + 15) / 16 * 16; }
// Accumulators per row of a thread: one (m <= 4), or two tokens per eight.
__host__ __device__ constexpr int acc_width(int M) { return M <= 4 ? 1 : M / 4; }

struct VSmem {
    uint8_t *ring;        // [R] slots of slot_bytes (R / halves per half of the warps)
    int rh;               // slots per half of the warps
    uint4 *bimg;          // [Pmax] x xfrag_bytes: B fragments of X (Q4_0: [2][NQ][entry_lanes];
                          // int8: [entries][32 lanes][2])
    float4 *xp;           // Q4_0, M <= 4: [Pmax][2][M] {hi and lo columns' corrections, 2^e, 0}
    float *xs;            // Q4_0, M >= 8: [Pmax][2] 2^e of a block; int8: [Pmax][M] 2^e
    float *part;          // [NB][8][M][item_rows] the warps' partial rows of a group
    bool part_in_ring;    // single-group grids with the whole slice in the ring: warp c's
                          // partial rows sit in its first ring slot instead
    int part_stride;      // floats from one warp's partial rows to the next's
    float *red;           // [NR][S - 1][M][128] other slices' rows of a group (first CTA)
    int *flag;            // a staged block of X was not finite
    uint64_t *full;                   // [R]
    uint64_t *gfull, *gfree;          // [2] partials of a group parity written / summed
    uint64_t *red_full, *red_free;    // [2][8] a row slice's other slices landed / slot free
    uint64_t *red_tx;                 // single-group grids: the other slices' rows landed
};

// f(integral_constant<int, i>) for i = 0 .. N - 1, each a compile-time index
// (shared-memory offsets that depend on it fold into the loads).
template <typename Fn, int... I>
__device__ __forceinline__ void static_for_impl(Fn &&f, std::integer_sequence<int, I...>)
{
    (f(std::integral_constant<int, I>{}), ...);
}
template <int N, typename Fn>
__device__ __forceinline__ void static_for(Fn &&f)
{
    static_for_impl(f, std::make_integer_sequence<int, N>{});
}

__device__ __forceinline__ void fail(const DecodeArgs &a) { record_status(a.status, kErrTimeout); }

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait(bar, parity, limit_ns)) != 0;
}
__device__ __forceinline__ bool warp_wait_cluster(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    return __all_sync(0xFFFFFFFFu, mbar_wait_cluster(bar, parity, limit_ns)) != 0;
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
// The same at a compile-time byte offset from `addr` (folded into the load).
template <int OFF>
__device__ __forceinline__ uint32_t ld32o(uint32_t addr)
{
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1+%2];" : "=r"(v) : "r"(addr), "n"(OFF));
    return v;
}
template <int OFF>
__device__ __forceinline__ uint4 ld128o(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4+%5];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr), "n"(OFF));
    return v;
}
__device__ __forceinline__ float2 ld64f(uint32_t addr)
{
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}

// D += A * B, m16n8k16, fp16 operands, fp32 accumulate in place (exact fp16
// weights times X's fp16 terms). Volatile, so that an item's MMAs, which
// consume its shared-memory loads, are issued before its slot is refilled.
__device__ __forceinline__ void mma_acc_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// D = A * B + C, m16n8k16, fp16 operands, fp32 accumulate, C left as it is
// (a start shared by many tiles).
__device__ __forceinline__ void mma_f16_c(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1,
                                          const float (&c)[4])
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(c[0]), "f"(c[1]), "f"(c[2]),
                   "f"(c[3]));
}

// D = A * B, m16n8k16, fp16 operands, fp32 result from a zero start.
__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
                 : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

// (y0, y1) += (v0, v1) * s as one packed fp32 operation (each lane one
// rounding, as two fmaf).
__device__ __forceinline__ void fma2(float &y0, float &y1, float v0, float v1, float s)
{
    asm("{\n\t.reg .b64 y, v, s;\n\t"
        "mov.b64 y, {%0, %1};\n\tmov.b64 v, {%2, %3};\n\tmov.b64 s, {%4, %4};\n\t"
        "fma.rn.f32x2 y, v, s, y;\n\tmov.b64 {%0, %1}, y;\n\t}"
        : "+f"(y0), "+f"(y1)
        : "f"(v0), "f"(v1), "f"(s));
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
// Arrive with release semantics: this CTA's writes so far (its barriers'
// initialisation) are visible to the cluster once the others have waited.
__device__ __forceinline__ void cluster_arrive_release()
{
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}

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
// low half, block 1 in the high half), at a bit offset sh of 0 or 16.
__device__ __forceinline__ float half_at(uint32_t w, int sh)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> sh)));
}
// The same for a block given as 0 or 1.
__device__ __forceinline__ float half_of(uint32_t w, int hi)
{
    return __half2float(__ushort_as_half(static_cast<unsigned short>(hi ? (w >> 16) : (w & 0xFFFFu))));
}

// The eight weights of one word of split-half nibbles (bytes 4t .. 4t+3 of a
// block's qs) as fp16 pairs, the low nibbles for k-step 0
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

// m <= 4: stage the CTA's slice of X (pairs p0 .. p0 + P - 1) as B
// fragments. A task is one (pair, block, token): four lanes of a warp
// (t = 0..3) hold its 32 values, eight each (elements 4t .. 4t+3 and
// 16 + 4t .. 19 + 4t), agree on its scale by two shuffles, split them into hi
// and lo and store them where the consumer lanes read them: entry (p, b),
// column pair c (c = b for m = 1, 2b + token for m = 2, token for m = 4): hi
// at lane 4 (2c) + t, lo at lane 4 (2c + 1) + t (for m <= 2 the entry stores
// only the block's own lanes). A fragment register holds, for k-step 0,
// elements (4t, 4t+2) and (4t+1, 4t+3); for k-step 1, the same elements plus
// 16, divided by 16.
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
                if (!q4_check(xrow >= 0, a.status)) continue;
                const float *xr = a.X + static_cast<int64_t>(xrow) * a.ldx + 32 * blk + 4 * t;
                xa[i] = __ldg(reinterpret_cast<const float4 *>(xr));
                xb[i] = __ldg(reinterpret_cast<const float4 *>(xr + 16));
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            if (e0 + 8 * kWarps * i >= E) break;    // warp-uniform: none of the warp's tasks is left
            const int e = e0 + 8 * kWarps * i + q;
            const int tok = e % M, pb = e / M;
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
            // lo is kept scaled by 2^8 (on the same 2^-7 grid as hi); the
            // high-nibble half of the block (elements 16..31, k-step 1) is
            // divided by 16 to meet weights of 1024 + 16q
            constexpr float kLoScale = 256.0f;
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
                if (j >= 4) hi[j] *= 0.0625f, lo[j] *= 0.0625f;
            }
            uint4 *ent = sm.bimg + static_cast<size_t>(pb * kNQ) * entry_lanes(M);
            const float su = __uint_as_float(static_cast<unsigned>(127 + ex) << 23);   // 2^ex
            {
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
                    // (k-step 1) carries 1032 x or 72 x = 1152 (x / 16) beyond
                    // (q - 8) x; each column's correction, a multiple of 2^-4
                    // below 2^16, is exact
                    sm.xp[pb * M + tok] = fin ? make_float4(-1032.0f * s0h - 1152.0f * s1h,
                                                            -1032.0f * s0l - 1152.0f * s1l, su, 0.f)
                                              : make_float4(0.f, 0.f, su, 0.f);
                }
            }
            if (!fin && t == 0) *reinterpret_cast<volatile int *>(sm.flag) = 1;
        }
    }
}

// m >= 8: stage the CTA's slice of X as one fp16 term per element. A task is
// one block of the slice for all tokens: lane 4 j + t holds token 8h + j's
// elements 4t .. 4t+3 and 16 + 4t .. 19 + 4t, for each h. The warp agrees on
// the block's scale 2^e, from the largest finite |x| of any token (it lands
// in [1, 2)), and stores x * 2^-e rounded to fp16 (k-step 0: elements
// (4t, 4t+2), (4t+1, 4t+3); k-step 1: those plus 16, divided by 16 to meet
// weights of 16 (q - 8)) at lane 4 j + t of entry (p, b, h), which is the
// lane that reads it. Every element keeps 11 significant bits (relative error
// at most 2^-11) unless it lies 2^14 below the block's largest, and NaN and
// infinity pass unchanged.
template <int M>
__device__ __forceinline__ void stage_x_wide(const DecodeArgs &a, const VSmem &sm, int p0, int P, int w, int lane)
{
    constexpr int H = M / 8;
    constexpr int kBatch = 64 / M;                  // blocks per warp whose loads are in flight together
    const int j = lane >> 2, t = lane & 3;
    const int E = 2 * P;                            // blocks of the slice
    int xrow[H];
#pragma unroll
    for (int h = 0; h < H; ++h) {
        const int tok = 8 * h + j;
        xrow[h] = tok < a.m ? (a.rows ? __ldg(a.rows + tok) : tok) : -1;
        if (tok < a.m && !q4_check(xrow[h] >= 0, a.status)) xrow[h] = -1;
    }
    for (int e0 = w; e0 < E; e0 += kWarps * kBatch) {
        float4 xa[kBatch][H], xb[kBatch][H];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int blk = 2 * p0 + e0 + kWarps * i;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                xa[i][h] = make_float4(0.f, 0.f, 0.f, 0.f);
                xb[i][h] = xa[i][h];
                if (e0 + kWarps * i < E && blk < a.nb && xrow[h] >= 0) {
                    const float *xr = a.X + static_cast<int64_t>(xrow[h]) * a.ldx + 32 * blk + 4 * t;
                    xa[i][h] = __ldg(reinterpret_cast<const float4 *>(xr));
                    xb[i][h] = __ldg(reinterpret_cast<const float4 *>(xr + 16));
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
            const int pb = e0 + kWarps * i;         // 2p + b within the slice
            if (pb >= E) break;                     // warp-uniform
            unsigned mb = 0u;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                const float v[8] = {xa[i][h].x, xa[i][h].y, xa[i][h].z, xa[i][h].w,
                                    xb[i][h].x, xb[i][h].y, xb[i][h].z, xb[i][h].w};
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const unsigned bits = __float_as_uint(v[q]) & 0x7FFFFFFFu;
                    if (bits < 0x7F800000u) mb = max(mb, bits);
                }
            }
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
            int ex = 0;                             // largest finite |x| in [2^ex, 2^(ex + 1))
            if (mb >= 0x00800000u) ex = min(static_cast<int>(mb >> 23) - 127, 126);
            else if (mb != 0u) ex = -126;           // subnormal: scaled below 1
            const float sd = __uint_as_float(static_cast<unsigned>(127 - ex) << 23);   // 2^-ex
            const float sd16 = sd * 0.0625f;
            uint4 *ent = sm.bimg + static_cast<size_t>(pb * H) * 32;
#pragma unroll
            for (int h = 0; h < H; ++h) {
                uint4 f;
                f.x = pack_half2_rn(xa[i][h].x * sd, xa[i][h].z * sd);
                f.y = pack_half2_rn(xa[i][h].y * sd, xa[i][h].w * sd);
                f.z = pack_half2_rn(xb[i][h].x * sd16, xb[i][h].z * sd16);
                f.w = pack_half2_rn(xb[i][h].y * sd16, xb[i][h].w * sd16);
                ent[h * 32 + lane] = f;
            }
            if (lane == 0) sm.xs[pb] = __uint_as_float(static_cast<unsigned>(127 + ex) << 23);   // 2^ex
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
                if (!q4_check(xrow >= 0, a.status)) continue;
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

// One item (a record; for m >= 8 half of one) for all its row tiles:
// y[rt][r][i] += the part of the item's row 16 rt + g + 8r for the token (and
// block, m <= 2) thread t holds:
//   m = 1:  token 0, block t of the record (t < 2; summed over t at the end);
//   m = 2:  token t & 1, block t >> 1 (summed over t, t ^ 2 at the end);
//   m = 4:  token t;
//   m = 8:  token 2t + i;
//   m = 16: token 8 (i >> 1) + 2t + (i & 1).
// `p` is the record's pair within the slice (its X entries).
template <int M, bool EXACT>
__device__ __forceinline__ void record_mma(const VSmem &sm, uint32_t rec, int p, int lane,
                                           float (&y)[item_tiles(M)][2][acc_width(M)])
{
    constexpr int kNQ = entries_per_block(M);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bimg = smem_u32(sm.bimg) + static_cast<uint32_t>(p * 2 * kNQ * entry_bytes(M) + lane * 16);
    // this lane's words of row g (nibbles) and its scale word; row tiles and
    // the rows + 8 are compile-time offsets from these
    const uint32_t bq = rec + static_cast<uint32_t>(16 * g + 4 * t), bs = rec + static_cast<uint32_t>(4 * g);
    if constexpr (M <= 2) {
        // one accumulator tile for both blocks: lanes outside a block's own
        // columns take zeros for its MMAs
        constexpr int SH = M == 1 ? 3 : 4;          // block of the columns of lane (g, t)
        const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
        const uint32_t bl = smem_u32(sm.bimg) +
                            static_cast<uint32_t>((p * 2 + (lane >> SH)) * entry_bytes(M) + (lane & (entry_lanes(M) - 1)) * 16);
        const uint4 B0 = (lane >> SH) == 0 ? ld128(bl) : zero;
        const uint4 B1 = (lane >> SH) == 1 ? ld128(bl) : zero;
        // this thread's (block, token) column pair: corrections and 2^e (for
        // m = 1, lanes t = 2, 3 hold columns without X and are never stored;
        // they read block t & 1's)
        const int bt = M == 1 ? (t & 1) : (t >> 1);
        const float4 cr = ld128f(smem_u32(sm.xp + (p * 2 + bt) * M + (M == 1 ? 0 : (t & 1))));
        const float su = cr.z;
        const int sh = 16 * bt;                     // the block's half of a scale word
        const float cq[4] = {EXACT ? 0.f : cr.x, EXACT ? 0.f : cr.y, EXACT ? 0.f : cr.x, EXACT ? 0.f : cr.y};
        static_for<8>([&](auto RT) {
            constexpr int rt = decltype(RT)::value;
            const uint32_t w00 = ld32o<kRecQs0Off + 256 * rt>(bq), w01 = ld32o<kRecQs0Off + 256 * rt + 128>(bq);
            const uint32_t w10 = ld32o<kRecQs1Off + 256 * rt>(bq), w11 = ld32o<kRecQs1Off + 256 * rt + 128>(bq);
            const uint32_t s0 = ld32o<kRecScaleOff + 64 * rt>(bs), s1 = ld32o<kRecScaleOff + 64 * rt + 32>(bs);
            uint32_t a[2][2][4];                    // [block][k-step][fragment]
            weights_f16<EXACT>(w00, a[0][0][0], a[0][0][2], a[0][1][0], a[0][1][2]);
            weights_f16<EXACT>(w01, a[0][0][1], a[0][0][3], a[0][1][1], a[0][1][3]);
            weights_f16<EXACT>(w10, a[1][0][0], a[1][0][2], a[1][1][0], a[1][1][2]);
            weights_f16<EXACT>(w11, a[1][0][1], a[1][0][3], a[1][1][1], a[1][1][3]);
            // both k-steps of both blocks into one tile, from the columns'
            // corrections
            float D[4];
            mma_f16_c(D, a[0][0], B0.x, B0.y, cq);
            mma_acc_f16(D, a[1][0], B1.x, B1.y);
            mma_acc_f16(D, a[0][1], B0.z, B0.w);
            mma_acc_f16(D, a[1][1], B1.z, B1.w);
            const float d0 = half_at(s0, sh), d1 = half_at(s1, sh);
            // hi column + lo column (kept 2^8 larger)
            y[rt][0][0] = fmaf(d0 * su, fmaf(D[1], 0x1p-8f, D[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(d1 * su, fmaf(D[3], 0x1p-8f, D[2]), y[rt][1][0]);
        });
    } else if constexpr (M == 4) {
        // a tile per block: thread t holds token t
        const uint4 B0 = ld128(bimg), B1 = ld128(bimg + 512);
        const float4 c0 = ld128f(smem_u32(sm.xp + p * 2 * 4 + t));
        const float4 c1 = ld128f(smem_u32(sm.xp + (p * 2 + 1) * 4 + t));
        const float su0 = c0.z, su1 = c1.z;
        const float cq0[4] = {EXACT ? 0.f : c0.x, EXACT ? 0.f : c0.y, EXACT ? 0.f : c0.x, EXACT ? 0.f : c0.y};
        const float cq1[4] = {EXACT ? 0.f : c1.x, EXACT ? 0.f : c1.y, EXACT ? 0.f : c1.x, EXACT ? 0.f : c1.y};
        static_for<8>([&](auto RT) {
            constexpr int rt = decltype(RT)::value;
            const uint32_t w00 = ld32o<kRecQs0Off + 256 * rt>(bq), w01 = ld32o<kRecQs0Off + 256 * rt + 128>(bq);
            const uint32_t w10 = ld32o<kRecQs1Off + 256 * rt>(bq), w11 = ld32o<kRecQs1Off + 256 * rt + 128>(bq);
            const uint32_t s0 = ld32o<kRecScaleOff + 64 * rt>(bs), s1 = ld32o<kRecScaleOff + 64 * rt + 32>(bs);
            uint32_t a[2][2][4];
            weights_f16<EXACT>(w00, a[0][0][0], a[0][0][2], a[0][1][0], a[0][1][2]);
            weights_f16<EXACT>(w01, a[0][0][1], a[0][0][3], a[0][1][1], a[0][1][3]);
            weights_f16<EXACT>(w10, a[1][0][0], a[1][0][2], a[1][1][0], a[1][1][2]);
            weights_f16<EXACT>(w11, a[1][0][1], a[1][0][3], a[1][1][1], a[1][1][3]);
            float D0[4], D1[4];
            mma_f16_c(D0, a[0][0], B0.x, B0.y, cq0);
            mma_f16_c(D1, a[1][0], B1.x, B1.y, cq1);
            mma_acc_f16(D0, a[0][1], B0.z, B0.w);
            mma_acc_f16(D1, a[1][1], B1.z, B1.w);
            y[rt][0][0] = fmaf(half_of(s0, 0) * su0, fmaf(D0[1], 0x1p-8f, D0[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(half_of(s1, 0) * su0, fmaf(D0[3], 0x1p-8f, D0[2]), y[rt][1][0]);
            y[rt][0][0] = fmaf(half_of(s0, 1) * su1, fmaf(D1[1], 0x1p-8f, D1[0]), y[rt][0][0]);
            y[rt][1][0] = fmaf(half_of(s1, 1) * su1, fmaf(D1[3], 0x1p-8f, D1[2]), y[rt][1][0]);
        });
    } else {
        // a half record (64 rows, scales and nibbles at 0, 256 and 1280);
        // tiles (block b, tokens 8h .. 8h + 7): exact weights q - 8 (k-step 0)
        // and 16 (q - 8) (k-step 1) against the block's single fp16 term
        constexpr int H = M / 8;
        uint4 B[2][H];
#pragma unroll
        for (int b = 0; b < 2; ++b)
#pragma unroll
            for (int h = 0; h < H; ++h) B[b][h] = ld128(bimg + static_cast<uint32_t>((b * H + h) * 512));
        const float2 su = ld64f(smem_u32(sm.xs + 2 * p));   // 2^e of blocks 0 and 1
        static_for<item_tiles(M)>([&](auto RT) {
            constexpr int rt = decltype(RT)::value;
            const uint32_t w00 = ld32o<kHalfQs0Off + 256 * rt>(bq), w01 = ld32o<kHalfQs0Off + 256 * rt + 128>(bq);
            const uint32_t w10 = ld32o<kHalfQs1Off + 256 * rt>(bq), w11 = ld32o<kHalfQs1Off + 256 * rt + 128>(bq);
            const uint32_t s0 = ld32o<64 * rt>(bs), s1 = ld32o<64 * rt + 32>(bs);
            uint32_t a[2][2][4];
            weights_f16<true>(w00, a[0][0][0], a[0][0][2], a[0][1][0], a[0][1][2]);
            weights_f16<true>(w01, a[0][0][1], a[0][0][3], a[0][1][1], a[0][1][3]);
            weights_f16<true>(w10, a[1][0][0], a[1][0][2], a[1][1][0], a[1][1][2]);
            weights_f16<true>(w11, a[1][0][1], a[1][0][3], a[1][1][1], a[1][1][3]);
#pragma unroll
            for (int b = 0; b < 2; ++b) {
                const float sb = b ? su.y : su.x;
                const float ds0 = half_of(s0, b) * sb, ds1 = half_of(s1, b) * sb;
#pragma unroll
                for (int h = 0; h < H; ++h) {
                    float D[4];
                    mma_f16(D, a[b][0], B[b][h].x, B[b][h].y);
                    mma_acc_f16(D, a[b][1], B[b][h].z, B[b][h].w);
                    fma2(y[rt][0][2 * h], y[rt][0][2 * h + 1], D[0], D[1], ds0);
                    fma2(y[rt][1][2 * h], y[rt][1][2 * h + 1], D[2], D[3], ds1);
                }
            }
        });
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

// One int8 item (a record; for m >= 8 its 64-row half) for all its row tiles:
// y[rt][r][i] += 2^-e * (row's
// codes . X's pair), for the token thread t holds (m <= 4: token t; m = 8:
// 2t + i; m = 16: 8 (i >> 1) + 2t + (i & 1)); the row's scale comes when Y is
// written.
template <int M>
__device__ __forceinline__ void record_mma_w8(const VSmem &sm, uint32_t rec, int p, int lane,
                                              float (&y)[item_tiles(M)][2][acc_width(M)])
{
    constexpr int kNE = w8_entries(M);
    const int g = lane >> 2, t = lane & 3;
    const uint32_t bimg = smem_u32(sm.bimg) + static_cast<uint32_t>(p * xfrag_bytes(M, kFmtW8) + lane * 32);
    const uint32_t bq = rec + static_cast<uint32_t>(kPairK * g + 16 * t);   // row g's 16 codes of this lane
    if constexpr (M <= 4) {
        const uint4 e0 = ld128(bimg), e1 = ld128(bimg + 16);
        const float su = t < M ? sm.xs[p * M + t] : 0.f;
        static_for<item_tiles(M)>([&](auto RT) {
            constexpr int rt = decltype(RT)::value;
            const uint4 qa = ld128o<1024 * rt>(bq), qb = ld128o<1024 * rt + 512>(bq);
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
        });
    } else {
        constexpr int H = M / 8;
        float2 su[H];
#pragma unroll
        for (int h = 0; h < H; ++h) su[h] = ld64f(smem_u32(sm.xs + p * M + 8 * h + 2 * t));
        static_for<item_tiles(M)>([&](auto RT) {
            constexpr int rt = decltype(RT)::value;
            const uint4 qa = ld128o<1024 * rt>(bq), qb = ld128o<1024 * rt + 512>(bq);
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
        });
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

// This warp's partial rows of buffer tb.
__device__ __forceinline__ float *part_of(const VSmem &sm, int tb, int c, int M)
{
    if (sm.part_in_ring) {
        // the warp's first ring slot
        const int first = halves(M) == 2 ? (c >> 2) * sm.rh + (c & 3) : c;
        return sm.part + static_cast<size_t>(first) * sm.part_stride;
    }
    return sm.part + static_cast<size_t>(tb * kWarps + c) * sm.part_stride;
}

// Store this warp's partial rows of a group (the item rows of its half,
// [M][item_rows] floats) into buffer tb.
template <int M>
__device__ __forceinline__ void store_partials(const VSmem &sm, int tb, int c, int lane,
                                               float (&y)[item_tiles(M)][2][acc_width(M)])
{
    constexpr int NY = acc_width(M);
    constexpr int RI = item_rows(M);
    const int g = lane >> 2, t = lane & 3;
    // m = 1: blocks 0 and 1 of a row sit in threads t = 0, 1; m = 2: blocks
    // 0 and 1 of a token in threads t and t ^ 2
#pragma unroll
    for (int rt = 0; rt < item_tiles(M); ++rt)
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            if constexpr (M == 1) y[rt][r][0] += __shfl_xor_sync(0xFFFFFFFFu, y[rt][r][0], 1);
            if constexpr (M == 2) y[rt][r][0] += __shfl_xor_sync(0xFFFFFFFFu, y[rt][r][0], 2);
        }
    const bool writes = M == 1 ? t == 0 : (M == 2 ? t < 2 : true);
    float *pp = part_of(sm, tb, c, M);
    if (writes)
#pragma unroll
        for (int rt = 0; rt < item_tiles(M); ++rt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < NY; ++i) pp[acc_token<M>(t, i) * RI + 16 * rt + g + 8 * r] = y[rt][r][i];
}

// Rows of a warp's slice in the reduction: lane l handles row 16c + (l & 15)
// and tokens l / 16, + 2, ...
template <int M>
struct SliceRows {
    static constexpr int NT = (M + 1) / 2;
    float v[NT];
};

// Sum the partials of a group (buffer tb) for this warp's rows, in warp
// order: the eight warps' (m <= 4), or the four warps' of this half (m >= 8).
template <int M>
__device__ __forceinline__ void sum_partials(const VSmem &sm, int tb, int c, int lane, SliceRows<M> &s)
{
    constexpr int RI = item_rows(M);
    constexpr int NW = kWarps / halves(M);
    const int row = (c * kSliceRows) % RI + (lane & (kSliceRows - 1));   // within the half
    const int w0 = halves(M) == 2 ? (c >> 2) * NW : 0;
    const int t0 = lane >> 4;
#pragma unroll
    for (int h = 0; h < SliceRows<M>::NT; ++h) {
        const int tok = t0 + 2 * h;
        float v = 0.0f;
        if (tok < M)
#pragma unroll
            for (int w = 0; w < NW; ++w) v += part_of(sm, tb, w0 + w, M)[tok * RI + row];
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
            if (q4_check(yr >= 0, a.status)) a.Y[static_cast<int64_t>(yr) * a.ldy + grow] = v;
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

// Issue the copy of the item of group gi, pair j of the CTA's slice (the
// whole record, or rows 64 hf .. 64 hf + 63 of it) into ring slot s. Lane 0
// of the slot's warp only.
template <int M, int F>
__device__ __forceinline__ void load_item(const DecodeArgs &a, const VSmem &sm, int gi, int j, int hf, int s, int G0,
                                          int p0, uint64_t pol)
{
    constexpr int kRB = rec_bytes(F), kSB = slot_bytes(M, F);
    // (checked build: a record outside the layer or a slot outside the ring
    // is not copied; a slot's barrier still completes, without data)
    if (!q4_check(G0 + gi * a.clusters < a.groups && j >= 0 && p0 + j < a.np && s >= 0 && s < a.ring, a.status)) {
        if (s >= 0 && s < a.ring) mbar_arrive(&sm.full[s]);
        return;
    }
    const int64_t rec = static_cast<int64_t>(G0 + gi * a.clusters) * a.np + p0 + j;
    const uint8_t *src = a.W + rec * kRB;
    uint8_t *dst = sm.ring + static_cast<size_t>(s) * kSB;
    mbar_arrive_expect_tx(&sm.full[s], kSB);
    if constexpr (halves(M) == 1) {
        bulk_g2s_hint(dst, src, kRB, &sm.full[s], pol);
    } else if constexpr (F == kFmtW8) {
        bulk_g2s_hint(dst, src + hf * kSB, kSB, &sm.full[s], pol);
    } else {
        // the half's scales and the nibbles of its rows in either block
        bulk_g2s_hint(dst, src + kRecScaleOff + 256 * hf, 256, &sm.full[s], pol);
        bulk_g2s_hint(dst + kHalfQs0Off, src + kRecQs0Off + 1024 * hf, 1024, &sm.full[s], pol);
        bulk_g2s_hint(dst + kHalfQs1Off, src + kRecQs1Off + 1024 * hf, 1024, &sm.full[s], pol);
    }
}

// The warp's items, group by group: products into registers, partial rows
// into shared memory at each group's end, the previous group's reduction.
// Warp c takes items c, c + 8, ... of the CTA's sequence (m >= 8: warp c of
// half c / 4 takes items c % 4, c % 4 + 4, ... of that half's sequence) and
// their ring slots. `pending` tracks the warp's first item not yet read (for
// the drain after a failure).
template <int M, bool EXACT, int F>
__device__ __forceinline__ bool consume(const DecodeArgs &a, const VSmem &sm, int c, int lane, int rank, int G0, int p0,
                                        int P, int ntiles, bool merged, uint64_t pol, int &pending,
                                        SliceRows<M> &keep)
{
    constexpr int NY = acc_width(M), KT = item_tiles(M), NS = kWarps / halves(M);
    const int hf = c / NS, cs = c % NS;
    const int RH = sm.rh;
    const int total = ntiles * P;
    const uint32_t ring0 = smem_u32(sm.ring);
    int n = cs;                                       // the warp's next item
    int sl = cs, ph = 0;                              // its slot within the half's ring, the slot's parity
    int fg = (cs + RH) / P, fj = cs + RH - fg * P;    // group and pair of the item RH ahead (the refill)
    for (int g = 0; g < ntiles; ++g) {
        float y[KT][2][NY];
#pragma unroll
        for (int rt = 0; rt < KT; ++rt)
#pragma unroll
            for (int r = 0; r < 2; ++r)
#pragma unroll
                for (int i = 0; i < NY; ++i) y[rt][r][i] = 0.f;
        for (; n < (g + 1) * P; n += NS) {
            const int s = hf * RH + sl;
            if (!warp_wait(&sm.full[s], static_cast<uint32_t>(ph), a.wait_ns)) return false;
            const uint32_t rec = ring0 + static_cast<uint32_t>(s * slot_bytes(M, F));
            if constexpr (F == kFmtW8) record_mma_w8<M>(sm, rec, n - g * P, lane, y);
            else record_mma<M, EXACT>(sm, rec, n - g * P, lane, y);
            // the item's MMAs, which consume its loads, are issued: refill
            // the slot with the item RH places ahead (same warp)
            __syncwarp();
            if (lane == 0 && n + RH < total) load_item<M, F>(a, sm, fg, fj, hf, s, G0, p0, pol);
            pending = n + NS;
            for (fj += NS; fj >= P; fj -= P) ++fg;
            sl += NS;
            if (sl >= RH) sl -= RH, ph ^= 1;
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
    constexpr int kSB = slot_bytes(M, F);
    constexpr int NS = kWarps / halves(M);
    extern __shared__ __align__(128) uint8_t smem_raw[];
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
    const int total = ntiles * P;                   // items of each half's sequence
    const int R = a.ring;
    // Every CTA of the cluster lays out its shared memory for the largest
    // slice, so that a barrier or a row buffer sits at the same offset in all
    // of them (remote accesses map this CTA's offsets onto another CTA's).
    const int Pmax = a.pbase + (a.prem > 0 ? 1 : 0);
    const bool merged = S > 1 && a.groups <= a.clusters;   // every CTA has a single group
    const int NB = a.groups > a.clusters ? 2 : 1;          // partial-row buffers

    VSmem sm;
    sm.ring = smem_raw;
    sm.rh = R / halves(M);
    sm.bimg = reinterpret_cast<uint4 *>(sm.ring + static_cast<size_t>(R) * kSB);
    uint8_t *after_b = sm.ring + static_cast<size_t>(R) * kSB + static_cast<size_t>(Pmax) * xfrag_bytes(M, F);
    sm.xp = reinterpret_cast<float4 *>(after_b);
    sm.xs = reinterpret_cast<float *>(after_b);
    float *after_x = reinterpret_cast<float *>(after_b + xparam_region(M, F, Pmax));
    // With a single group per CTA and the whole slice in the ring (no slot is
    // refilled), warp c's partial rows go into its first ring slot, which it
    // has read by then.
    const bool part_in_ring =
        a.groups <= a.clusters && sm.rh >= Pmax && sm.rh >= NS && M * item_rows(M) * 4 <= kSB;
    sm.part_in_ring = part_in_ring;
    sm.part = part_in_ring ? reinterpret_cast<float *>(sm.ring) : after_x;
    sm.red = after_x + (part_in_ring ? 0 : static_cast<size_t>(NB) * kWarps * M * item_rows(M));
    sm.part_stride = part_in_ring ? kSB / 4 : M * item_rows(M);
    const int red_floats = S > 1 ? (merged ? 1 : 2) * (S - 1) * M * kGroupRows : 0;
    sm.flag = reinterpret_cast<int *>(sm.red + red_floats);
    sm.full = reinterpret_cast<uint64_t *>(sm.flag + 4);
    sm.gfull = sm.full + R;
    sm.gfree = sm.gfull + 2;
    sm.red_full = sm.gfree + 2;
    sm.red_free = sm.red_full + 2 * kWarps;
    sm.red_tx = sm.red_free + 2 * kWarps;

#ifdef Q4MM_CHECKED
    {
        // the layout must end inside the launch's dynamic shared memory (the
        // same for every CTA of the grid: all return together, before any
        // barrier or copy)
        uint32_t dyn;
        asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
        const size_t used = static_cast<size_t>(reinterpret_cast<uint8_t *>(sm.red_tx + 1) - smem_raw);
        if (!q4_check(used <= dyn && R <= max_ring(M) && R >= kWarps / halves(M) * halves(M), a.status)) return;
    }
#endif
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
    // every CTA's barriers are initialised before any remote access: the
    // cluster barrier's arrive here, its wait after X is staged (no remote
    // access comes before that), so that its latency hides behind the
    // staging
    if (S > 1) cluster_arrive_release();

    // Weights may stream before the preceding kernel has finished only when
    // the caller declared them read-only.
    const uint64_t pol = policy_evict_first();
    if (!a.prefetch_w) pdl_wait();
    if (lane == 0)
        for (int n = c % NS; n < sm.rh && n < total; n += NS)
            load_item<M, F>(a, sm, n / P, n % P, c / NS, (c / NS) * sm.rh + n, G0, p0, pol);
    __syncwarp();
    pdl_wait();                                       // X, Y and the slot rows are the preceding kernel's
    if constexpr (F == kFmtW8) stage_x_w8<M>(a, sm, p0, P, c, lane);
    else if constexpr (M >= 8) stage_x_wide<M>(a, sm, p0, P, c, lane);
    else stage_x<M>(a, sm, p0, P, c, lane);
    __syncthreads();
    if (S > 1) cluster_wait();

    int pending = c % NS;                             // the warp's first item not yet read
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
        const uint64_t drain_ns = a.wait_ns > kDrainNs ? a.wait_ns : kDrainNs;
        for (int n = pending; n < total && n < pending + sm.rh; n += NS)
            if (!warp_wait(&sm.full[(c / NS) * sm.rh + n % sm.rh], static_cast<uint32_t>((n / sm.rh) & 1), drain_ns))
                break;
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
            if (!got) warp_wait_cluster(sm.red_tx, 0u, a.wait_ns > kDrainNs ? a.wait_ns : kDrainNs);
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
    const int rh = ring / halves(M);
    const bool part_in_ring =
        parts == 1 && rh >= Pmax && rh >= kWarps / halves(M) && M * item_rows(M) * 4 <= slot_bytes(M, F);
    size_t b = static_cast<size_t>(ring) * slot_bytes(M, F);
    b += static_cast<size_t>(Pmax) * xfrag_bytes(M, F);
    b += static_cast<size_t>(xparam_region(M, F, Pmax));
    b += part_in_ring ? 0 : static_cast<size_t>(parts) * kWarps * M * item_rows(M) * 4;
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
    // (int8 weights run the four-token instance from m = 1)
    case 1: return reinterpret_cast<const void *>(&matvec_kernel<F == kFmtW8 ? 4 : 1, F>);
    case 2: return reinterpret_cast<const void *>(&matvec_kernel<F == kFmtW8 ? 4 : 2, F>);
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

// Issue time of one record (Q4_0 bytes) on an SM running one CTA, in
// microseconds: fitted to graph-replay timings of this kernel on GB300.
double record_us(int M) { return M <= 1 ? 0.115 : M == 2 ? 0.13 : M == 4 ? 0.195 : M == 8 ? 0.206 : 0.291; }

bool plan_matvec_search(int M, int F, int fmt, int64_t k, int64_t n, int sm_count, MatvecPlan *plan);

} // namespace

// Choose the cluster size S (K slices per 128-row group), the number of
// persistent clusters and the ring depth (slots; the whole slice, or a
// multiple of 8). Candidates: every S and depth whose shared memory fits,
// with as many clusters as the device holds at once (up to one per group).
// Their time is estimated in microseconds from constants fitted to graph-
// replay timings of this kernel on GB300:
//   the busiest SM's records at the kernel's issue time per record (two CTAs
//   of one call on an SM hide each other's latencies), or the layer's HBM
//   stream if longer, slowed when a refilled ring keeps too few bytes in
//   flight per SM; a fixed start; X staging in rounds of loads; the slices'
//   exchange; per-group handshakes of CTAs with several groups and a K
//   split; and the
//   start-up that cannot overlap the preceding call when no SM has room for
//   the next call's CTA.
bool plan_matvec(int64_t m, int64_t k, int64_t n, int sm_count, MatvecPlan *plan, int fmt)
{
    if (m < 1 || m > 16 || sm_count < 1) return false;
    const int F = fmt == kMatvecInt8 ? kFmtW8 : kFmtQ4;
    // int8 weights stage all four token columns of a tile (m <= 4 share the
    // four-token instance)
    const int M = F == kFmtW8 ? std::max(4, instance_of(m)) : instance_of(m);
    // a plan depends on the instance, the shape, the format and the device
    // (its SM count and cluster occupancy): computed once per such key
    static std::mutex mu;
    static std::map<std::tuple<int, int, int64_t, int64_t, int, int>, MatvecPlan> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    const auto key = std::make_tuple(dev, M, k, n, fmt, sm_count);
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = cache.find(key);
        if (it != cache.end()) {
            if (it->second.ctas == 0) return false;
            *plan = it->second;
            return true;
        }
    }
    MatvecPlan found;
    const bool ok = plan_matvec_search(M, F, fmt, k, n, sm_count, &found);
    std::lock_guard<std::mutex> lock(mu);
    cache.emplace(key, ok ? found : MatvecPlan{});
    if (!ok) return false;
    *plan = found;
    return true;
}

namespace {

bool plan_matvec_search(int M, int F, int fmt, int64_t k, int64_t n, int sm_count, MatvecPlan *plan)
{
    const int hv = halves(M);
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t np = ceil_div(k, kPairK);
    const size_t half = kSmemPerSM / 2 - 1024;
    const double rec_t = record_us(M) * rec_bytes(F) / kRecordBytes;
    const double sm_bw = 6.77e6 / 152.0;                     // bytes per microsecond per SM
    const double hbm_t = static_cast<double>(groups * np) * rec_bytes(F) / (sm_bw * sm_count);
    MatvecPlan best;
    double best_cost = 1e300;
    // With four or more 128-row groups per SM every SM has whole groups to
    // work on: no K split (measured on the 151936-row logit head at m = 1, 4,
    // 8 and 16, where the split plans the model would pick were slower).
    const int max_slices = groups >= 4 * static_cast<int64_t>(sm_count) ? 1 : kMaxSlices;
    for (int S = 1; S <= max_slices && S <= np; ++S) {
        const int64_t P = ceil_div(np, S);
        for (int parts = 1; parts <= 2; ++parts) {
            for (int ring = kWarps; ring <= max_ring(M); ++ring) {
                const size_t smem = matvec_smem(M, F, static_cast<int>(P), S, ring, parts);
                if (smem > kSmemOptIn) break;                 // deeper rings only grow
                // the exact ring (the whole slice, hv x a multiple of P: no
                // refills) or a multiple of 8
                if (ring % kWarps != 0 && ring % (hv * P) != 0) continue;
                const int64_t cm = matvec_max_clusters(M, F, S, smem);
                if (cm < 1) continue;
                const int64_t clusters = std::min<int64_t>(groups, cm);
                const int64_t tiles = ceil_div(groups, clusters);
                if ((tiles > 1 ? 2 : 1) != parts) continue;
                const int64_t recs = tiles * P;               // records of a CTA
                const int64_t exact = hv * std::max<int64_t>(kWarps / hv, recs);
                if (ring > exact) break;
                if (ring != exact && ring % kWarps != 0) continue;
                const int64_t ctas = clusters * S;
                const int per_sm = static_cast<int>(ceil_div(ctas, sm_count));
                const bool two_fit = smem <= half;
                const double issue = per_sm * static_cast<double>(recs) * rec_t / (per_sm >= 2 ? 1.512 : 1.0);
                double eff = 1.0;
                if (ring != exact)
                    eff = std::min(1.0, std::max(0.05, per_sm * ring * static_cast<double>(slot_bytes(M, F)) /
                                                           (sm_bw * 2.24)));
                const double loop = std::max(issue, hbm_t / eff);
                const int64_t tasks = M <= 4 ? 2 * P * M : 2 * P;
                const int64_t per_round = M <= 4 ? 8 * 32 : 8 * (64 / M);
                const double stage = 0.3 * static_cast<double>(ceil_div(tasks, per_round));
                const double slices = S > 1 ? 0.15 * (S - 2) : 0.0;
                // (the handshake crosses the cluster; without a K split the
                // group's rows are summed inside the CTA)
                const double hand = tiles > 1 && S > 1 ? 0.565 * static_cast<double>(tiles * S) : 0.0;
                // (a second CTA of this call on a few SMs delays only those)
                const double two_share = std::min(1.0, 4.0 * std::max<double>(0.0, ctas - sm_count) / sm_count);
                const double no_overlap = 1.476 * (two_fit ? two_share : 1.0);
                const double cost = 3.0 + stage + loop + slices + hand + no_overlap;
                if (cost < best_cost - 1e-9) {
                    best_cost = cost;
                    best.M = M;
                    best.fmt = fmt;
                    best.S = S;
                    best.clusters = static_cast<int>(clusters);
                    best.ctas = static_cast<int>(ctas);
                    best.ring = ring;
                    best.smem = smem;
                    best.est_us = cost;
                }
            }
        }
    }
    if (best.ctas == 0) return false;
    *plan = best;
    return true;
}

} // namespace

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
            const int hv = halves(M);
            const int exact = hv * static_cast<int>(std::max<int64_t>(kWarps / hv, P));
            if (P * hv <= max_ring(M) && matvec_smem(M, kFmtQ4, static_cast<int>(P), S, exact, 1) <= limit)
                ring = exact;
            for (int64_t r = std::min<int64_t>(max_ring(M), P * hv / kWarps * kWarps); r >= kWarps && ring == 0;
                 r -= kWarps)
                if (matvec_smem(M, kFmtQ4, static_cast<int>(P), S, static_cast<int>(r), 1) <= limit)
                    ring = static_cast<int>(r);
            if (ring == 0) continue;
            const size_t smem = matvec_smem(M, kFmtQ4, static_cast<int>(P), S, ring, 1);
            const int64_t cmax = matvec_max_clusters(M, kFmtQ4, S, smem);
            if (cmax < 1) continue;
            const int64_t clusters = groups * experts;
            const double waves = static_cast<double>(ceil_div(clusters, cmax));
            const double cost = waves * (static_cast<double>(P) + 4.0) + (S > 1 ? 2.0 : 0.0) +
                                (P * hv > ring ? static_cast<double>(P - ring / hv) : 0.0);
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
