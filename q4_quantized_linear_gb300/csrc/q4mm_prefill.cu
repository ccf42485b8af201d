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
//      elements follow the same order the weight dequantiser emits), so the
//      GEMM fetches each X tile with one 1-D bulk copy.
//   2. gemm: one CTA per (128 weight rows) x (T tokens). Warp roles:
//        warp 0     producer: bulk copies of raw packed W records and X tiles
//        warp 1     TMEM allocation and the single MMA-issuing thread
//        warps 2-9  dequantise W (split-half nibbles -> exact bf16 (q-8),
//                   times d rounded to bf16) into 128B-swizzled K-major shared
//                   tiles, one 16-row tile per warp, then the epilogue
//                   (TMEM -> registers -> Y), two warps per TMEM sub-partition
//      tcgen05.mma kind::f16 (bf16 x bf16, fp32 accumulate in TMEM), M = 128
//      weight rows, N = T tokens (split into 256 + rest when T > 256).
//      Every ring is an mbarrier pipeline; every wait is time-bounded.
#include <algorithm>
#include <cuda_runtime.h>

#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kErrTimeout = 5;
constexpr int kDequantWarps = 8;
constexpr int kGemmThreads = (2 + kDequantWarps) * 32;
constexpr int kAStageBytes = 128 * 128; // 128 rows x 64 bf16

// ------------------------------------------------------------- xcast -----

__global__ void __launch_bounds__(256) xcast_kernel(const XcastArgs a)
{
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
    pdl_launch_dependents();
}

// -------------------------------------------------------------- gemm -----

struct Smem {
    uint8_t *b, *a, *w;
    uint64_t *full_b, *empty_b, *full_a, *empty_a, *full_w, *empty_w, *done;
    uint32_t *tmem_slot;
    int *abort;
};

__device__ __forceinline__ bool aborted(const Smem &sm) { return *reinterpret_cast<volatile int *>(sm.abort) != 0; }

__device__ __forceinline__ void fail(const Smem &sm, const PrefillArgs &a)
{
    *reinterpret_cast<volatile int *>(sm.abort) = 1;
    record_status(a.status, kErrTimeout);
}

// bf16 (q-8) times d: d is rounded to bf16 and the product rounded once,
// so |w - (q-8)*d| <= 2^-8 |(q-8)*d|; (q-8) itself is exact.
__device__ __forceinline__ uint32_t scale_splat_bf16(float d)
{
    const uint32_t h = bf16_rn_bits(d);
    return h | (h << 16);
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_kernel(const PrefillArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rt = blockIdx.x / a.ts; // 128-row tile
    const int jt = blockIdx.x % a.ts; // token tile
    const int T = a.T;
    const int np = a.np;
    const int G0 = 2 * rt;
    const bool has_g1 = G0 + 1 < a.groups;
    const uint32_t bstage = static_cast<uint32_t>(T) * 128u;

    Smem sm;
    sm.b = base;
    sm.a = sm.b + static_cast<size_t>(a.rb) * bstage;
    sm.w = sm.a + static_cast<size_t>(a.ra) * kAStageBytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sm.w + static_cast<size_t>(a.rw) * 2 * kPairBytes);
    sm.full_b = bars;
    sm.empty_b = sm.full_b + a.rb;
    sm.full_a = sm.empty_b + a.rb;
    sm.empty_a = sm.full_a + a.ra;
    sm.full_w = sm.empty_a + a.ra;
    sm.empty_w = sm.full_w + a.rw;
    sm.done = sm.empty_w + a.rw;
    sm.tmem_slot = reinterpret_cast<uint32_t *>(sm.done + 1);
    sm.abort = reinterpret_cast<int *>(sm.tmem_slot + 1);

    if (tid == 0) {
        for (int i = 0; i < a.rb; ++i) mbar_init(&sm.full_b[i], 1), mbar_init(&sm.empty_b[i], 1);
        for (int i = 0; i < a.ra; ++i) mbar_init(&sm.full_a[i], kDequantWarps), mbar_init(&sm.empty_a[i], 1);
        for (int i = 0; i < a.rw; ++i) mbar_init(&sm.full_w[i], 1), mbar_init(&sm.empty_w[i], kDequantWarps);
        mbar_init(sm.done, 1);
        *sm.abort = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(sm.tmem_slot, static_cast<uint32_t>(a.tmem_cols));
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *sm.tmem_slot;

    // The raw weight records never come from the preceding kernel (that is
    // always this call's X cast, which writes only the X image), so the first
    // weight stages are requested before the dependency wait.
    const uint8_t *xsrc = a.ximg + static_cast<size_t>(jt) * np * bstage;
    const uint32_t wbytes = (has_g1 ? 2u : 1u) * kPairBytes;
    auto issue_w = [&](int p, uint64_t pol) {
        const int sw = p % a.rw;
        mbar_arrive_expect_tx(&sm.full_w[sw], wbytes);
        uint8_t *wdst = sm.w + static_cast<size_t>(sw) * 2 * kPairBytes;
        bulk_g2s_hint(wdst, a.W + (static_cast<int64_t>(G0) * np + p) * kPairBytes, kPairBytes, &sm.full_w[sw], pol);
        if (has_g1)
            bulk_g2s_hint(wdst + kPairBytes, a.W + (static_cast<int64_t>(G0 + 1) * np + p) * kPairBytes, kPairBytes,
                          &sm.full_w[sw], pol);
    };
    int w_issued = 0;
    if (warp == 0 && lane == 0) {
        const uint64_t pol_w = policy_evict_last();
        for (; w_issued < min(a.rw, np); ++w_issued) issue_w(w_issued, pol_w);
    }

    pdl_wait();

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        int b_issued = 0;
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_last();
            const uint64_t pol_x = policy_evict_last();
            for (int p = 0; p < np && !aborted(sm); ++p) {
                const int sb = p % a.rb;
                if (!mbar_wait(&sm.empty_b[sb], ((p / a.rb) & 1) ^ 1, a.wait_ns)) { fail(sm, a); break; }
                mbar_arrive_expect_tx(&sm.full_b[sb], bstage);
                bulk_g2s_hint(sm.b + static_cast<size_t>(sb) * bstage, xsrc + static_cast<size_t>(p) * bstage, bstage,
                              &sm.full_b[sb], pol_x);
                ++b_issued;
                // refill the weight slot that stage p used once it is free
                const int pw = p + a.rw;
                if (pw < np) {
                    if (!mbar_wait(&sm.empty_w[p % a.rw], (p / a.rw) & 1, a.wait_ns)) { fail(sm, a); break; }
                    issue_w(pw, pol_w);
                    ++w_issued;
                }
            }
            // drain our copies before the CTA may exit
            for (int i = 0; i < a.rw; ++i) {
                int last = -1;
                for (int p = w_issued - 1; p >= 0 && p >= w_issued - a.rw; --p)
                    if (p % a.rw == i) { last = p; break; }
                if (last >= 0 && !mbar_wait(&sm.full_w[i], (last / a.rw) & 1, a.wait_ns)) fail(sm, a);
            }
            for (int i = 0; i < a.rb; ++i) {
                int last = -1;
                for (int p = b_issued - 1; p >= 0 && p >= b_issued - a.rb; --p)
                    if (p % a.rb == i) { last = p; break; }
                if (last >= 0 && !mbar_wait(&sm.full_b[i], (last / a.rb) & 1, a.wait_ns)) fail(sm, a);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // --------------------------------------------------------------- MMA
        if (lane == 0) {
            const int N1 = T > 256 ? 256 : T;
            const int N2 = T - N1;
            const uint32_t id1 = idesc_bf16_f32(128, static_cast<uint32_t>(N1));
            const uint32_t id2 = idesc_bf16_f32(128, static_cast<uint32_t>(N2 > 0 ? N2 : 16));
            const uint32_t a0 = smem_u32(sm.a), b0 = smem_u32(sm.b);
            for (int p = 0; p < np && !aborted(sm); ++p) {
                const int sa = p % a.ra, sb = p % a.rb;
                if (!mbar_wait(&sm.full_a[sa], (p / a.ra) & 1, a.wait_ns)) { fail(sm, a); break; }
                if (!mbar_wait(&sm.full_b[sb], (p / a.rb) & 1, a.wait_ns)) { fail(sm, a); break; }
                tc_fence_after();
                const uint32_t as = a0 + static_cast<uint32_t>(sa) * kAStageBytes;
                const uint32_t bs = b0 + static_cast<uint32_t>(sb) * bstage;
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {
                    const uint64_t ad = smem_desc_sw128(as + kk * 32);
                    const uint32_t acc = (p | kk) != 0;
                    tc_mma_f16(tmem, ad, smem_desc_sw128(bs + kk * 32), id1, acc);
                    if (N2 > 0) tc_mma_f16(tmem + 256, ad, smem_desc_sw128(bs + 256 * 128 + kk * 32), id2, acc);
                }
                tc_commit(&sm.empty_a[sa]);
                tc_commit(&sm.empty_b[sb]);
            }
            tc_commit(sm.done); // also taken on abort: no MMA of ours is in flight past this
        }
        __syncwarp();
    } else {
        // ----------------------------------------------- dequantise W, epilogue
        const int tt = warp - 2; // 16-row tile of this warp, 0..7
        const int grp = tt >> 2;
        const int g = lane >> 2, c4 = lane & 3;
        const bool have = grp == 0 || has_g1;
        for (int p = 0; p < np && !aborted(sm); ++p) {
            const int sw = p % a.rw, sa = p % a.ra;
            if (!mbar_wait(&sm.full_w[sw], (p / a.rw) & 1, a.wait_ns)) { fail(sm, a); break; }
            if (!mbar_wait(&sm.empty_a[sa], ((p / a.ra) & 1) ^ 1, a.wait_ns)) { fail(sm, a); break; }
            const uint8_t *wst = sm.w + static_cast<size_t>(sw) * 2 * kPairBytes;
            uint8_t *ast = sm.a + static_cast<size_t>(sa) * kAStageBytes;
            uint4 nib = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
            uint2 sc = make_uint2(0u, 0u);
            if (have) {
                const uint8_t *rec = wst + grp * kPairBytes + (tt & 3) * kRecordBytes;
                nib = lds128(rec + 64 + lane * 16);
                sc = lds64(rec + g * 8);
            }
            // o[h][blk]: 8 weights of row (g + 8h), block blk, elements 4c4 + {0,2,16,18,1,3,17,19}
            const uint32_t words[4] = {nib.x, nib.y, nib.z, nib.w};
            const uint32_t sbits[4] = {sc.x & 0xFFFF, sc.x >> 16, sc.y & 0xFFFF, sc.y >> 16};
            uint4 o[2][2];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int blk = i >> 1, h = i & 1;
                const uint32_t dd =
                    scale_splat_bf16(__half2float(__ushort_as_half(static_cast<unsigned short>(sbits[i]))));
                uint32_t v[4];
                unpack_word_bf16(words[i], v);
                o[h][blk] = make_uint4(bf16x2_mul(v[0], dd), bf16x2_mul(v[1], dd), bf16x2_mul(v[2], dd),
                                       bf16x2_mul(v[3], dd));
            }
            // Store order: lanes of odd g write the other block first, so each
            // 8-lane phase of a 16-byte store hits 8 distinct bank groups.
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int h = i & 1;
                const int blk = (i >> 1) ^ (g & 1);
                const int row = tt * 16 + g + 8 * h;
                const int chunk = blk * 4 + c4;
                sts128(ast + row * 128 + ((chunk ^ (row & 7)) << 4), blk ? o[h][1] : o[h][0]);
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&sm.full_a[sa]);
                mbar_arrive(&sm.empty_w[sw]);
            }
        }

        // epilogue: this warp's TMEM sub-partition, half of the token columns
        const int q = warp & 3;
        const int half = (warp - 2) >> 2;
        const int row = q * 32 + lane;
        const int64_t grow = static_cast<int64_t>(rt) * 128 + row;
        if (!mbar_wait(sm.done, 0, a.wait_ns)) fail(sm, a);
        tc_fence_after();
        pdl_launch_dependents();
        const int chunks = T / 16;
        const int c_lo = half * ((chunks + 1) / 2), c_hi = half ? chunks : (chunks + 1) / 2;
        for (int cc = c_lo; cc < c_hi; ++cc) {
            const int c0 = cc * 16;
            uint32_t r[16];
            tmem_ld_32x32b_x16(tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(c0), r);
            tmem_wait_ld();
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

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, static_cast<uint32_t>(a.tmem_cols));
    }
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

size_t gemm_smem_bytes(int T, int rb, int ra, int rw)
{
    return 1024 + static_cast<size_t>(rb) * T * 128 + static_cast<size_t>(ra) * kAStageBytes +
           static_cast<size_t>(rw) * 2 * kPairBytes + static_cast<size_t>(2 * rb + 2 * ra + 2 * rw + 1) * 8 + 16;
}

} // namespace

// Choose the token tile T (multiple of 16, at most 480) and the number of
// token tiles so that (128-row tiles) x (token tiles) fills the SMs in as few
// waves as possible, then the deepest rings that fit in shared memory.
bool plan_prefill(int64_t m, int64_t k, int64_t n, int sm_count, PrefillPlan *plan)
{
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t rowtiles = ceil_div(groups, 2);
    const int64_t np = ceil_div(k, kPairK);
    PrefillPlan best;
    double best_cost = 1e300;
    for (int64_t ts = ceil_div(m, 480); ts <= std::max<int64_t>(1, ceil_div(m, 16)); ++ts) {
        const int64_t T = round_up(ceil_div(m, ts), 16);
        if (T > 480) continue;
        const int64_t ctas = rowtiles * ts;
        const int64_t waves = ceil_div(ctas, sm_count);
        const double cost = static_cast<double>(waves) * (static_cast<double>(T) + 48.0);
        if (cost < best_cost - 1e-9) {
            best_cost = cost;
            best.T = static_cast<int>(T);
            best.ts = static_cast<int>(ts);
        }
        if (ts > 4096) break;
    }
    if (best.T == 0) return false;
    best.rowtiles = static_cast<int>(rowtiles);
    best.ra = 3;
    best.rw = 4;
    best.rb = 6;
    while (best.rb > 2 && gemm_smem_bytes(best.T, best.rb, best.ra, best.rw) > kSmemOptIn) --best.rb;
    while (best.ra > 2 && gemm_smem_bytes(best.T, best.rb, best.ra, best.rw) > kSmemOptIn) --best.ra;
    best.smem = gemm_smem_bytes(best.T, best.rb, best.ra, best.rw);
    if (best.smem > kSmemOptIn) return false;
    int cols = 32;
    while (cols < best.T) cols <<= 1;
    best.tmem_cols = cols;
    best.ws_ximg_off = kWsCounterBytes;
    best.ws_bytes = kWsCounterBytes + static_cast<size_t>(best.ts) * np * best.T * 128;
    *plan = best;
    return true;
}

cudaError_t launch_prefill(const PrefillPlan &plan, const XcastArgs &xa, const PrefillArgs &pa, cudaStream_t s)
{
    {
        XcastArgs a = xa;
        void *kargs[] = {&a};
        const int64_t total = static_cast<int64_t>(xa.ts) * xa.np * xa.T * 8;
        const int64_t grid = std::min<int64_t>(ceil_div(total, 256), 65535);
        cudaError_t e = launch_pdl(reinterpret_cast<const void *>(&xcast_kernel), dim3(static_cast<unsigned>(grid)),
                                   dim3(256), 0, s, kargs);
        if (e != cudaSuccess) return e;
    }
    const void *fn = reinterpret_cast<const void *>(&gemm_kernel);
    cudaError_t e = set_max_smem(fn, plan.smem);
    if (e != cudaSuccess) return e;
    PrefillArgs a = pa;
    void *kargs[] = {&a};
    return launch_pdl(fn, dim3(static_cast<unsigned>(plan.rowtiles * plan.ts)), dim3(kGemmThreads), plan.smem, s, kargs);
}

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t s)
{
    wait_selftest_kernel<<<1, 32, 0, s>>>(status, limit_ns);
    return cudaGetLastError();
}

} // namespace q4
