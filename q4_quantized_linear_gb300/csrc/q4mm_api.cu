// q4mm_api.cu -- the C ABI of libq4mm (declared in include/q4mm.h): argument
// validation, per-device state, workspace handling and dispatch between the
// decode kernels (m <= 16: warp-MMA, CUDA-core or tcgen05) and the
// tensor-core prefill kernels (m > 16).
//
// The decode/prefill dispatch point follows golem, "Reading a prompt on the
// card": the mat-vec is built up to sixteen columns and tiled products take
// over beyond.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/q4mm.h"
#include "q4mm_internal.h"

namespace q4 {

__device__ int g_device_status = 0;

namespace {

constexpr int kMaxDevices = 64;
constexpr int64_t kDecodeMaxM = 16;

std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int> g_prefetch_w{0};
std::atomic<int> g_decode_kernel{Q4_DECODE_AUTO};
std::mutex g_trace_mutex;
TraceSettings g_trace;

struct DeviceSlot {
    std::once_flag once;
    int rc = Q4_OK;
    DeviceInfo info;
};
DeviceSlot g_dev[kMaxDevices];

struct Workspace {
    void *ptr = nullptr;
    size_t bytes = 0;
};
std::mutex g_ws_mutex;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Current device, checked to be a GB300-class part (compute capability 10.3).
int current_device(DeviceInfo *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    DeviceSlot &slot = g_dev[dev];
    std::call_once(slot.once, [&] {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            slot.rc = Q4_ERR_CUDA;
            return;
        }
        if (major != 10 || minor != 3) {
            slot.rc = Q4_ERR_UNSUPPORTED_DEVICE;
            return;
        }
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            slot.rc = Q4_ERR_CUDA;
            return;
        }
        slot.info.device = dev;
        slot.info.sm_count = sms;
        slot.info.status = static_cast<int *>(addr);
        slot.rc = Q4_OK;
    });
    if (slot.rc == Q4_OK) *out = slot.info;
    return slot.rc;
}

int map_cuda(cudaError_t e)
{
    if (e == cudaSuccess) return Q4_OK;
    cudaGetLastError();
    return Q4_ERR_CUDA;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool valid_nk(int64_t n, int64_t k)
{
    return n >= 1 && k >= 32 && (k % 32) == 0 && n <= (int64_t(1) << 31) - 64 && k <= (int64_t(1) << 24);
}

// Library-owned scratch for the forms without a workspace argument: one
// buffer per (device, stream), grown on demand. Its contents need no
// initialisation: every call writes the X image it reads.
int library_workspace(int dev, cudaStream_t s, size_t need, void **out)
{
    *out = nullptr;
    if (need == 0) return Q4_OK;
    std::lock_guard<std::mutex> lock(g_ws_mutex);
    Workspace &w = g_ws[{dev, s}];
    if (w.bytes >= need) {
        *out = w.ptr;
        return Q4_OK;
    }
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    if (cap != cudaStreamCaptureStatusNone) return Q4_ERR_WORKSPACE;
    if (w.ptr) {
        if (cudaStreamSynchronize(s) != cudaSuccess || cudaFree(w.ptr) != cudaSuccess) {
            cudaGetLastError();
            return Q4_ERR_CUDA;
        }
        w.ptr = nullptr;
        w.bytes = 0;
    }
    const size_t bytes = static_cast<size_t>(round_up(static_cast<int64_t>(need), 1 << 20));
    if (cudaMalloc(&w.ptr, bytes) != cudaSuccess) {
        cudaGetLastError();
        w.ptr = nullptr;
        return Q4_ERR_NO_MEMORY;
    }
    w.bytes = bytes;
    *out = w.ptr;
    return Q4_OK;
}

size_t workspace_size(int64_t m, int64_t k, int64_t n, int sm_count)
{
    if (m <= 0) return 0;
    if (m <= kDecodeMaxM) return 0;
    PrefillPlan p;
    return plan_prefill(m, k, n, sm_count, &p) ? p.ws_bytes : 0;
}

// Shared body of every matmul entry point. rows == nullptr: plain X/Y rows.
int matmul_impl(const void *W, const float *X, int64_t ldx, const int32_t *rows, float *Y, int64_t ldy,
                int64_t m, int64_t k, int64_t n, void *workspace, size_t ws_bytes, bool library_ws, cudaStream_t s)
{
    if (!W || !X || !Y || m < 0 || !valid_nk(n, k) || ldx < k || ldy < n) return Q4_ERR_INVALID_ARG;
    if (m > (int64_t(1) << 24)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W, 16) || !aligned(X, 16) || (ldx % 4) != 0 || !aligned(Y, 4)) return Q4_ERR_ALIGNMENT;
    if (workspace && !aligned(workspace, 256)) return Q4_ERR_ALIGNMENT;
    if (m == 0) return Q4_OK;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    const uint64_t wait_ns = g_wait_ns.load();

    // 17..32 rows: the mat-vec in two pieces (16 rows, then the rest) where
    // that is estimated faster than the GEMM. golem ("Reading a prompt on
    // the card") builds the mat-vec sixteen wide and takes tiled products
    // from thirty-two columns; which side wins in between depends on the
    // layer. The two planners' estimates decide; two mat-vec calls back to
    // back measured about 3 us above the sum of their estimates.
    if (m > kDecodeMaxM && m <= 2 * kDecodeMaxM && g_decode_kernel.load() == Q4_DECODE_AUTO) {
        MatvecPlan p16, prest;
        PrefillPlan pp;
        if (plan_matvec(kDecodeMaxM, k, n, dev.sm_count, &p16) &&
            plan_matvec(m - kDecodeMaxM, k, n, dev.sm_count, &prest) && plan_prefill(m, k, n, dev.sm_count, &pp)) {
            const double gemm_us = pp.est_us;
            if (p16.est_us + prest.est_us + 3.0 < gemm_us) {
                rc = matmul_impl(W, X, ldx, rows, Y, ldy, kDecodeMaxM, k, n, nullptr, 0, false, s);
                if (rc != Q4_OK) return rc;
                return matmul_impl(W, rows ? X : X + kDecodeMaxM * ldx, ldx, rows ? rows + kDecodeMaxM : nullptr,
                                   rows ? Y : Y + kDecodeMaxM * ldy, ldy, m - kDecodeMaxM, k, n, nullptr, 0, false,
                                   s);
            }
        }
    }

    if (m <= kDecodeMaxM) {
        // the decode paths need no scratch: K slices meet in cluster shared memory
        DecodeArgs a{};
        a.W = static_cast<const uint8_t *>(W);
        a.X = X;
        a.rows = rows;
        a.ldx = ldx;
        a.Y = Y;
        a.ldy = ldy;
        a.status = dev.status;
        a.wait_ns = wait_ns;
        a.m = static_cast<int>(m);
        a.n = static_cast<int>(n);
        a.nb = static_cast<int>(k / 32);
        a.np = static_cast<int>(ceil_div(k, kPairK));
        a.groups = static_cast<int>(ceil_div(n, kGroupRows));
        a.prefetch_w = g_prefetch_w.load();
        int kind = g_decode_kernel.load();
        // Measured on GB300 (graph replays, weights cycled beyond L2): whole
        // records per warp on the warp-level MMA are fastest for m <= 4 on
        // every layer measured, and for m = 5..8 on layers of up to two
        // 128-row groups per SM (on the 151936-row logit layer the row-tiled
        // warp-MMA kernel is faster there); the warp-MMA kernel above m = 8
        // (the record-MMA mode, built up to m = 16, was slower at m = 16 on
        // 14336 x 4096, 2560 x 9728 and 151936 x 2560).
        if (kind == Q4_DECODE_AUTO) kind = Q4_DECODE_MATVEC;
        if (kind == Q4_DECODE_MATVEC) {
            // the mat-vec stages the CTA's slice of X in shared memory; where
            // no plan leaves room for it (long K at m > 8), the whole-record
            // kernel, which reads X where it is used, serves the call
            MatvecPlan vp;
            if (plan_matvec(m, k, n, dev.sm_count, &vp)) return map_cuda(launch_matvec(vp, a, s));
            kind = Q4_DECODE_RECORD_MMA;
        }
        if (kind == Q4_DECODE_CUDA_CORE && m > kGemvMaxM) kind = Q4_DECODE_WARP_MMA;
        if (kind == Q4_DECODE_RECORD_MMA && m > kRecordMmaMaxM) kind = Q4_DECODE_WARP_MMA;
        if (kind == Q4_DECODE_WARP_MMA) {
            MmvPlan mp;
            if (!plan_mmv(m, k, n, dev.sm_count, &mp)) return Q4_ERR_INVALID_ARG;
            return map_cuda(launch_mmv(mp, a, s));
        }
        if (kind == Q4_DECODE_CUDA_CORE || kind == Q4_DECODE_RECORD_MMA) {
            GemvPlan gp;
            if (!plan_gemv(m, k, n, dev.sm_count, &gp)) return Q4_ERR_INVALID_ARG;
            return map_cuda(launch_gemv(gp, a, kind == Q4_DECODE_RECORD_MMA ? kGemvModeRecordMma : kGemvModeFma, s));
        }
        DecodePlan plan;
        if (!plan_decode(m, k, n, dev.sm_count, &plan)) return Q4_ERR_INVALID_ARG;
        return map_cuda(launch_decode(plan, a, s));
    }

    PrefillPlan plan;
    if (!plan_prefill(m, k, n, dev.sm_count, &plan)) return Q4_ERR_INVALID_ARG;
    if (library_ws) {
        rc = library_workspace(dev.device, s, plan.ws_bytes, &workspace);
        if (rc != Q4_OK) return rc;
        ws_bytes = plan.ws_bytes;
    }
    if (!workspace || ws_bytes < plan.ws_bytes) return Q4_ERR_WORKSPACE;
    XcastArgs xa{};
    xa.X = X;
    xa.rows = rows;
    xa.ldx = ldx;
    xa.ximg = static_cast<uint8_t *>(workspace) + plan.ws_ximg_off;
    xa.m = static_cast<int>(m);
    xa.nb = static_cast<int>(k / 32);
    xa.np = static_cast<int>(ceil_div(k, kPairK));
    xa.T = plan.T;
    xa.ts = plan.ts;
    PrefillArgs pa{};
    pa.W = static_cast<const uint8_t *>(W);
    pa.ximg = static_cast<const uint8_t *>(workspace) + plan.ws_ximg_off;
    pa.Y = Y;
    pa.rows = rows;
    pa.ldy = ldy;
    pa.status = dev.status;
    pa.wait_ns = wait_ns;
    pa.m = static_cast<int>(m);
    pa.n = static_cast<int>(n);
    pa.np = xa.np;
    pa.groups = static_cast<int>(ceil_div(n, kGroupRows));
    pa.T = plan.T;
    pa.ts = plan.ts;
    pa.ks = plan.ks;
    pa.bring = plan.bring;
    pa.wring = plan.wring;
    pa.astages = plan.astages;
    pa.prefetch_w = g_prefetch_w.load();
    return map_cuda(launch_prefill(plan, xa, pa, s));
}

} // namespace

// One launch of the mat-vec over an expert set (each expert at most 16
// rows). Q4_ERR_INVALID_ARG when no plan fits (the caller then runs the
// experts one by one).
int launch_expert_set(const ExpertSet &set, int max_m, const float *X, float *Y, int64_t k, int64_t n,
                      cudaStream_t s)
{
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    DecodeArgs a{};
    a.W = set.W[0];
    a.X = X;
    a.rows = nullptr;
    a.ldx = k;
    a.Y = Y;
    a.ldy = n;
    a.status = dev.status;
    a.wait_ns = g_wait_ns.load();
    a.m = max_m;
    a.n = static_cast<int>(n);
    a.nb = static_cast<int>(k / 32);
    a.np = static_cast<int>(ceil_div(k, kPairK));
    a.groups = static_cast<int>(ceil_div(n, kGroupRows));
    a.prefetch_w = g_prefetch_w.load();
    MatvecPlan plan;
    if (!plan_matvec_experts(max_m, k, n, set.count, dev.sm_count, &plan)) return Q4_ERR_INVALID_ARG;
    return map_cuda(launch_matvec_experts(plan, a, set, s));
}

TraceSettings trace_settings()
{
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    return g_trace;
}

cudaError_t set_max_smem(const void *func, size_t bytes)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    auto it = done.find({dev, func});
    if (it == done.end()) {
        // the dynamic limit plus the kernel's static shared memory may not
        // exceed the device's per-block opt-in maximum
        int optin = 0;
        cudaFuncAttributes fa{};
        e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, func);
        if (e != cudaSuccess) return e;
        const size_t limit = static_cast<size_t>(optin) - fa.sharedSizeBytes;
        e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(limit));
        if (e != cudaSuccess) return e;
        it = done.emplace(std::make_pair(dev, func), limit).first;
    }
    return bytes <= it->second ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void **args,
                       int cluster_x)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[na].val.programmaticStreamSerializationAllowed = 1;
    ++na;
    if (cluster_x > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = static_cast<unsigned>(cluster_x);
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelExC(&cfg, func, args);
}

} // namespace q4

using namespace q4;

extern "C" {

Q4MM_API size_t q4_0_packed_size(int64_t n, int64_t k)
{
    if (!valid_nk(n, k)) return 0;
    return static_cast<size_t>(ceil_div(n, kGroupRows) * ceil_div(k, kPairK) * kRecordBytes);
}

Q4MM_API int q4_0_pack(void *W_packed, const void *blocks, int64_t n, int64_t k, q4mm_stream_t stream)
{
    if (!W_packed || !blocks || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(blocks, 2)) return Q4_ERR_ALIGNMENT;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    return map_cuda(launch_pack(static_cast<uint8_t *>(W_packed), static_cast<const uint8_t *>(blocks), n, k,
                                reinterpret_cast<cudaStream_t>(stream)));
}

Q4MM_API int q4_0_unpack(void *blocks, const void *W_packed, int64_t n, int64_t k, q4mm_stream_t stream)
{
    if (!W_packed || !blocks || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(blocks, 2)) return Q4_ERR_ALIGNMENT;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    return map_cuda(launch_unpack(static_cast<uint8_t *>(blocks), static_cast<const uint8_t *>(W_packed), n, k,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

Q4MM_API size_t q4_0_matmul_workspace_size(int64_t m, int64_t k, int64_t n)
{
    if (m <= 0 || !valid_nk(n, k)) return 0;
    DeviceInfo dev;
    if (current_device(&dev) != Q4_OK) return 0;
    return workspace_size(m, k, n, dev.sm_count);
}

Q4MM_API int q4_0_matmul(const void *W_packed, const float *X, float *Y, int64_t m, int64_t k, int64_t n,
                         q4mm_stream_t stream)
{
    return matmul_impl(W_packed, X, k, nullptr, Y, n, m, k, n, nullptr, 0, true,
                       reinterpret_cast<cudaStream_t>(stream));
}

Q4MM_API int q4_0_matmul_w4a8(const void *W_packed, const float *X, float *Y, int64_t m, int64_t k, int64_t n,
                              q4mm_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!W_packed || !X || !Y || m < 0 || m > kRecordMmaMaxM || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W_packed, 16) || !aligned(X, 16) || !aligned(Y, 4)) return Q4_ERR_ALIGNMENT;
    if (m == 0) return Q4_OK;
    DeviceInfo dev;
    int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    DecodeArgs a{};
    a.W = static_cast<const uint8_t *>(W_packed);
    a.X = X;
    a.rows = nullptr;
    a.ldx = k;
    a.Y = Y;
    a.ldy = n;
    a.status = dev.status;
    a.wait_ns = g_wait_ns.load();
    a.m = static_cast<int>(m);
    a.n = static_cast<int>(n);
    a.nb = static_cast<int>(k / 32);
    a.np = static_cast<int>(ceil_div(k, kPairK));
    a.groups = static_cast<int>(ceil_div(n, kGroupRows));
    a.prefetch_w = g_prefetch_w.load();
    GemvPlan gp;
    if (!plan_gemv(m, k, n, dev.sm_count, &gp)) return Q4_ERR_INVALID_ARG;
    return map_cuda(launch_gemv(gp, a, kGemvModeW4A8, s));
}

Q4MM_API size_t q4_w8_packed_size(int64_t n, int64_t k)
{
    if (!valid_nk(n, k)) return 0;
    return w8_packed_bytes(n, k);
}

Q4MM_API int q4_w8_quantize(void *W8_packed, const float *W, int64_t n, int64_t k, q4mm_stream_t stream)
{
    if (!W8_packed || !W || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W8_packed, 16) || !aligned(W, 16)) return Q4_ERR_ALIGNMENT;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    return map_cuda(launch_w8_quantize(static_cast<uint8_t *>(W8_packed), W, n, k, reinterpret_cast<cudaStream_t>(stream)));
}

Q4MM_API int q4_w8_unpack(int8_t *codes, float *scales, const void *W8_packed, int64_t n, int64_t k,
                          q4mm_stream_t stream)
{
    if (!codes || !scales || !W8_packed || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W8_packed, 16) || !aligned(codes, 4) || !aligned(scales, 4)) return Q4_ERR_ALIGNMENT;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    return map_cuda(launch_w8_unpack(codes, scales, static_cast<const uint8_t *>(W8_packed), n, k,
                                     reinterpret_cast<cudaStream_t>(stream)));
}

Q4MM_API int q4_w8_matmul(const void *W8_packed, const float *X, float *Y, int64_t m, int64_t k, int64_t n,
                          q4mm_stream_t stream)
{
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (!W8_packed || !X || !Y || m < 0 || m > (int64_t(1) << 24) || !valid_nk(n, k)) return Q4_ERR_INVALID_ARG;
    if (!aligned(W8_packed, 16) || !aligned(X, 16) || !aligned(Y, 4)) return Q4_ERR_ALIGNMENT;
    if (m == 0) return Q4_OK;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    const int64_t groups = ceil_div(n, kW8GroupRows), np = ceil_div(k, kPairK);
    const float *row_scale = reinterpret_cast<const float *>(static_cast<const uint8_t *>(W8_packed) +
                                                             static_cast<size_t>(groups * np) * kW8RecordBytes);
    // up to 16 rows of X per launch, each one weight pass; where no plan fits
    // a launch of 16 rows (long k), 8 or 4
    for (int64_t t0 = 0, mt = 0; t0 < m; t0 += mt) {
        MatvecPlan vp;
        mt = std::min<int64_t>(16, m - t0);
        while (!plan_matvec(mt, k, n, dev.sm_count, &vp, kMatvecInt8) && mt > 4) mt = mt > 8 ? 8 : 4;
        if (!plan_matvec(mt, k, n, dev.sm_count, &vp, kMatvecInt8)) return Q4_ERR_INVALID_ARG;
        DecodeArgs a{};
        a.W = static_cast<const uint8_t *>(W8_packed);
        a.X = X + t0 * k;
        a.rows = nullptr;
        a.ldx = k;
        a.Y = Y + t0 * n;
        a.ldy = n;
        a.status = dev.status;
        a.wait_ns = g_wait_ns.load();
        a.m = static_cast<int>(mt);
        a.n = static_cast<int>(n);
        a.nb = static_cast<int>(k / 32);
        a.np = static_cast<int>(np);
        a.groups = static_cast<int>(groups);
        a.prefetch_w = g_prefetch_w.load();
        a.row_scale = row_scale;
        const int e = map_cuda(launch_matvec(vp, a, s));
        if (e != Q4_OK) return e;
    }
    return Q4_OK;
}

Q4MM_API int q4_0_matmul_ws(const void *W_packed, const float *X, float *Y, int64_t m, int64_t k, int64_t n,
                            void *workspace, size_t workspace_bytes, q4mm_stream_t stream)
{
    return matmul_impl(W_packed, X, k, nullptr, Y, n, m, k, n, workspace, workspace_bytes, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

Q4MM_API int q4_0_matmul_batched_slots(const void *W_packed, const float *X_slots, int64_t ldx,
                                       const int32_t *slot_ids, int64_t m, float *Y_slots, int64_t ldy, int64_t k,
                                       int64_t n, q4mm_stream_t stream)
{
    if (m > 0 && !slot_ids) return Q4_ERR_INVALID_ARG;
    if (slot_ids && !aligned(slot_ids, 4)) return Q4_ERR_ALIGNMENT;
    return matmul_impl(W_packed, X_slots, ldx, slot_ids, Y_slots, ldy, m, k, n, nullptr, 0, true,
                       reinterpret_cast<cudaStream_t>(stream));
}

Q4MM_API int q4_0_matmul_batched_slots_ws(const void *W_packed, const float *X_slots, int64_t ldx,
                                          const int32_t *slot_ids, int64_t m, float *Y_slots, int64_t ldy, int64_t k,
                                          int64_t n, void *workspace, size_t workspace_bytes, q4mm_stream_t stream)
{
    if (m > 0 && !slot_ids) return Q4_ERR_INVALID_ARG;
    if (slot_ids && !aligned(slot_ids, 4)) return Q4_ERR_ALIGNMENT;
    return matmul_impl(W_packed, X_slots, ldx, slot_ids, Y_slots, ldy, m, k, n, workspace, workspace_bytes, false,
                       reinterpret_cast<cudaStream_t>(stream));
}

Q4MM_API const char *q4_status_string(int status)
{
    switch (status) {
    case Q4_OK: return "ok";
    case Q4_ERR_INVALID_ARG: return "invalid argument";
    case Q4_ERR_ALIGNMENT: return "misaligned pointer or leading dimension";
    case Q4_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs compute capability 10.3)";
    case Q4_ERR_CUDA: return "CUDA runtime error";
    case Q4_ERR_DEVICE_TIMEOUT: return "a device-side wait ran out of time";
    case Q4_ERR_WORKSPACE: return "workspace missing or too small";
    case Q4_ERR_NO_MEMORY: return "out of device memory";
    case Q4_ERR_IO: return "file could not be opened or read";
    case Q4_ERR_FORMAT: return "file breaks the GGUF layout";
    case Q4_ERR_DEVICE_CHECK: return "a kernel's range check failed (checked build)";
    default: return "unknown status";
    }
}

Q4MM_API int q4_build_flags(void)
{
    int f = 0;
#ifdef Q4MM_CHECKED
    f |= 1;
#endif
#ifdef Q4MM_TRACE
    f |= 2;
#endif
    return f;
}

Q4MM_API int q4_last_device_status(int clear)
{
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    if (cudaDeviceSynchronize() != cudaSuccess) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int)) != cudaSuccess) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    if (clear) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int)) != cudaSuccess) {
            cudaGetLastError();
            return Q4_ERR_CUDA;
        }
    }
    return v;
}

Q4MM_API int q4_set_wait_limit_ns(uint64_t ns)
{
    if (ns == 0) return Q4_ERR_INVALID_ARG;
    g_wait_ns.store(ns);
    return Q4_OK;
}

Q4MM_API int q4_set_weight_prefetch(int enable)
{
    g_prefetch_w.store(enable ? 1 : 0);
    return Q4_OK;
}

Q4MM_API int q4_set_decode_kernel(int kind)
{
    if (kind < Q4_DECODE_AUTO || kind > Q4_DECODE_MATVEC) return Q4_ERR_INVALID_ARG;
    g_decode_kernel.store(kind);
    return Q4_OK;
}

Q4MM_API int q4_debug_set_trace(void *buffer, size_t bytes, uint32_t cta)
{
#ifdef Q4MM_TRACE
    std::lock_guard<std::mutex> lock(g_trace_mutex);
    if (!buffer || bytes < 64) {
        g_trace = TraceSettings{};
        return Q4_OK;
    }
    if (!aligned(buffer, 16)) return Q4_ERR_ALIGNMENT;
    g_trace.buf = static_cast<unsigned long long *>(buffer);
    g_trace.cap = static_cast<unsigned>(bytes / 16 / kTraceRegions);
    g_trace.cta = cta;
    return Q4_OK;
#else
    (void)buffer, (void)bytes, (void)cta;
    return Q4_ERR_INVALID_ARG;
#endif
}

Q4MM_API int q4_selftest_wait_timeout(uint64_t limit_ns, q4mm_stream_t stream)
{
    if (limit_ns == 0 || limit_ns > 10000000000ull) return Q4_ERR_INVALID_ARG;
    DeviceInfo dev;
    const int rc = current_device(&dev);
    if (rc != Q4_OK) return rc;
    return map_cuda(launch_wait_selftest(dev.status, limit_ns, reinterpret_cast<cudaStream_t>(stream)));
}

} // extern "C"
