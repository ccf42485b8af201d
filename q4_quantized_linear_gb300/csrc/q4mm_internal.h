// q4mm_internal.h -- host-side interfaces between the translation units of
// libq4mm (argument structs passed by value to the kernels, planners and
// launchers). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace q4 {

// Packed layout: records of 128 rows (a group) x 2 blocks (a pair).
constexpr int kGroupRows = 128;
constexpr int kPairK = 64;
constexpr int kRecordBytes = 4608;     // 128 x 2 x 18
constexpr int kRecScaleOff = 0;        // 4 bytes per row: fp16 d of block 0 | block 1
constexpr int kRecQs0Off = 512;        // 16 bytes per row: qs of block 0
constexpr int kRecQs1Off = 2560;       // 16 bytes per row: qs of block 1

// 227 KB per CTA on sm_100-family parts, less room for a kernel's static
// shared variables; plans never ask for more dynamic shared memory than this.
constexpr size_t kSmemOptIn = 232448 - 256;
constexpr size_t kSmemPerSM = 233472;  // 228 KB per SM

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// Per-device facts the launchers need.
struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int *status = nullptr;   // device address of the status word
};

// Raise a kernel's dynamic shared-memory limit to the opt-in maximum, once per
// (device, kernel).
cudaError_t set_max_smem(const void *func, size_t bytes);

// Event-trace destination the kernels record into (profiling builds only):
// one region of records per recording thread, lanes 0..3 of warps 0..23.
constexpr unsigned kTraceRegions = 96;
struct TraceSettings {
    unsigned long long *buf = nullptr;
    unsigned cap = 0, cta = 0;
};
TraceSettings trace_settings();

// Launch helper: programmatic-dependent launch on `stream`, optionally as
// clusters of `cluster_x` CTAs along x.
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void **args,
                       int cluster_x = 1);

// ------------------------------------------------------------------ pack --

cudaError_t launch_pack(uint8_t *packed, const uint8_t *blocks, int64_t n, int64_t k, cudaStream_t s);
cudaError_t launch_unpack(uint8_t *blocks, const uint8_t *packed, int64_t n, int64_t k, cudaStream_t s);

// ---------------------------------------------------------------- decode --

struct DecodeArgs {
    const uint8_t *W;
    const float *X;
    const int32_t *rows;   // slot rows (nullptr: row t)
    int64_t ldx;
    float *Y;
    int64_t ldy;
    int *status;
    uint64_t wait_ns;
    int m, n, nb, np, groups;
    int pass_p0;           // first pair of this launch's K range
    int S, pbase, prem;    // K slices of the range: slice s has pbase + (s < prem) pairs
    int clusters;          // clusters in the grid: cluster c owns groups c, c + clusters, ...
    int ring;              // weight-record ring depth (>= 4)
    int accumulate;        // add into Y instead of overwriting it
    int xs_bytes;          // shared bytes of the staged X image
    int prefetch_w;        // stream W before waiting on the preceding kernel
    const float *row_scale;   // int8 weights: the rows' scales (nullptr: Q4_0)
    unsigned long long *trace_buf;
    unsigned trace_cap, trace_cta;
};

struct DecodePlan {
    int N = 16;            // MMA N: hi and lo rows of X, 16 (m <= 8) or 32
    int S = 1;             // K slices = cluster size
    int passes = 1;        // launches over consecutive K ranges
    int pairs_per_pass = 0;
    int clusters = 0;      // persistent clusters per launch
    int ctas = 0;          // clusters x S
    int ring = 8;          // weight-record ring depth (multiple of 4 and of sets)
    int sets = 2;          // dequantiser sets (2 or 3)
    int xs_bytes = 0;
    size_t smem = 0;
};

bool plan_decode(int64_t m, int64_t k, int64_t n, int sm_count, DecodePlan *plan);
cudaError_t launch_decode(const DecodePlan &plan, const DecodeArgs &args, cudaStream_t s);

// ------------------------------------------------------------------ gemv --

// Widest call the CUDA-core GEMV kernel is built for.
constexpr int kGemvMaxM = 4;
// Widest call the record-MMA mode of the same kernel is built for.
constexpr int kRecordMmaMaxM = 16;

struct GemvPlan {
    int M = 1;             // token rows (the kernel instance)
    int S = 1;             // K slices = cluster size
    int clusters = 0;      // persistent clusters: cluster c owns groups c, c + clusters, ...
    int ctas = 0;          // clusters x S
    int ring = 8;          // weight-record ring depth (multiple of 8)
    size_t smem = 0;
    double est_us = 0.0;   // the planner's estimate of a call back to back, in microseconds
};

bool plan_gemv(int64_t m, int64_t k, int64_t n, int sm_count, GemvPlan *plan);
// Modes of the kernel; the same plan serves all three.
constexpr int kGemvModeFma = 0;         // fp32 FMAs on the CUDA cores (m <= 4)
constexpr int kGemvModeRecordMma = 1;   // exact fp16 (q - 8) times X split into fp16 hi + lo, mma.sync
constexpr int kGemvModeW4A8 = 2;        // X coded to int8 per block, integer block dots on mma.sync
cudaError_t launch_gemv(const GemvPlan &plan, const DecodeArgs &args, int mode, cudaStream_t s);

// ------------------------------------------------------------ warp MMA --

struct MmvPlan {
    int NT = 1;            // MMA column tiles: four tokens (hi, lo) each
    int S = 1;             // K slices = cluster size
    int clusters = 0;      // persistent clusters: cluster c owns groups c, c + clusters, ...
    int ctas = 0;          // clusters x S
    int ring = 8;          // weight-record ring depth
    size_t smem = 0;
};

bool plan_mmv(int64_t m, int64_t k, int64_t n, int sm_count, MmvPlan *plan);
cudaError_t launch_mmv(const MmvPlan &plan, const DecodeArgs &args, cudaStream_t s);

// ---------------------------------------------------------------- matvec --

// A set of experts for one launch of the mat-vec: expert i multiplies rows
// row0[i] .. row0[i] + m[i] - 1 of X (m[i] <= 16) by its weights W[i] into
// the same rows of Y. count == 0: a plain call.
constexpr int kMaxExpertSet = 32;
struct ExpertSet {
    int count = 0;
    int row0[kMaxExpertSet] = {};
    int m[kMaxExpertSet] = {};
    const uint8_t *W[kMaxExpertSet] = {};
};

// Weight formats of the mat-vec.
constexpr int kMatvecQ4 = 0;     // Q4_0 records
constexpr int kMatvecInt8 = 1;   // per-output-channel int8 records

struct MatvecPlan {
    int M = 1;             // kernel instance: tokens 1, 2, 4, 8 or 16
    int fmt = kMatvecQ4;   // weight format
    int S = 1;             // K slices = cluster size
    int clusters = 0;      // persistent clusters: cluster c owns groups c, c + clusters, ...
    int ctas = 0;          // clusters x S
    int ring = 8;          // weight-record ring depth (multiple of 8)
    size_t smem = 0;
    double est_us = 0.0;   // the planner's estimate of a call back to back, in microseconds
};

bool plan_matvec(int64_t m, int64_t k, int64_t n, int sm_count, MatvecPlan *plan, int fmt = kMatvecQ4);
cudaError_t launch_matvec(const MatvecPlan &plan, const DecodeArgs &args, cudaStream_t s);
// An expert set: every cluster holds one group of one expert (m = the set's
// largest row count).
bool plan_matvec_experts(int64_t m, int64_t k, int64_t n, int experts, int sm_count, MatvecPlan *plan);
cudaError_t launch_matvec_experts(const MatvecPlan &plan, const DecodeArgs &args, const ExpertSet &set,
                                  cudaStream_t s);
// The library's launch of an expert set on the current device (status code).
int launch_expert_set(const ExpertSet &set, int max_m, const float *X, float *Y, int64_t k, int64_t n,
                      cudaStream_t s);

// ------------------------------------------------ int8 per-channel weights --

// Records of 128 rows x 64 columns of int8 codes (stored as 128 + c), ordered
// [group][pair]; then one fp32 scale per row of the padded rows.
constexpr int kW8GroupRows = 128;
constexpr int kW8RecordBytes = 8192;

inline size_t w8_packed_bytes(int64_t n, int64_t k)
{
    const int64_t groups = ceil_div(n, kW8GroupRows), np = ceil_div(k, kPairK);
    return static_cast<size_t>(groups * np * kW8RecordBytes + groups * kW8GroupRows * 4);
}

cudaError_t launch_w8_quantize(uint8_t *packed, const float *W, int64_t n, int64_t k, cudaStream_t s);
cudaError_t launch_w8_unpack(int8_t *codes, float *scales, const uint8_t *packed, int64_t n, int64_t k, cudaStream_t s);

// --------------------------------------------------------------- prefill --

struct PrefillArgs {
    const uint8_t *W;
    const uint8_t *ximg;    // bf16 X tiles in the swizzled shared-memory image
    float *Y;
    const int32_t *rows;    // slot rows (nullptr: row t)
    int64_t ldy;
    int *status;
    uint64_t wait_ns;
    int m, n, np, groups;
    int T, ts;              // tokens per tile, token tiles
    int ks;                 // K slices: CTAs of a cluster that share one (row tile, token tile)
    int bring;              // X-tile ring depth
    int wring;              // weight-record ring depth (even: two dequantiser sets)
    int astages;            // dequantised weight stages in tensor memory
    int prefetch_w;         // stream W before waiting on the preceding kernel
    unsigned long long *trace_buf;
    unsigned trace_cap, trace_cta;
};

struct XcastArgs {
    const float *X;
    const int32_t *rows;
    int64_t ldx;
    uint8_t *ximg;
    int m, nb, np, T, ts;
};

struct PrefillPlan {
    int T = 0, ts = 0;
    int ks = 1;             // K slices per (row tile, token tile): the cluster size
    int rowtiles = 0;
    int bring = 0, wring = 0, astages = 0;
    size_t smem = 0;
    size_t ws_bytes = 0;    // X image bytes
    double est_us = 0.0;    // the planner's estimate of a call, in microseconds
    size_t ws_ximg_off = 0;
    int xcast_blocks = 0;   // grid of the X cast (grid-stride)
};

bool plan_prefill(int64_t m, int64_t k, int64_t n, int sm_count, PrefillPlan *plan);
cudaError_t launch_prefill(const PrefillPlan &plan, const XcastArgs &xa, const PrefillArgs &pa, cudaStream_t s);

// -------------------------------------------------------------- selftest --

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t s);

} // namespace q4
