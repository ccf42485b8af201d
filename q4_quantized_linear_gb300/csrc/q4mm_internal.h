// q4mm_internal.h -- host-side interfaces between the translation units of
// libq4mm (argument structs passed by value to the kernels, planners and
// launchers). Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace q4 {

constexpr int kRecordBytes = 576;     // one 16-row tile x one pair of blocks
constexpr int kPairBytes = 4 * 576;   // one 64-row group x one pair of blocks
constexpr int kGroupRows = 64;
constexpr int kPairK = 64;
// 227 KB per CTA on sm_100-family parts, less room for a kernel's static
// shared variables; plans never ask for more dynamic shared memory than this.
constexpr size_t kSmemOptIn = 232448 - 256;
constexpr size_t kSmemPerSM = 233472; // 228 KB per SM
// Split-K counters of the decode kernel live in the first kDecodeCounterSlots
// words of every workspace (one per 64-row group), so plans with K slices are
// limited to n <= 64 * kDecodeCounterSlots rows. Every plan that uses a
// workspace keeps this region in place (and only the decode kernel writes it,
// leaving it zero), so calls of any shape can share one workspace.
constexpr int64_t kDecodeCounterSlots = 65536;
constexpr size_t kWsCounterBytes = kDecodeCounterSlots * 4;

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

// Launch helper: PDL-enabled launch on `stream`.
cudaError_t launch_pdl(const void *func, dim3 grid, dim3 block, size_t smem, cudaStream_t stream, void **args);

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
    float *partials;       // [S][m][groups*64] when S > 1
    unsigned *counters;    // [groups] when S > 1
    int *status;
    uint64_t wait_ns;
    int m, n, nb, np, groups;
    int S, pbase, prem;    // K slices: slice s has pbase + (s < prem) pairs
    int stages;            // ring depth per warp
    int xs_bytes;          // shared bytes reserved for the staged X slice
    int prefetch_w;        // stream W before waiting on the preceding kernel
};

struct DecodePlan {
    int NT = 1;            // n8 token tiles (1: m <= 8, 2: m <= 16)
    int S = 1;
    int pbase = 0, prem = 0;
    int stages = 8;
    int ctas = 0;          // grid size (multiple of S)
    int xs_bytes = 0;
    size_t smem = 0;
    size_t ws_bytes = 0;   // workspace: partials + counters
    size_t ws_partials_off = 0, ws_counters_off = 0;
};

bool plan_decode(int64_t m, int64_t k, int64_t n, int sm_count, DecodePlan *plan);
cudaError_t launch_decode(const DecodePlan &plan, const DecodeArgs &args, cudaStream_t s);
size_t decode_smem_bytes(int NT, int P, int stages);

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
    int rb, ra, rw;         // ring depths: X tiles, dequantised W tiles, raw W records
    int tmem_cols;
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
    int rowtiles = 0;
    int rb = 0, ra = 0, rw = 0;
    int tmem_cols = 0;
    size_t smem = 0;
    size_t ws_bytes = 0;    // counter region + X image bytes
    size_t ws_ximg_off = 0;
};

bool plan_prefill(int64_t m, int64_t k, int64_t n, int sm_count, PrefillPlan *plan);
cudaError_t launch_prefill(const PrefillPlan &plan, const XcastArgs &xa, const PrefillArgs &pa, cudaStream_t s);

// -------------------------------------------------------------- selftest --

cudaError_t launch_wait_selftest(int *status, uint64_t limit_ns, cudaStream_t s);

} // namespace q4
