// q4mm_w8.cu -- per-output-channel int8 weights (rembed "Architecture",
// "int8 quantization", the weight-only form: dense weights quantised once at
// load to symmetric int8 with one scale per output channel, dequantised in
// registers, the channel's scale applied once in the epilogue). This file
// holds the quantiser that writes the packed int8 layout and its inverse; the
// products run in the mat-vec kernels (q4mm_matvec.cu).
//
// Quantisation of row j of W [n x k] (fp32), every step one IEEE fp32
// operation: amax = max |w|; scale s = amax / 127; code
// c = round-half-even(w * (127 / amax)), so |c| <= 127; a row with amax = 0
// has codes 0 and s = 0.
//
// Packed layout: records of 128 rows x 64 columns (8192 bytes), ordered
// [group of 128 rows][pair of 32-column blocks] like the Q4_0 records; byte
// 64 r + e of a record is c + 128 for row r, column 64 p + e (codes stored
// with the sign bit flipped, so that a byte is the unsigned 128 + c the
// kernels OR into an fp16 pattern). Rows past n and columns past k hold
// c = 0. After the records, one fp32 scale per row, groups x 128 of them
// (0 for rows past n).
#include <cuda_runtime.h>

#include "q4mm_internal.h"

namespace q4 {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerCta = kThreads / 32;   // one warp per row

// One warp per row of the padded layout: the row's largest |w| by a warp
// maximum, then the codes, four columns per lane per step.
__global__ void __launch_bounds__(kThreads) w8_quantize_kernel(uint8_t *packed, const float *W, int64_t n, int64_t k,
                                                                 int np, int groups)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp;
    if (j >= static_cast<int64_t>(groups) * kW8GroupRows) return;
    const int64_t G = j / kW8GroupRows;
    const int r = static_cast<int>(j - G * kW8GroupRows);
    const int64_t kp = static_cast<int64_t>(np) * kPairK;   // padded columns
    float *scales = reinterpret_cast<float *>(packed + static_cast<size_t>(groups) * np * kW8RecordBytes);
    const float *wr = W + j * k;
    unsigned mb = 0u;
    if (j < n)
        for (int64_t c = 4 * lane; c < k; c += 128) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(wr + c));
            mb = max(mb, max(max(__float_as_uint(v.x) & 0x7FFFFFFFu, __float_as_uint(v.y) & 0x7FFFFFFFu),
                             max(__float_as_uint(v.z) & 0x7FFFFFFFu, __float_as_uint(v.w) & 0x7FFFFFFFu)));
        }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mb = max(mb, __shfl_xor_sync(0xFFFFFFFFu, mb, o));
    const float amax = __uint_as_float(mb);
    const float inv = mb != 0u ? __fdiv_rn(127.0f, amax) : 0.0f;
    if (lane == 0) scales[j] = __fdiv_rn(amax, 127.0f);
    for (int64_t c = 4 * lane; c < kp; c += 128) {
        uint32_t word = 0x80808080u;                        // c = 0 past k and past n
        if (j < n && c < k) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(wr + c));
            const float f[4] = {v.x, v.y, v.z, v.w};
            word = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int code = __float2int_rn(__fmul_rn(f[i], inv));
                word |= static_cast<uint32_t>((code + 128) & 0xFF) << (8 * i);
            }
        }
        const int64_t p = c / kPairK;
        const int e = static_cast<int>(c - p * kPairK);
        uint8_t *rec = packed + static_cast<size_t>(G * np + p) * kW8RecordBytes;
        *reinterpret_cast<uint32_t *>(rec + r * kPairK + e) = word;
    }
}

// The inverse: codes int8 [n x k] and scales fp32 [n] from the packed layout.
__global__ void __launch_bounds__(kThreads) w8_unpack_kernel(int8_t *codes, float *scales, const uint8_t *packed,
                                                               int64_t n, int64_t k, int np, int groups)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t j = static_cast<int64_t>(blockIdx.x) * kRowsPerCta + warp;
    if (j >= n) return;
    const int64_t G = j / kW8GroupRows;
    const int r = static_cast<int>(j - G * kW8GroupRows);
    const float *sc = reinterpret_cast<const float *>(packed + static_cast<size_t>(groups) * np * kW8RecordBytes);
    if (lane == 0) scales[j] = sc[j];
    for (int64_t c = 4 * lane; c < k; c += 128) {
        const int64_t p = c / kPairK;
        const int e = static_cast<int>(c - p * kPairK);
        const uint32_t word =
            *reinterpret_cast<const uint32_t *>(packed + static_cast<size_t>(G * np + p) * kW8RecordBytes + r * kPairK + e);
        *reinterpret_cast<uint32_t *>(codes + j * k + c) = word ^ 0x80808080u;
    }
}

} // namespace

cudaError_t launch_w8_quantize(uint8_t *packed, const float *W, int64_t n, int64_t k, cudaStream_t s)
{
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int groups = static_cast<int>(ceil_div(n, kW8GroupRows));
    const int64_t rows = static_cast<int64_t>(groups) * kW8GroupRows;
    w8_quantize_kernel<<<static_cast<unsigned>(ceil_div(rows, kRowsPerCta)), kThreads, 0, s>>>(packed, W, n, k, np,
                                                                                                groups);
    return cudaGetLastError();
}

cudaError_t launch_w8_unpack(int8_t *codes, float *scales, const uint8_t *packed, int64_t n, int64_t k, cudaStream_t s)
{
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int groups = static_cast<int>(ceil_div(n, kW8GroupRows));
    w8_unpack_kernel<<<static_cast<unsigned>(ceil_div(n, kRowsPerCta)), kThreads, 0, s>>>(codes, scales, packed, n, k,
                                                                                           np, groups);
    return cudaGetLastError();
}

} // namespace q4
