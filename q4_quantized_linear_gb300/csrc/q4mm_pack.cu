// q4mm_pack.cu -- the block repacker and its inverse.
//
// GGUF Q4_0 blocks [n][k/32] x 18 bytes (only 2-byte aligned) are rearranged
// into 576-byte records (16 rows x 2 blocks) so that, in the decode kernel,
// each lane of a warp fetches its whole share of a record -- the scale pair
// it needs and the nibble words that form its tensor-core fragment -- with
// one 8-byte and one 16-byte shared-memory load, and so that a 64-row group
// streams as one contiguous run. The layout is specified in include/q4mm.h.
// Repacking once at load for the kernel's access order is the layout step of
// goinfer ch. 10 ("Making Go fast enough", "Layout, concretely"); the nibble
// words themselves are moved unchanged, so the split-half order survives.
#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {

// One warp per record (group G, pair p, tile t).
__global__ void __launch_bounds__(256) pack_kernel(uint8_t *__restrict__ packed, const uint8_t *__restrict__ blocks,
                                                   int n, int nb, int np, int64_t records)
{
    const int64_t rec = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (rec >= records) return;
    const int lane = threadIdx.x & 31;
    const int t = static_cast<int>(rec & 3);
    const int64_t gp = rec >> 2;            // G * np + p
    const int p = static_cast<int>(gp % np);
    const int64_t G = gp / np;
    uint8_t *out = packed + rec * kRecordBytes;

    // scales: lane L is scale index s = 4g + 2blk + h
    {
        const int g = lane >> 2, blk = (lane >> 1) & 1, h = lane & 1;
        const int64_t row = G * 64 + t * 16 + g + 8 * h;
        const int b = 2 * p + blk;
        uint16_t d = 0;
        if (row < n && b < nb)
            d = *reinterpret_cast<const uint16_t *>(blocks + (row * nb + b) * 18);
        reinterpret_cast<uint16_t *>(out)[lane] = d;
    }
    // nibble words: lane L = 4g + c, words (g, blk0), (g+8, blk0), (g, blk1), (g+8, blk1)
    {
        const int g = lane >> 2, c = lane & 3;
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int blk = i >> 1, h = i & 1;
            const int64_t row = G * 64 + t * 16 + g + 8 * h;
            const int b = 2 * p + blk;
            if (row < n && b < nb) {
                const uint16_t *src = reinterpret_cast<const uint16_t *>(blocks + (row * nb + b) * 18 + 2 + 4 * c);
                w[i] = static_cast<uint32_t>(src[0]) | (static_cast<uint32_t>(src[1]) << 16);
            } else {
                w[i] = 0x88888888u;
            }
        }
        reinterpret_cast<uint4 *>(out + 64)[lane] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// One thread per (row, block): gather the 18 bytes back.
__global__ void __launch_bounds__(256) unpack_kernel(uint8_t *__restrict__ blocks, const uint8_t *__restrict__ packed,
                                                     int n, int nb, int np)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(n) * nb) return;
    const int64_t row = idx / nb;
    const int b = static_cast<int>(idx % nb);
    const int64_t G = row >> 6;
    const int r64 = static_cast<int>(row & 63);
    const int t = r64 >> 4, r16 = r64 & 15, g = r16 & 7, h = r16 >> 3;
    const int p = b >> 1, blk = b & 1;
    const uint8_t *rec = packed + ((G * np + p) * 4 + t) * kRecordBytes;
    uint16_t *dst = reinterpret_cast<uint16_t *>(blocks + idx * 18);
    dst[0] = reinterpret_cast<const uint16_t *>(rec)[4 * g + 2 * blk + h];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const uint32_t w = *reinterpret_cast<const uint32_t *>(rec + 64 + (4 * g + c) * 16 + (2 * blk + h) * 4);
        dst[1 + 2 * c] = static_cast<uint16_t>(w & 0xFFFF);
        dst[2 + 2 * c] = static_cast<uint16_t>(w >> 16);
    }
}

cudaError_t launch_pack(uint8_t *packed, const uint8_t *blocks, int64_t n, int64_t k, cudaStream_t s)
{
    const int nb = static_cast<int>(k / 32);
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int64_t groups = ceil_div(n, kGroupRows);
    const int64_t records = groups * np * 4;
    const int64_t grid = ceil_div(records, 8);
    pack_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(packed, blocks, static_cast<int>(n), nb, np, records);
    return cudaGetLastError();
}

cudaError_t launch_unpack(uint8_t *blocks, const uint8_t *packed, int64_t n, int64_t k, cudaStream_t s)
{
    const int nb = static_cast<int>(k / 32);
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int64_t total = n * nb;
    const int64_t grid = ceil_div(total, 256);
    unpack_kernel<<<static_cast<unsigned>(grid), 256, 0, s>>>(blocks, packed, static_cast<int>(n), nb, np);
    return cudaGetLastError();
}

} // namespace q4
