// q4mm_pack.cu -- the block repacker and its inverse.
//
// GGUF Q4_0 blocks [n][k/32] x 18 bytes (only 2-byte aligned) are rearranged
// into 4608-byte records of 128 rows x 2 blocks: first every row's pair of
// fp16 scales, then every row's 16 nibble bytes of the first block, then of
// the second. A kernel thread that owns one row of a 128-row tile reads its
// share of a record with one 4-byte and two 16-byte shared-memory loads,
// conflict-free across the warp, and a group's pairs stream as one contiguous
// run. The nibble bytes are moved unchanged, so the split-half order of the
// format survives. Repacking once at load for the kernel's access order is
// the layout step of goinfer ch. 10 ("Making Go fast enough", "Layout,
// concretely"). The layout is specified in include/q4mm.h.
#include "q4mm_device.cuh"
#include "q4mm_internal.h"

namespace q4 {

// One thread per (group, pair, row).
__global__ void __launch_bounds__(256) pack_kernel(uint8_t *__restrict__ packed, const uint8_t *__restrict__ blocks,
                                                   int n, int nb, int np, int64_t total)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= total) return;
    const int r = static_cast<int>(idx & 127);
    const int64_t gp = idx >> 7;             // G * np + p
    const int p = static_cast<int>(gp % np);
    const int64_t G = gp / np;
    const int64_t row = G * kGroupRows + r;
    uint8_t *rec = packed + gp * kRecordBytes;
    uint32_t dpair = 0;
#pragma unroll
    for (int blk = 0; blk < 2; ++blk) {
        const int b = 2 * p + blk;
        uint32_t w[4] = {0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u};
        if (row < n && b < nb) {
            const uint16_t *src = reinterpret_cast<const uint16_t *>(blocks + (row * nb + b) * 18);
            dpair |= static_cast<uint32_t>(src[0]) << (16 * blk);
#pragma unroll
            for (int c = 0; c < 4; ++c)
                w[c] = static_cast<uint32_t>(src[1 + 2 * c]) | (static_cast<uint32_t>(src[2 + 2 * c]) << 16);
        }
        *reinterpret_cast<uint4 *>(rec + (blk ? kRecQs1Off : kRecQs0Off) + 16 * r) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    *reinterpret_cast<uint32_t *>(rec + kRecScaleOff + 4 * r) = dpair;
}

// One thread per (row, block): gather the 18 bytes back.
__global__ void __launch_bounds__(256) unpack_kernel(uint8_t *__restrict__ blocks, const uint8_t *__restrict__ packed,
                                                     int n, int nb, int np)
{
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (idx >= static_cast<int64_t>(n) * nb) return;
    const int64_t row = idx / nb;
    const int b = static_cast<int>(idx % nb);
    const int64_t G = row / kGroupRows;
    const int r = static_cast<int>(row % kGroupRows);
    const int p = b >> 1, blk = b & 1;
    const uint8_t *rec = packed + (G * np + p) * kRecordBytes;
    uint16_t *dst = reinterpret_cast<uint16_t *>(blocks + idx * 18);
    dst[0] = reinterpret_cast<const uint16_t *>(rec + kRecScaleOff + 4 * r)[blk];
    const uint4 q = *reinterpret_cast<const uint4 *>(rec + (blk ? kRecQs1Off : kRecQs0Off) + 16 * r);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        dst[1 + 2 * c] = static_cast<uint16_t>(w[c] & 0xFFFF);
        dst[2 + 2 * c] = static_cast<uint16_t>(w[c] >> 16);
    }
}

cudaError_t launch_pack(uint8_t *packed, const uint8_t *blocks, int64_t n, int64_t k, cudaStream_t s)
{
    const int nb = static_cast<int>(k / 32);
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int64_t total = ceil_div(n, kGroupRows) * np * kGroupRows;
    pack_kernel<<<static_cast<unsigned>(ceil_div(total, 256)), 256, 0, s>>>(packed, blocks, static_cast<int>(n), nb,
                                                                             np, total);
    return cudaGetLastError();
}

cudaError_t launch_unpack(uint8_t *blocks, const uint8_t *packed, int64_t n, int64_t k, cudaStream_t s)
{
    const int nb = static_cast<int>(k / 32);
    const int np = static_cast<int>(ceil_div(k, kPairK));
    const int64_t total = n * nb;
    unpack_kernel<<<static_cast<unsigned>(ceil_div(total, 256)), 256, 0, s>>>(blocks, packed, static_cast<int>(n), nb,
                                                                               np);
    return cudaGetLastError();
}

} // namespace q4
