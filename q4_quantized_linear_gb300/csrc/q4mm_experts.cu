// q4mm_experts.cu -- the expert-grouped product (host code: it launches only
// through q4_0_matmul).
//
// golem-server, "Several conversations, in one pass" (mixture layers): the
// cost of a mixture layer is set by which expert matrices are read, once per
// pass, for the columns routed to them, with the page's measured switch from
// per-column to per-expert work at about thirty-two columns. Here X's rows
// come grouped by expert (offsets[e] .. offsets[e+1] - 1 for expert e) and
// each expert's weights are read once for its rows (twice for 17..32 rows):
//   up to 32 rows: the decode mat-vec, in pieces of at most 16 rows; pieces
//     of the same mat-vec instance (1, 2, 4, 8 or 16 token columns) share one
//     launch, a cluster per 128-row group of an expert's piece;
//   more rows: the tensor-core GEMM, one call per expert.
// The switch at 32 rows is measured on GB300 for a 9728 x 2560 expert: the
// mat-vec in pieces of 16 rows is faster up to 32 rows (19.8 us at 17 rows
// and 22.4 us at 32 against 24.4-24.6 us for the GEMM), the GEMM from 48 rows
// on (24.8 us against 33.6 us).
#include <algorithm>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/q4mm.h"
#include "q4mm_internal.h"

namespace {

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

} // namespace

extern "C" Q4MM_API int q4_0_matmul_experts(const void *const *W_packed, int64_t n_experts, const int64_t *offsets,
                                            const float *X, float *Y, int64_t k, int64_t n, q4mm_stream_t stream)
{
    // the arguments are checked before anything is launched; a group refused
    // later (its plan or the library workspace) leaves earlier groups written
    if (!W_packed || !offsets || !X || !Y || n_experts < 1 || n_experts > (int64_t(1) << 20) || n < 1 || k < 32 ||
        k % 32 != 0 || n > (int64_t(1) << 31) || k > (int64_t(1) << 31))
        return Q4_ERR_INVALID_ARG;
    if (offsets[0] != 0) return Q4_ERR_INVALID_ARG;
    for (int64_t e = 0; e < n_experts; ++e) {
        if (offsets[e + 1] < offsets[e] || offsets[e + 1] > (int64_t(1) << 24)) return Q4_ERR_INVALID_ARG;
        if (offsets[e + 1] > offsets[e]) {
            if (!W_packed[e]) return Q4_ERR_INVALID_ARG;
            if (!aligned_to(W_packed[e], 16)) return Q4_ERR_ALIGNMENT;
        }
    }
    if (!aligned_to(X, 16) || !aligned_to(Y, 4)) return Q4_ERR_ALIGNMENT;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Pieces of up to 16 rows of the experts with up to kMatvecRows rows, set
    // by set: one launch of the mat-vec per instance and per 32 pieces.
    constexpr int64_t kMatvecRows = 32;
    constexpr int kInstances[5] = {1, 2, 4, 8, 16};
    int rc = Q4_OK;
    for (int inst = 0; inst < 5 && rc == Q4_OK; ++inst) {
        const int lo = inst == 0 ? 1 : kInstances[inst - 1] + 1, hi = kInstances[inst];
        q4::ExpertSet set;
        int max_m = 0;
        auto flush = [&]() -> int {
            if (set.count == 0) return Q4_OK;
            int r = q4::launch_expert_set(set, max_m, X, Y, k, n, s);
            if (r == Q4_ERR_INVALID_ARG)   // no plan for this shape: piece by piece
                for (int i = 0; i < set.count && (r == Q4_ERR_INVALID_ARG || r == Q4_OK); ++i)
                    r = q4_0_matmul(set.W[i], X + static_cast<int64_t>(set.row0[i]) * k,
                                    Y + static_cast<int64_t>(set.row0[i]) * n, set.m[i], k, n, stream);
            set.count = 0;
            max_m = 0;
            return r;
        };
        for (int64_t e = 0; e < n_experts && rc == Q4_OK; ++e) {
            const int64_t m = offsets[e + 1] - offsets[e];
            if (m == 0 || m > kMatvecRows) continue;
            for (int64_t r0 = offsets[e]; r0 < offsets[e + 1] && rc == Q4_OK; r0 += 16) {
                const int pm = static_cast<int>(std::min<int64_t>(16, offsets[e + 1] - r0));
                if (pm < lo || pm > hi) continue;
                set.row0[set.count] = static_cast<int>(r0);
                set.m[set.count] = pm;
                set.W[set.count] = static_cast<const uint8_t *>(W_packed[e]);
                ++set.count;
                max_m = std::max(max_m, pm);
                if (set.count == q4::kMaxExpertSet) rc = flush();
            }
        }
        if (rc == Q4_OK) rc = flush();
    }
    if (rc != Q4_OK) return rc;
    for (int64_t e = 0; e < n_experts; ++e) {
        const int64_t r0 = offsets[e], m = offsets[e + 1] - offsets[e];
        if (m <= kMatvecRows) continue;
        // row r0 of X starts on a 16-byte boundary: k is a multiple of 32
        rc = q4_0_matmul(W_packed[e], X + r0 * k, Y + r0 * n, m, k, n, stream);
        if (rc != Q4_OK) return rc;
    }
    return Q4_OK;
}
