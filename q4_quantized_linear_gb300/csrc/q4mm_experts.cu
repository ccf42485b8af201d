// q4mm_experts.cu -- the expert-grouped product (host code: it launches only
// through q4_0_matmul).
//
// golem-server, "Several conversations, in one pass": a mixture answers a
// single column by reading the matrices that column was routed to, and a
// prompt by reading each expert once for the columns that chose it; the two
// costs cross near thirty-two columns. Here X's rows come grouped by expert
// (offsets[e] .. offsets[e+1] - 1 for expert e) and each expert's weights are
// read once for its rows: q4_0_matmul runs the decode kernels for up to 16
// rows and the tensor-core GEMM above, so a handful of rows costs a weight
// read and a prompt-sized group a tiled product.
#include <cstdint>

#include "../../include/q4mm.h"

namespace {

bool aligned_to(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

} // namespace

extern "C" Q4MM_API int q4_0_matmul_experts(const void *const *W_packed, int64_t n_experts, const int64_t *offsets,
                                            const float *X, float *Y, int64_t k, int64_t n, q4mm_stream_t stream)
{
    // every argument is checked before anything is launched
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
    for (int64_t e = 0; e < n_experts; ++e) {
        const int64_t r0 = offsets[e], m = offsets[e + 1] - offsets[e];
        if (m == 0) continue;
        // row r0 of X starts on a 16-byte boundary: k is a multiple of 32
        const int rc = q4_0_matmul(W_packed[e], X + r0 * k, Y + r0 * n, m, k, n, stream);
        if (rc != Q4_OK) return rc;
    }
    return Q4_OK;
}
