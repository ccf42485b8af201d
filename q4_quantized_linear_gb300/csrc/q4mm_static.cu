// q4mm_static.cu -- q4_0_matmul_static_scratch: q4_0_matmul with its scratch
// in a fixed device array of the library instead of any allocation, for
// callers that must not allocate device memory. Only the prefill path
// (m > 16) uses scratch: its bf16 X image (see q4_0_matmul_workspace_size).
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/q4mm.h"
#include "q4mm_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = Q4_STATIC_SCRATCH_BYTES;

// One array per device the library runs on (a __device__ variable exists
// once in every device context that loads the module).
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

} // namespace

extern "C" Q4MM_API int q4_0_matmul_static_scratch(const void *W_packed, const float *X, float *Y,
                                                  int64_t m, int64_t k, int64_t n, q4mm_stream_t stream)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return Q4_ERR_UNSUPPORTED_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return Q4_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return Q4_ERR_UNSUPPORTED_DEVICE;
    // Refuse, before touching anything, a shape whose scratch exceeds the array.
    if (q4_0_matmul_workspace_size(m, k, n) > kStaticScratchBytes) return Q4_ERR_WORKSPACE;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_addr[dev]) {
            // Set-up, once per device, with that device current. The array
            // needs no zeroing: each call writes the part it then reads.
            void *addr = nullptr;
            if (cudaGetSymbolAddress(&addr, g_static_scratch) != cudaSuccess || !addr) {
                cudaGetLastError();
                return Q4_ERR_CUDA;
            }
            g_addr[dev] = addr;
        }
        scratch = g_addr[dev];
    }
    return q4_0_matmul_ws(W_packed, X, Y, m, k, n, scratch, kStaticScratchBytes, stream);
}
