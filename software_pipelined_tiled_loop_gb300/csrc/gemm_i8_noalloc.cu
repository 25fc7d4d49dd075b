// gemm_i8_noalloc: the exact int8 GEMM without any device allocation.
//
// For callers that cannot let the library allocate device memory (their own
// allocator owns the GPU's memory, a fixed memory budget, or a path where an
// allocation call is not allowed or could block), the int8 operands are
// widened to fp16 into one file-scope device array instead of stream-ordered
// scratch.  The array is PGEMM_NOALLOC_SCRATCH_BYTES (32 MiB) and every GPU
// that loads the library holds it until the process exits.
#include <cuda_runtime.h>

#include <mutex>

#include "pgemm.h"
#include "kernels.h"

namespace {

// The widened A and B of the most recent call (shared by all calls).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PGEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per
// device.  In host code the array's name stands for a host-side shadow, not
// for device memory, so the kernels are given this address instead.  The
// GEMM calls this only after it has checked the arguments and set up the
// device (an sm_103 device is current), and only when it needs the array.
pgemm_status scratch_address(void **out, long long *bytes) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PGEMM_ERR_UNSUPPORTED_DEVICE;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();  // leave no error behind for the caller's next check
            return PGEMM_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    *bytes = static_cast<long long>(PGEMM_NOALLOC_SCRATCH_BYTES);
    return PGEMM_OK;
}

}  // namespace

extern "C" pgemm_status gemm_i8_noalloc(int M, int N, int K, int32_t alpha, const int8_t *A,
                                        const int8_t *B, int32_t beta, int32_t *C,
                                        pgemm_stream_t stream) {
    return pg::gemm_i8_fixed_scratch(M, N, K, alpha, A, B, beta, C, scratch_address, stream);
}
