// Exact int8 GEMM on the tensor cores.
//
// sm_103a has no integer tcgen05.mma kind, so the int8 products run as fp16
// products: every int8 value is exact in fp16 (|v| <= 128 < 2^11), every
// product is exact in fp32 (|a*b| <= 2^14), and a sum of at most KC*64 = 256
// such products stays an integer of magnitude <= 2^22, exact in fp32.  The
// tensor core therefore accumulates each K-chunk of 256 exactly in TMEM, and
// the epilogue warps convert each chunk to int32 and add it into registers
// (int32 arithmetic modulo 2^32), finally writing alpha*acc + beta*C modulo
// 2^32.  Bit-exact against the int64 oracle.
//
// The widening int8 -> fp16 is a separate, HBM-bound pass over A and B into
// stream-ordered scratch (rows padded to 16-byte pitches for TMA); widening
// inside the GEMM would put about three times the tensor core's own operand
// traffic through shared memory.
#include <cuda_fp16.h>

#include "tc_gemm.cuh"

namespace pg {

constexpr int kI8ChunkTiles = 4;  // 4 K-tiles of 64 = 256 products per exact fp32 round

// Each epilogue thread keeps a 128-column row of int32 sums in registers:
// 128-wide tiles use four epilogue warps, 256-wide tiles eight.
template <int BN, int STAGES>
using I8Cfg = TcCfg<BN, STAGES, kI8ChunkTiles, /*BF16=*/0, /*INT_FOLD=*/true, BN == 256 ? 8 : 4>;

template <int BN, int STAGES>
static KernelInfo info_i8() {
    KernelInfo k = tc_info<I8Cfg<BN, STAGES>>();
    k.launch_i8 = launch_tc<I8Cfg<BN, STAGES>, LaunchI8>;
    return k;
}

const KernelInfo *i8_kernels(int *count) {
    static const KernelInfo table[] = {
        info_i8<256, 1>(), info_i8<256, 2>(), info_i8<256, 3>(), info_i8<256, 4>(),
        info_i8<128, 2>(), info_i8<128, 3>(), info_i8<128, 4>(), info_i8<128, 5>(),
        info_i8<128, 6>(), info_i8<128, 1>(),
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

// dst[r][c] = (fp16) src[r][c] for r < rows, c < cols; src pitch `sld`
// elements, dst pitch `dld` elements.  16 values per thread when both rows
// are 16-byte aligned, else one value per thread.
__global__ void widen_i8_to_f16_kernel(const int8_t *__restrict__ src, long long sld,
                                       __half *__restrict__ dst, long long dld, int rows,
                                       int cols, int vec) {
    const long long per_row = vec ? (cols + 15) / 16 : cols;
    const long long total = per_row * rows;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
         idx < total; idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long r = idx / per_row;
        const long long cc = idx - r * per_row;
        if (vec) {
            const int c0 = static_cast<int>(cc * 16);
            const int8_t *s = src + r * sld + c0;
            __half *d = dst + r * dld + c0;
            if (c0 + 16 <= cols) {
                const int4 v = *reinterpret_cast<const int4 *>(s);
                const int8_t *b = reinterpret_cast<const int8_t *>(&v);
                __align__(16) __half h[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) h[e] = __short2half_rn(static_cast<short>(b[e]));
                reinterpret_cast<int4 *>(d)[0] = reinterpret_cast<const int4 *>(h)[0];
                reinterpret_cast<int4 *>(d)[1] = reinterpret_cast<const int4 *>(h)[1];
            } else {
                for (int e = 0; c0 + e < cols; ++e) d[e] = __short2half_rn(static_cast<short>(s[e]));
            }
        } else {
            dst[r * dld + cc] = __short2half_rn(static_cast<short>(src[r * sld + cc]));
        }
    }
}

cudaError_t launch_widen_i8(const int8_t *src, long long sld, void *dst, long long dld, int rows,
                            int cols, int sm_count, cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && sld % 16 == 0 &&
                     (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && dld % 8 == 0)
                        ? 1
                        : 0;
    const long long per_row = vec ? (cols + 15) / 16 : cols;
    const long long total = per_row * rows;
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    widen_i8_to_f16_kernel<<<static_cast<int>(blocks), 256, 0, stream>>>(
        src, sld, static_cast<__half *>(dst), dld, rows, cols, vec);
    return cudaGetLastError();
}

}  // namespace pg
