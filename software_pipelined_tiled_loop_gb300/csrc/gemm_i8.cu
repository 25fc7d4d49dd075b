// Exact int8 GEMM on the tensor cores.
//
// sm_103a has no integer tcgen05.mma kind, so the int8 products run as fp16
// products: every int8 value is exact in fp16 (|v| <= 128 < 2^11), every
// product is exact in fp32 (|a*b| <= 2^14), and a sum of at most KC*64 = 1024
// such products is an integer of magnitude <= 2^24, which fp32 represents
// exactly.  The tensor core therefore accumulates each K-round of 1024
// exactly in TMEM, and the epilogue warps convert each round to int32 and add
// it into registers (int32 arithmetic modulo 2^32), finally writing
// alpha*acc + beta*C modulo 2^32.  Bit-exact against the int64 oracle.
//
// The widening int8 -> fp16 is a separate, HBM-bound pass over A and B into
// stream-ordered scratch (rows padded to 16-byte pitches for TMA).  The CTA
// pair kernels also exist with a register-staged producer that reads the
// int8 operands itself and widens them on the way into the stage ring (the
// LDG-to-register prefetch of the pages, PROD = 1); with one K-tile of loads
// in flight per register buffer it runs at about a third of the TMA ring's
// rate, so the TMA-fed kernel after the widening pass stays the default.
#include <cuda_fp16.h>

#include <vector>

#include "tc_gemm.cuh"
#include "widen.cuh"

namespace pg {

constexpr int kI8ChunkTiles = 16;  // 16 K-tiles of 64 = 1024 products per exact fp32 round

// Each epilogue thread keeps a 128-column row of int32 sums in registers:
// 128-wide tiles use four epilogue warps, 256-wide tiles eight.
// KSUB = 2: stages of 128 K columns; a round is then 8 stages (1024 products).
template <int BN, int STAGES, int CM = 1, int PROD = 0, int S8 = 0, int XG = 1, int KSUB = 1>
using I8Cfg = TcCfg<BN, STAGES, kI8ChunkTiles / KSUB, /*BF16=*/0, /*INT_FOLD=*/true,
                    BN == 256 ? 8 : 4, CM, CM, PROD, S8, XG, KSUB>;

template <int BN, int STAGES, int CM = 1, int PROD = 0, int S8 = 0, int XG = 1, int KSUB = 1>
static KernelInfo info_i8() {
    using Cfg = I8Cfg<BN, STAGES, CM, PROD, S8, XG, KSUB>;
    KernelInfo k = tc_info<Cfg>();
    k.launch_i8 = launch_tc<Cfg, LaunchI8>;
    return k;
}

// The staged producer on the CTA pair: `stages` names the depth of the int8
// ring (the one that covers the memory latency); the fp16 ring behind it is
// F16 deep (it only covers the widening); two transform groups taking
// alternate K-tiles where the ring depth is even, else one.
template <int S8, int F16>
static KernelInfo info_i8_staged() {
    KernelInfo k = info_i8<256, F16, 2, 2, S8, S8 % 2 == 0 ? 2 : 1>();
    k.stages = S8;
    return k;
}

const KernelInfo *i8_kernels(int *count) {
    // the exact-fp16 tcgen05 kernels, then the mma.sync engine's
    static const std::vector<KernelInfo> table = [] {
        std::vector<KernelInfo> t = {
            info_i8<256, 1>(), info_i8<256, 2>(), info_i8<256, 3>(), info_i8<256, 4>(),
            info_i8<128, 2>(), info_i8<128, 3>(), info_i8<128, 4>(), info_i8<128, 5>(),
            info_i8<128, 6>(), info_i8<128, 1>(),
            info_i8<256, 4, 2>(), info_i8<256, 5, 2>(), info_i8<256, 6, 2>(),
            // CTA pair with the register-staged producer (int8 read directly)
            info_i8<256, 4, 2, 1>(), info_i8<256, 5, 2, 1>(), info_i8<256, 6, 2, 1>(),
            // CTA pair with int8 stages by TMA, widened in shared memory
            info_i8_staged<4, 3>(), info_i8_staged<5, 3>(), info_i8_staged<6, 2>(),
            // CTA pair with the widening inside the GEMM (its int8 ring takes
            // the room of a sixth fp16 stage)
            info_i8<256, 4, 2, 3>(), info_i8<256, 5, 2, 3>(),
            // the CTA pair with 128-column stages
            info_i8<256, 2, 2, 0, 0, 1, 2>(), info_i8<256, 3, 2, 0, 0, 1, 2>(),
        };
        int n = 0;
        const KernelInfo *imma = i8_imma_kernels(&n);
        t.insert(t.end(), imma, imma + n);
        return t;
    }();
    *count = static_cast<int>(table.size());
    return table.data();
}

struct WidenJob {
    const int8_t *src;
    long long sld;   // source pitch (elements)
    __half *dst;
    long long dld;   // destination pitch (elements)
    int rows, cols;
    int vec;         // 1: 16-byte vectors (aligned rows, cols % 16 == 0);
                     // 2: the same for rows of fewer than 512 groups of 8,
                     //    walked flat (rows * groups < 2^30, so that a
                     //    thread's 32-bit index cannot overflow)
};

// dst[r][c] = (fp16) src[r][c] for r < rows, c < cols, for the two operands
// (blockIdx.y selects A or B).  Vector path: a block takes kWidenRows rows at
// a time; its threads walk the rows' 8-value groups (an 8-byte load, a
// 16-byte store each; consecutive lanes take consecutive groups, so every
// warp store is 512 contiguous bytes of whole sectors).  Each thread loads
// kWidenGroups groups of every row before converting any, keeping
// kWidenRows * kWidenGroups independent loads in flight: one dependent load
// per thread at a time covers only a fraction of the latency-bandwidth
// product.  Rows of fewer than blockDim * kWidenGroups groups (under 4096
// columns) would leave threads of that walk idle, so there the threads take
// the operand's (row, group) pairs in one flat sequence instead, each
// kWidenFlat of them in flight.  The fp16 output is written back through L2, where the GEMM that
// follows finds most of it.
constexpr int kWidenRows = 2;
constexpr int kWidenGroups = 2;
constexpr int kWidenFlat = 4;

__global__ void __launch_bounds__(256, 6) widen_i8_to_f16_kernel(WidenJob ja, WidenJob jb,
                                                                 uint32_t *zero, int zero_words) {
    // the GEMM's stream-K tickets start at zero (it reads them only after this
    // grid has completed)
    if (blockIdx.x == 0 && blockIdx.y == 0)
        for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero[i] = 0u;
    const WidenJob &j = blockIdx.y == 0 ? ja : jb;
    if (j.rows <= 0 || j.cols <= 0) return;
    if (j.vec == 2) {
        // narrow rows: flat over (row, group), consecutive threads on
        // consecutive groups of a row and then of the next row (rows x
        // groups < 2^30 on this path: 32-bit indices)
        const int groups = j.cols / 8;
        const int total = j.rows * groups;
        const int stride = static_cast<int>(gridDim.x * blockDim.x);
        for (int i0 = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x); i0 < total;
             i0 += stride * kWidenFlat) {
            uint2 w[kWidenFlat];
#pragma unroll
            for (int u = 0; u < kWidenFlat; ++u) {
                const int i = i0 + u * stride;
                if (i < total) {
                    const int r = i / groups;
                    w[u] = __ldg(reinterpret_cast<const uint2 *>(j.src + r * j.sld) + (i - r * groups));
                }
            }
#pragma unroll
            for (int u = 0; u < kWidenFlat; ++u) {
                const int i = i0 + u * stride;
                if (i < total) {
                    const int r = i / groups;
                    __half2 o[4];
                    widen4(w[u].x, o[0], o[1]);
                    widen4(w[u].y, o[2], o[3]);
                    reinterpret_cast<uint4 *>(j.dst + r * j.dld)[i - r * groups] =
                        *reinterpret_cast<const uint4 *>(o);
                }
            }
        }
    } else if (j.vec) {
        const int groups = j.cols / 8;  // cols % 16 == 0 on this path
        const int step = static_cast<int>(blockDim.x) * kWidenGroups;
        for (long long r0 = static_cast<long long>(blockIdx.x) * kWidenRows; r0 < j.rows;
             r0 += static_cast<long long>(gridDim.x) * kWidenRows) {
            const int nr = j.rows - r0 < kWidenRows ? static_cast<int>(j.rows - r0) : kWidenRows;
            for (int c0 = threadIdx.x; c0 < groups; c0 += step) {
                uint2 w[kWidenRows][kWidenGroups];
#pragma unroll
                for (int u = 0; u < kWidenRows; ++u)
#pragma unroll
                    for (int h = 0; h < kWidenGroups; ++h) {
                        const int c = c0 + h * static_cast<int>(blockDim.x);
                        if (u < nr && c < groups)
                            w[u][h] = __ldg(reinterpret_cast<const uint2 *>(j.src + (r0 + u) * j.sld) + c);
                    }
#pragma unroll
                for (int u = 0; u < kWidenRows; ++u)
#pragma unroll
                    for (int h = 0; h < kWidenGroups; ++h) {
                        const int c = c0 + h * static_cast<int>(blockDim.x);
                        if (u < nr && c < groups) {
                            __half2 o[4];
                            widen4(w[u][h].x, o[0], o[1]);
                            widen4(w[u][h].y, o[2], o[3]);
                            reinterpret_cast<uint4 *>(j.dst + (r0 + u) * j.dld)[c] =
                                *reinterpret_cast<const uint4 *>(o);
                        }
                    }
            }
        }
    } else {
        const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
        const long long t0 = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x;
        const long long total = static_cast<long long>(j.rows) * j.cols;
        for (long long i = t0; i < total; i += stride) {
            const long long r = i / j.cols, c = i - r * j.cols;
            j.dst[r * j.dld + c] = __short2half_rn(static_cast<short>(j.src[r * j.sld + c]));
        }
    }
    grid_launch_dependents();  // this block's share is written
}

static WidenJob make_job(const int8_t *src, long long sld, void *dst, long long dld, int rows,
                         int cols) {
    WidenJob j{src, sld, static_cast<__half *>(dst), dld, rows, cols, 0};
    j.vec = ((reinterpret_cast<uintptr_t>(src) & 15u) == 0 && sld % 16 == 0 &&
             (reinterpret_cast<uintptr_t>(dst) & 15u) == 0 && dld % 8 == 0 && cols % 16 == 0)
                ? 1
                : 0;
    if (j.vec && cols / 8 < 256 * kWidenGroups &&
        static_cast<long long>(rows) * (cols / 8) < (1LL << 30))
        j.vec = 2;
    return j;
}

cudaError_t launch_widen_i8_pair(const int8_t *a, long long lda, void *a_dst, long long a_dld,
                                 int a_rows, int a_cols, const int8_t *b, long long ldb,
                                 void *b_dst, long long b_dld, int b_rows, int b_cols,
                                 uint32_t *zero, int zero_words, int sm_count,
                                 cudaStream_t stream) {
    const WidenJob ja = make_job(a, lda, a_dst, a_dld, a_rows, a_cols);
    const WidenJob jb = make_job(b, ldb, b_dst, b_dld, b_rows, b_cols);
    // vector path: one block per kWidenRows rows; scalar path: about four
    // values per thread
    auto blocks_for = [](const WidenJob &j) -> long long {
        if (!j.vec) return (static_cast<long long>(j.rows) * j.cols + 1023) / 1024;
        if (j.vec == 2)  // flat walk: kWidenFlat groups a thread
            return (static_cast<long long>(j.rows) * (j.cols / 8) + 256 * kWidenFlat - 1) /
                   (256 * kWidenFlat);
        return (static_cast<long long>(j.rows) + kWidenRows - 1) / kWidenRows;
    };
    long long blocks = blocks_for(ja) > blocks_for(jb) ? blocks_for(ja) : blocks_for(jb);
    const long long cap = static_cast<long long>(sm_count) * 16;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    widen_i8_to_f16_kernel<<<dim3(static_cast<unsigned>(blocks), 2), 256, 0, stream>>>(ja, jb, zero,
                                                                                 zero_words);
    return cudaGetLastError();
}

}  // namespace pg
