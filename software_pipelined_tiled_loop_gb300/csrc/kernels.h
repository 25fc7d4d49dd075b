// Host-side interface between the dispatch layer (api.cu) and the kernel
// translation units: one KernelInfo per compiled (tile, stages) instance.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pgemm.h"
#include "ptx.cuh"

namespace pg {

// Shared memory per SM on sm_100-family GPUs and the per-block reservation.
constexpr int kSmemPerSm = 233472;
constexpr int kSmemReservedPerBlock = 1024;

// Dynamic shared memory to request so that (a) `used` bytes fit and (b) no
// more than `max_blocks` blocks can be resident on one SM.
constexpr int smem_request(int used, int max_blocks) {
    const int cap = kSmemPerSm / (max_blocks + 1) - kSmemReservedPerBlock + 1;
    return used > cap ? used : cap;
}

// How a call's output tiles are spread over a persistent grid: `slots`
// units run at once (resident blocks, or CTA pairs); the `split_tiles`
// leftover tiles of a partial last wave have their K-iterations dealt out to
// `sk_slots` slots (stream-K), at most `parts` slots sharing one tile.
// partials / counters: the meeting area of those pieces (counters zeroed
// before the launch).
struct TileSchedule {
    long long tiles = 0;
    int slots = 0;
    long long split_tiles = 0;
    // leftover tiles run as two half-width units each instead (no exchange)
    long long half_tiles = 0;
    int sk_slots = 0;
    int parts = 1;
    long long partial_words = 0, counter_words = 0;
    uint32_t *partials = nullptr;
    uint32_t *counters = nullptr;
};

struct LaunchCommon {
    int M, N, K;
    long long ldc;
    int group_m;        // raster group (0 = kernel default)
    int sm_count;
    int blocks_per_sm;  // resident blocks per SM for this kernel (occupancy query)
    const CUtensorMap *tmap_a;
    const CUtensorMap *tmap_b;
    const CUtensorMap *tmap_c;  // C as a 32 x 32-box, 128-byte-swizzled map, or nullptr
    // in-kernel widening: the caller's int8 A (128 x 64-byte boxes) and B
    // (64 x 128-byte boxes), unswizzled; nullptr otherwise
    const CUtensorMap *tmap_a8, *tmap_b8;
    bool after_prepass;         // a widening / repack kernel of this call precedes the GEMM
    KernelCtx ctx;
    TileSchedule sched;         // persistent kernels only
    // The operands as the kernels read them (after any repack / widening):
    // base pointers and pitches in elements, rows 16-byte aligned.  Used by
    // kernels whose threads load the operands themselves.
    const void *a_ptr, *b_ptr;
    long long lda, ldb;
    // In-kernel widening: the caller's int8 operands (pitches in bytes), the
    // destination being a_ptr / b_ptr above, and the per-chunk counters.
    const void *widen_src_a, *widen_src_b;
    long long widen_lda, widen_ldb;
    uint32_t *widen_ready;
};

struct LaunchBf16 : LaunchCommon {
    float alpha, beta;
    float *C;
};

struct LaunchF32 : LaunchCommon {
    float alpha, beta;
    float *C;
};

struct LaunchI8 : LaunchCommon {
    int32_t alpha, beta;
    int32_t *C;
};

struct KernelInfo {
    int bm = 0, bn = 0, bk = 0, stages = 0;
    int threads = 0;
    int smem_bytes = 0;
    // Operand boxes the tensor maps must be encoded with (elements, x = innermost).
    int a_box_x = 0, a_box_y = 0, b_box_x = 0, b_box_y = 0;
    bool a_swizzle128 = true, b_swizzle128 = true;
    bool c_tma = false;  // the kernel can store C through a tensor map
    int producer = PGEMM_PRODUCER_TMA;
    int engine = PGEMM_ENGINE_DEFAULT;
    // Persistent kernels: K-tiles per accumulation round (0 = all of K) and
    // the number of schedule slots (resident CTAs or CTA pairs) for a
    // launch; nullptr for kernels with one block per tile.
    int kc = 0;
    int slabs_per_tile = 0;  // epilogue warps per tile (all CTAs of a pair)
    // FFMA kernels: the stream-K pieces run as a second grid (aux_func)
    // behind the whole tiles, one ticket per leftover tile and no default cap
    // on pieces; the tensor-core kernels run them in-kernel, two counters per
    // tile and epilogue warp, at most two pieces a tile by default.
    bool stream_k = false;
    // The kernel can run a tile as two half-width units (BN = 256 tensor-core
    // kernels fed by TMA): the leftover tiles of a partial last wave are then
    // cut along N, into 2R units on as many slots, rather than along K.
    bool halves = false;
    cudaError_t (*schedule_slots)(const LaunchCommon &, int *slots) = nullptr;
    const void *func = nullptr;
    const void *aux_func = nullptr;  // a second kernel of the same launch (same attributes)
    cudaError_t (*launch_bf16)(const LaunchBf16 &, cudaStream_t) = nullptr;
    cudaError_t (*launch_f32)(const LaunchF32 &, cudaStream_t) = nullptr;
    cudaError_t (*launch_i8)(const LaunchI8 &, cudaStream_t) = nullptr;
};

const KernelInfo *bf16_kernels(int *count);
const KernelInfo *f32_kernels(int *count);
const KernelInfo *i8_kernels(int *count);
const KernelInfo *i8_imma_kernels(int *count);  // gemm_i8_imma.cu (listed by i8_kernels)

}  // namespace pg

namespace pg {
// int8 -> fp16 widening of A and B in one launch (gemm_i8.cu); destination
// rows have pitches a_dld / b_dld elements.
cudaError_t launch_widen_i8_pair(const int8_t *a, long long lda, void *a_dst, long long a_dld,
                                 int a_rows, int a_cols, const int8_t *b, long long ldb,
                                 void *b_dst, long long b_dld, int b_rows, int b_cols,
                                 uint32_t *zero, int zero_words, int sm_count,
                                 cudaStream_t stream);
}  // namespace pg

namespace pg {
// gemm_i8_imma.cu: dst = src or src^T for an int8 matrix (rows x cols, pitch
// sld) into pitch dld; the operand pre-pass of the mma.sync int8 engine.
cudaError_t launch_i8_relayout(const int8_t *src, long long sld, void *dst, long long dld,
                               int rows, int cols, bool transpose, int sm_count,
                               cudaStream_t stream);
}  // namespace pg

namespace pg {
// api.cu: the int8 GEMM using a fixed device buffer for its widened operands
// instead of allocating; PGEMM_ERR_TOO_LARGE if they do not fit.  `scratch`
// gives the buffer's address and size on the current device; it is called
// after the arguments are checked and the device is set up, and only when
// the call needs scratch.
using FixedScratchFn = pgemm_status (*)(void **ptr, long long *bytes);
pgemm_status gemm_i8_fixed_scratch(int M, int N, int K, int32_t alpha, const int8_t *A,
                                   const int8_t *B, int32_t beta, int32_t *C,
                                   FixedScratchFn scratch, cudaStream_t stream);
}  // namespace pg

namespace pg {
// stage_reuse.cu: the two-stage copy-and-reduce hazard experiment.
cudaError_t launch_stage_reuse(const float *X, int rows, int cols, const int *perm, float *out,
                               int check_reuse, int delay_warp, unsigned delay_ns,
                               unsigned long long *trace_buf, int trace_cap, int blocks,
                               KernelCtx ctx, cudaStream_t stream);
}  // namespace pg
