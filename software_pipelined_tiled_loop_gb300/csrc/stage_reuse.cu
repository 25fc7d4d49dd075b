// The stage-reuse hazard experiment of "Software pipelines and asynchronous
// copies" (section "Practice"): a two-stage copy-and-compute kernel over a
// 4096 x 4096 array whose stages are loaded by one producer thread and
// consumed by a deterministic reduction, run with and without the
// consume-before-reuse wait while one consumer warp is artificially delayed.
//
// Per block: one producer thread (warp 4) and four consumer warps.  Block b
// handles the rows perm[b], perm[b + gridDim.x], ... in that order ("tiles"
// t = 0, 1, 2, ...); tile t lives in stage t % 2.  out[r] = sum_c X[perm[r]][c]
// (the caller zeroes out; every warp adds its quarter-row sum).
//
// Readiness and reuse are tracked with per-stage monotone sequence numbers
// in shared memory (not mbarrier phases, which alias once a producer laps a
// consumer):
//   full_seq[s]    = t + 1 once tile t has landed in stage s  (readiness edge)
//   done_seq[s][w] = t + 1 once warp w has finished reading tile t   (reuse)
// The producer waits for its own bulk copy to complete (a private mbarrier)
// before publishing full_seq.  With check_reuse != 0 it also waits, before
// overwriting stage s with tile t, until every warp's done_seq[s] >= t - 1,
// i.e. tile t - 2 has been consumed.  With check_reuse == 0 that one wait is
// skipped and nothing else changes: a slow warp can then read a stage that has
// already been overwritten by a later tile, and its row sum goes wrong.
//
// Every access stays in bounds in both variants (two fixed stage buffers, rows
// named by perm), and every wait is bounded: consumers wait for full_seq to
// reach their tile (the producer never waits on consumers in the hazard
// variant, so it always gets there), the producer waits on its own copies.
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pg {

namespace {

constexpr int kConsumerWarps = 4;

enum TraceEvent : uint32_t {
    kEvLoadIssue = 1,   // producer issued the copy of tile t into stage s
    kEvLoadDone = 2,    // the copy landed; full_seq published
    kEvReuseWait = 3,   // producer starts waiting for tile t-2 to be consumed
    kEvReuseOk = 4,     // ... and may now overwrite the stage
    kEvReadBegin = 5,   // consumer warp w starts reading tile t
    kEvReadEnd = 6,     // consumer warp w finished reading tile t
};

__device__ __forceinline__ void trace(unsigned long long *buf, int cap, uint32_t ev, int t, int s,
                                      int w) {
    if (buf == nullptr || blockIdx.x != 0) return;
    const unsigned long long i = atomicAdd(buf, 1ull);  // buf[0] = event count
    if (static_cast<long long>(i) >= cap) return;
    buf[1 + 2 * i] = globaltimer_ns();
    buf[2 + 2 * i] = (static_cast<unsigned long long>(ev) << 56) |
                     (static_cast<unsigned long long>(s & 0xff) << 48) |
                     (static_cast<unsigned long long>(w & 0xff) << 40) |
                     static_cast<unsigned long long>(t & 0xffffffff);
}

// Bounded spin until *p >= target (volatile shared-memory read).
__device__ __forceinline__ bool wait_seq(const volatile int *p, int target, const KernelCtx &ctx,
                                         uint32_t site) {
    if (*p >= target) return true;
    const uint64_t t0 = globaltimer_ns();
    while (*p < target) {
        if (globaltimer_ns() - t0 > ctx.wait_limit_ns) {
            atomicCAS(ctx.status, 0u, kStatusTimeout | site);
            return false;
        }
    }
    return true;
}

}  // namespace

__global__ void __launch_bounds__(160, 1)
    stage_reuse_kernel(const float *__restrict__ X, int rows, int cols, const int *__restrict__ perm,
                       float *__restrict__ out, int check_reuse, int delay_warp,
                       unsigned delay_ns, unsigned long long *trace_buf, int trace_cap,
                       KernelCtx ctx) {
    extern __shared__ __align__(128) uint8_t smem_raw[];
    float *stage = reinterpret_cast<float *>(smem_raw);  // [2][cols]
    __shared__ int full_seq[2];
    __shared__ int done_seq[2][kConsumerWarps];
    __shared__ __align__(8) uint64_t copy_bar[2];

    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    if (threadIdx.x == 0) {
        for (int s = 0; s < 2; ++s) {
            full_seq[s] = 0;
            for (int w = 0; w < kConsumerWarps; ++w) done_seq[s][w] = 0;
            mbar_init(&copy_bar[s], 1);
        }
        fence_barrier_init();
    }
    __syncthreads();

    const int ntiles = rows > static_cast<int>(blockIdx.x)
                           ? (rows - static_cast<int>(blockIdx.x) + gridDim.x - 1) / gridDim.x
                           : 0;
    const uint32_t row_bytes = static_cast<uint32_t>(cols) * 4u;

    if (warp == kConsumerWarps) {
        if (lane == 0) {
            // ---------------- producer ----------------
            for (int t = 0; t < ntiles; ++t) {
                const int s = t & 1;
                if (t >= 2 && check_reuse) {
                    // the consume-before-reuse edge: tile t-2 must be fully read
                    trace(trace_buf, trace_cap, kEvReuseWait, t, s, 0);
                    bool ok = true;
                    for (int w = 0; ok && w < kConsumerWarps; ++w)
                        ok = wait_seq(&done_seq[s][w], t - 1, ctx, kSiteProducerEmpty);
                    if (!ok) break;
                    trace(trace_buf, trace_cap, kEvReuseOk, t, s, 0);
                }
                const int r = perm[blockIdx.x + static_cast<long long>(t) * gridDim.x];
                // the previous generic reads of this stage come before the async-proxy write
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(&copy_bar[s], row_bytes);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                    " [%0], [%1], %2, [%3];" ::"r"(smem_u32(stage + s * cols)),
                    "l"(X + static_cast<long long>(r) * cols), "r"(row_bytes),
                    "r"(smem_u32(&copy_bar[s]))
                    : "memory");
                trace(trace_buf, trace_cap, kEvLoadIssue, t, s, 0);
                if (!mbar_wait(&copy_bar[s], static_cast<uint32_t>(t >> 1) & 1u, ctx,
                               kSiteMmaFull))
                    break;
                trace(trace_buf, trace_cap, kEvLoadDone, t, s, 0);
                __threadfence_block();
                *reinterpret_cast<volatile int *>(&full_seq[s]) = t + 1;  // readiness edge
            }
        }
        return;
    }

    // ---------------- consumers: each warp sums a quarter of the row ----------------
    const int quarter = cols / kConsumerWarps;
    for (int t = 0; t < ntiles; ++t) {
        const int s = t & 1;
        if (!wait_seq(&full_seq[s], t + 1, ctx, kSiteConsumerFull)) break;
        __threadfence_block();
        if (warp == delay_warp && delay_ns > 0) __nanosleep(delay_ns);  // the artificial delay
        if (lane == 0) trace(trace_buf, trace_cap, kEvReadBegin, t, s, warp);
        const volatile float *src = stage + s * cols + warp * quarter;
        float acc = 0.f;
        for (int c = lane; c < quarter; c += 32) acc += src[c];
        __syncwarp();
        if (lane == 0) trace(trace_buf, trace_cap, kEvReadEnd, t, s, warp);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
        if (lane == 0) {
            atomicAdd(&out[blockIdx.x + static_cast<long long>(t) * gridDim.x], acc);
            __threadfence_block();
            *reinterpret_cast<volatile int *>(&done_seq[s][warp]) = t + 1;  // reuse edge
        }
        __syncwarp();
    }
}

cudaError_t launch_stage_reuse(const float *X, int rows, int cols, const int *perm, float *out,
                               int check_reuse, int delay_warp, unsigned delay_ns,
                               unsigned long long *trace_buf, int trace_cap, int blocks,
                               KernelCtx ctx, cudaStream_t stream) {
    const int smem = 2 * cols * 4;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(stage_reuse_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, 65536);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    stage_reuse_kernel<<<blocks, 160, smem, stream>>>(X, rows, cols, perm, out, check_reuse,
                                                      delay_warp, delay_ns, trace_buf, trace_cap,
                                                      ctx);
    return cudaGetLastError();
}

}  // namespace pg
