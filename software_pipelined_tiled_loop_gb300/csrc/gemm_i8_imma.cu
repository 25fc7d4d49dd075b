// Exact int8 GEMM on warp-level integer MMA: the alternative to the
// exact-fp16 tcgen05 route (pgemm_config.engine = PGEMM_ENGINE_MMA_SYNC).
//
// "GPU-Kernel pipelinen" (step 2, the tensor-core IGEMM of its measurements)
// pipelines an int8 GEMM whose consumers are warp-level tensor-core MMAs fed
// from shared memory.  On sm_103a the tcgen05 MMA has no integer kind, so the
// default int8 path multiplies exact fp16 copies; this path keeps the int8
// operands and uses mma.sync.m16n8k32 (s8 x s8 -> s32), exact by
// construction: every product and every partial sum is an integer in the
// s32 accumulator (modulo 2^32, which is also how the result wraps).
//
// Same S-stage TMA ring and mbarriers as the other kernels: warp 0 (one
// lane) loads K-tile t into slot t % S after waiting on empty[t % S]; four
// consumer warps (2 x 2 warp tiles of 64 x 64) wait on full[t % S], read
// fragments with ldmatrix and issue the MMAs, then arrive on empty[t % S].
//
// Operands as the tensor core wants them: A row-major (M x K, K contiguous)
// and B column-major, i.e. B^T (N x K, K contiguous), which a pre-pass writes
// (transpose_i8_kernel; it also repacks A when its pitch is not a multiple of
// 16 bytes).  Slots: A 128 rows (m) x 128 bytes (k), B^T 128 rows (n) x 128
// bytes, both 128-byte swizzled by TMA: byte k of row r at
// r * 128 + (((k / 16) ^ (r % 8)) * 16) + k % 16.  An ldmatrix 8 x 16-byte
// matrix of rows r0..r0+7 at one 16-byte chunk hits eight distinct chunks.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pg {

namespace {

template <int STAGES_>
struct ImmaCfg {
    static constexpr int BM = 128, BN = 128, BK = 128, STAGES = STAGES_;  // BK in int8 values
    static constexpr int A_BYTES = BM * BK, B_BYTES = BN * BK;           // 16 KB each
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CONSUMERS = 4;
    static constexpr int THREADS = 32 * (CONSUMERS + 1);
    static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int SMEM_BYTES = BAR_OFFSET + 2 * STAGES * 8 + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
};

__device__ __forceinline__ void ldmatrix_x4(uint32_t saddr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(saddr));
}

// d += a * b for one 16 x 8 x 32 block (s8 inputs, s32 accumulate).
__device__ __forceinline__ void imma_16832(int32_t (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                           uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t swz(uint32_t slot, int row, int chunk) {
    return slot + static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace

template <int STAGES>
__global__ void __launch_bounds__(ImmaCfg<STAGES>::THREADS, 1)
    imma_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                     const __grid_constant__ CUtensorMap tmap_bt,
                     const GemmArgs<int32_t, int32_t> args, const KernelCtx ctx) {
    using Cfg = ImmaCfg<STAGES>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * Cfg::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFFSET);
    uint64_t *empty = full + STAGES;

    const uint32_t warp = warp_id_uniform();
    const uint32_t lane = lane_id();
    if (threadIdx.x == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_bt);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CONSUMERS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    // the operands may still be being written by this call's pre-pass
    grid_dependency_wait();

    int m0, n0;
    tile_origin(blockIdx.x, args.num_m_tiles, args.num_n_tiles, args.group_m, BM, BN, m0, n0);
    const int T = args.num_k_tiles;

    if (warp == 0) {
        // ---------------- producer ----------------
        if (lane == 0) {
            for (int kt = 0; kt < T; ++kt) {
                const uint32_t s = kt % STAGES, ph = (kt / STAGES) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteProducerEmpty)) break;
                mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
                tma_load_2d(sA + s * Cfg::A_BYTES, &tmap_a, &full[s], kt * BK, m0);
                tma_load_2d(sB + s * Cfg::B_BYTES, &tmap_bt, &full[s], kt * BK, n0);
            }
        }
        return;
    }

    // ---------------- consumers: warp tile 64 x 64 ----------------
    const int c = static_cast<int>(warp) - 1;
    const int wm = c >> 1, wn = c & 1;
    const int mat = static_cast<int>(lane) >> 3, r8 = static_cast<int>(lane) & 7;
    // ldmatrix row addresses: A matrices (rows 0-7 | 8-15) x (k 0-15 | 16-31),
    // B^T matrices (n 0-7, k 0-15), (n 0-7, k 16-31), (n 8-15, k 0-15), (n 8-15, k 16-31)
    const int a_row = wm * 64 + r8 + (mat & 1) * 8, a_chunk = mat >> 1;
    const int b_row = wn * 64 + r8 + (mat >> 1) * 8, b_chunk = mat & 1;

    int32_t acc[4][8][4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 8; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[i][j][e] = 0;

    bool ok = true;
    for (int kt = 0; kt < T; ++kt) {
        const uint32_t s = kt % STAGES, ph = (kt / STAGES) & 1u;
        if (!mbar_wait(&full[s], ph, ctx, kSiteConsumerFull)) {
            ok = false;
            break;
        }
        const uint32_t a_slot = smem_u32(sA + s * Cfg::A_BYTES);
        const uint32_t b_slot = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 32; ++kk) {
            uint32_t a[4][4], b[4][4];
#pragma unroll
            for (int i = 0; i < 4; ++i) ldmatrix_x4(swz(a_slot, a_row + 16 * i, 2 * kk + a_chunk), a[i]);
#pragma unroll
            for (int j = 0; j < 4; ++j) ldmatrix_x4(swz(b_slot, b_row + 16 * j, 2 * kk + b_chunk), b[j]);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    imma_16832(acc[i][2 * j], a[i], b[j][0], b[j][1]);
                    imma_16832(acc[i][2 * j + 1], a[i], b[j][2], b[j][3]);
                }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) return;

    // ---------------- epilogue: alpha * acc + beta * C modulo 2^32 ----------------
    const int g = static_cast<int>(lane) >> 2, tig = static_cast<int>(lane) & 3;
    const bool read_c = args.beta != 0;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int row = m0 + wm * 64 + 16 * i + g + 8 * h;
            if (row >= args.M) continue;
            int32_t *crow = args.C + static_cast<long long>(row) * args.ldc;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int col = n0 + wn * 64 + 8 * j + 2 * tig;
                const int32_t v0 = acc[i][j][2 * h], v1 = acc[i][j][2 * h + 1];
                int32_t *cp = crow + col;
                if (col + 2 <= args.N && (reinterpret_cast<uintptr_t>(cp) & 7u) == 0) {
                    int2 o;
                    if (read_c) {
                        const int2 cv = *reinterpret_cast<const int2 *>(cp);
                        o = make_int2(axpby(args.alpha, v0, args.beta, cv.x),
                                      axpby(args.alpha, v1, args.beta, cv.y));
                    } else {
                        o = make_int2(axpby(args.alpha, v0, 0, 0), axpby(args.alpha, v1, 0, 0));
                    }
                    *reinterpret_cast<int2 *>(cp) = o;
                } else {
                    if (col < args.N)
                        cp[0] = read_c ? axpby(args.alpha, v0, args.beta, cp[0]) : axpby(args.alpha, v0, 0, 0);
                    if (col + 1 < args.N)
                        cp[1] = read_c ? axpby(args.alpha, v1, args.beta, cp[1]) : axpby(args.alpha, v1, 0, 0);
                }
            }
        }
}

// dst = src (transpose == 0) or src^T (transpose != 0) for an int8 matrix of
// rows x cols with pitch sld, into pitch dld.  A block moves a 64 x 64 tile
// through shared memory; reads and writes are byte-wide, consecutive threads
// taking consecutive bytes of a row.
__global__ void __launch_bounds__(256) transpose_i8_kernel(const int8_t *__restrict__ src,
                                                           long long sld, int8_t *__restrict__ dst,
                                                           long long dld, int rows, int cols,
                                                           int transpose) {
    __shared__ int8_t tile[64][65];
    const int tiles_c = (cols + 63) / 64;
    const long long ntiles = static_cast<long long>((rows + 63) / 64) * tiles_c;
    for (long long t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const int r0 = static_cast<int>(t / tiles_c) * 64, c0 = static_cast<int>(t % tiles_c) * 64;
        for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
            const int r = i >> 6, cc = i & 63;
            if (r0 + r < rows && c0 + cc < cols)
                tile[r][cc] = src[static_cast<long long>(r0 + r) * sld + c0 + cc];
        }
        __syncthreads();
        for (int i = threadIdx.x; i < 64 * 64; i += blockDim.x) {
            const int r = i >> 6, cc = i & 63;
            if (transpose) {
                // dst row c0 + r (a column of src), byte r0 + cc
                if (c0 + r < cols && r0 + cc < rows)
                    dst[static_cast<long long>(c0 + r) * dld + r0 + cc] = tile[cc][r];
            } else if (r0 + r < rows && c0 + cc < cols) {
                dst[static_cast<long long>(r0 + r) * dld + c0 + cc] = tile[r][cc];
            }
        }
        __syncthreads();
    }
    grid_launch_dependents();  // this block's share is written
}

cudaError_t launch_i8_relayout(const int8_t *src, long long sld, void *dst, long long dld,
                               int rows, int cols, bool transpose, int sm_count,
                               cudaStream_t stream) {
    if (rows <= 0 || cols <= 0) return cudaSuccess;
    const long long tiles = static_cast<long long>((rows + 63) / 64) * ((cols + 63) / 64);
    const long long cap = static_cast<long long>(sm_count) * 8;
    const int blocks = static_cast<int>(tiles < cap ? tiles : cap);
    transpose_i8_kernel<<<blocks, 256, 0, stream>>>(src, sld, static_cast<int8_t *>(dst), dld,
                                                    rows, cols, transpose ? 1 : 0);
    return cudaGetLastError();
}

// ----------------------------------------------------------------- host ---
template <int STAGES>
static cudaError_t launch_imma(const LaunchI8 &p, cudaStream_t stream) {
    using Cfg = ImmaCfg<STAGES>;
    GemmArgs<int32_t, int32_t> a{};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.num_m_tiles = (p.M + Cfg::BM - 1) / Cfg::BM;
    a.num_n_tiles = (p.N + Cfg::BN - 1) / Cfg::BN;
    a.num_k_tiles = (p.K + Cfg::BK - 1) / Cfg::BK;
    a.group_m = p.group_m > 0 ? p.group_m : 8;
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.C = p.C;
    a.ldc = p.ldc;
    const int tiles = a.num_m_tiles * a.num_n_tiles;
    if (tiles < 1) return cudaSuccess;
    cudaLaunchAttribute attr[1];
    int nattr = 0;
    if (p.after_prepass) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        nattr = 1;
    }
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(tiles);
    lc.blockDim = dim3(Cfg::THREADS);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = attr;
    lc.numAttrs = nattr;
    return cudaLaunchKernelEx(&lc, imma_gemm_kernel<STAGES>, *p.tmap_a, *p.tmap_b, a, p.ctx);
}

template <int STAGES>
static KernelInfo info_imma() {
    using Cfg = ImmaCfg<STAGES>;
    KernelInfo k;
    k.bm = Cfg::BM;
    k.bn = Cfg::BN;
    k.bk = Cfg::BK;
    k.stages = STAGES;
    k.threads = Cfg::THREADS;
    k.smem_bytes = Cfg::SMEM_BYTES;
    k.a_box_x = Cfg::BK;  // 128 int8 = 128 bytes, swizzled
    k.a_box_y = Cfg::BM;
    k.b_box_x = Cfg::BK;  // B^T rows: 128 int8 of K
    k.b_box_y = Cfg::BN;
    k.a_swizzle128 = k.b_swizzle128 = true;
    k.engine = PGEMM_ENGINE_MMA_SYNC;
    k.func = reinterpret_cast<const void *>(imma_gemm_kernel<STAGES>);
    k.launch_i8 = launch_imma<STAGES>;
    return k;
}

const KernelInfo *i8_imma_kernels(int *count) {
    static const KernelInfo table[] = {info_imma<2>(), info_imma<3>(), info_imma<4>(),
                                       info_imma<6>()};
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace pg
