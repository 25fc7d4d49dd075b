// fp32 GEMM with FFMA register tiles, fed by an S-stage TMA ring.
//
// This is the computation of the double-buffered SGEMM in "Double Buffering:
// Software Pipelining the K-Loop" (section "The Kernel": a block tile, warp
// tiles, per-thread register tiles of outer products, an alpha/beta epilogue)
// with its two-buffer cp.async / register-transpose K-loop replaced by the
// GB300 mechanism: K-tiles are streamed into S shared-memory slots with TMA
// bulk-tensor copies that complete on the slot's "full" mbarrier, and the
// consumer warps hand a slot back by arriving on its "empty" mbarrier
// ("Software pipelines and asynchronous copies", section "Producer-consumer
// synchronization").  No block-wide barrier remains in the steady state.
//
// The producer is lane 0 of warp 0, not a warp of its own: a fifth warp would
// put 10 warps on an SM running two blocks, and the register file would then
// allow only 168 registers a thread, too few for the 8 x 16 register tile.
// Lane 0 issues the prologue (tiles 0 .. min(S, T) - 1, never beyond K) and
// then, at the top of each K iteration, refills every slot whose "empty"
// phase has completed (a non-blocking test), keeping up to S tiles in flight;
// it blocks on "empty" only when the tile it is about to consume has not been
// issued yet.
//
// Tile: BM x BN = 128 x 128, BK = 32 floats.  Four consumer warps in a 2 x 2
// grid of 64 x 64 warp tiles; a warp's 32 lanes form 8 (m) x 4 (n) threads
// with an 8 x 16 register tile each.  Thread rows are m = 8*i + tr (i = 0..7)
// so the 8 rows a quarter-warp reads have distinct (m mod 8) and hit distinct
// 16-byte chunks of the 128-byte swizzle; thread columns are four float4
// groups n = 16*g + 4*tc.
//
// Shared-memory layouts (TMA-written):
//   A slot: 128 rows (m) x 32 floats (k), 128-byte swizzled: element (m, k)
//           at m*128 + (((k/4) ^ (m%8)) * 16) + (k%4)*4 bytes.  A thread reads
//           float4 along k for each of its rows (no transpose is needed, unlike
//           the page's k-major copy of A, which TMA cannot produce).
//   B slot: 32 rows (k) x 128 floats (n), unswizzled rows of 512 bytes; a
//           quarter-warp reads 4 consecutive float4 of one row.
//
// The products run as fma.rn.f32x2 (two fp32 FMAs per instruction, each
// rounded exactly like a scalar FFMA), which halves the issue slots the
// arithmetic takes so loads and address arithmetic fit beside it.
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace pg {

template <int BN_, int STAGES>
struct F32Cfg {
    static constexpr int BM = 128, BN = BN_, BK = 32;
    static constexpr int G = BN / 32;             // float4 column groups per thread
    static constexpr int MIN_BLOCKS = BN == 64 ? 3 : 2;  // register budget per thread
    static constexpr int A_BYTES = BM * BK * 4;  // 16 KB
    static constexpr int B_BYTES = BK * BN * 4;  // 16 KB
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int CONSUMER_WARPS = 4;
    static constexpr int THREADS = CONSUMER_WARPS * 32;
    static constexpr int BAR_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int USED = BAR_OFFSET + 2 * STAGES * 8;
    static constexpr int SMEM_BYTES = USED + 1024;
    static_assert(SMEM_BYTES <= 232448, "shared memory");
    static_assert(BN == 64 || BN == 128, "BN");
};

__device__ __forceinline__ float4 lds128(uint32_t saddr) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(saddr));
    return v;
}

// acc[i][2*g + h] holds columns 16*g + 4*tc + 2*h + {0,1} of row 8*i + tr of
// the thread's warp tile (64 rows x BN/2 columns; warp (wm, wn) of a 2 x 2 grid).
template <int BN>
using AccTile = float2[8][BN / 16];

// acc += the products of k-groups [K4B, K4E) (four k each) of the K-tile held
// in a shared-memory slot: a_base / b_base are the slot addresses plus this
// thread's row / column offsets (layouts above).
template <int BN, int K4B, int K4E>
__device__ __forceinline__ void mma_ktile(AccTile<BN> &acc, uint32_t a_base, uint32_t b_base, int tr) {
    constexpr int G = BN / 32;
#pragma unroll 2
    for (int k4 = K4B; k4 < K4E; ++k4) {
        float4 a[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)  // (m % 8) == tr for every row of this thread
            a[i] = lds128(a_base + i * 1024 + ((k4 ^ tr) << 4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float4 b[G];
            const uint32_t brow = b_base + (k4 * 4 + kk) * (BN * 4);
#pragma unroll
            for (int g = 0; g < G; ++g) b[g] = lds128(brow + g * 64);
            // the eight rows' A values, each broadcast to a pair
            float2 a2[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float av = kk == 0 ? a[i].x : kk == 1 ? a[i].y : kk == 2 ? a[i].z : a[i].w;
                a2[i] = make_float2(av, av);
            }
            // B-pair-major order: consecutive FFMA2s share an operand pair
            // (measured 62.4 vs 60.0 TFLOP/s for the row-major order)
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float2 b0 = make_float2(b[g].x, b[g].y), b1 = make_float2(b[g].z, b[g].w);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    acc[i][2 * g] = __ffma2_rn(a2[i], b0, acc[i][2 * g]);
                    acc[i][2 * g + 1] = __ffma2_rn(a2[i], b1, acc[i][2 * g + 1]);
                }
            }
        }
    }
}

// C[row][col .. col+3] as a float4 (zeros outside C): one 16-byte load where
// the four columns are in range and aligned, else element by element.
__device__ __forceinline__ float4 load_c4(const GemmArgs<float, float> &args, int row, int col) {
    float4 c = make_float4(0.f, 0.f, 0.f, 0.f);
    if (row >= args.M || col >= args.N) return c;
    const float *cp = args.C + static_cast<long long>(row) * args.ldc + col;
    if (col + 4 <= args.N && (reinterpret_cast<uintptr_t>(cp) & 15u) == 0)
        return *reinterpret_cast<const float4 *>(cp);
    c.x = cp[0];
    if (col + 1 < args.N) c.y = cp[1];
    if (col + 2 < args.N) c.z = cp[2];
    if (col + 3 < args.N) c.w = cp[3];
    return c;
}

// C[row][col .. col+3] <- alpha * v + beta * c (c: the old C values, read
// only when beta != 0), a 16-byte store where in range and aligned.
__device__ __forceinline__ void put_c4(const GemmArgs<float, float> &args, int row, int col,
                                       const float4 &v, const float4 &c) {
    if (row >= args.M || col >= args.N) return;
    float *cp = args.C + static_cast<long long>(row) * args.ldc + col;
    float4 o;
    if (args.beta != 0.f)
        o = make_float4(axpby(args.alpha, v.x, args.beta, c.x), axpby(args.alpha, v.y, args.beta, c.y),
                        axpby(args.alpha, v.z, args.beta, c.z), axpby(args.alpha, v.w, args.beta, c.w));
    else
        o = make_float4(args.alpha * v.x, args.alpha * v.y, args.alpha * v.z, args.alpha * v.w);
    if (col + 4 <= args.N && (reinterpret_cast<uintptr_t>(cp) & 15u) == 0) {
        *reinterpret_cast<float4 *>(cp) = o;
    } else {
        cp[0] = o.x;
        if (col + 1 < args.N) cp[1] = o.y;
        if (col + 2 < args.N) cp[2] = o.z;
        if (col + 3 < args.N) cp[3] = o.w;
    }
}

// The thread's float4 f = i * (BN/32) + k of a tile holds row 8*i + tr,
// columns 16*k + 4*tc .. +3 of its warp tile.
template <int BN>
__device__ __forceinline__ void c4_coords(int f, int m0, int n0, int wm, int wn, int tr, int tc,
                                          int &row, int &col) {
    row = m0 + wm * 64 + 8 * (f / (BN / 32)) + tr;
    col = n0 + wn * (BN / 2) + 16 * (f % (BN / 32)) + 4 * tc;
}

// C <- alpha * acc + beta * C for this thread's part of the tile at (m0, n0).
// With beta != 0 the old C values are read eight float4 at a time, all eight
// loads in flight before the first store, instead of one round trip each.
template <int BN>
__device__ __forceinline__ void store_tile(const GemmArgs<float, float> &args, const AccTile<BN> &acc,
                                           int m0, int n0, int wm, int wn, int tr, int tc) {
    constexpr int NF = 8 * (BN / 32);
    const bool read_c = args.beta != 0.f;
#pragma unroll
    for (int f0 = 0; f0 < NF; f0 += 8) {
        float4 c[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            int row, col;
            c4_coords<BN>(f0 + e, m0, n0, wm, wn, tr, tc, row, col);
            c[e] = read_c ? load_c4(args, row, col) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const int f = f0 + e, i = f / (BN / 32), k = f % (BN / 32);
            int row, col;
            c4_coords<BN>(f, m0, n0, wm, wn, tr, tc, row, col);
            put_c4(args, row, col,
                   make_float4(acc[i][2 * k].x, acc[i][2 * k].y, acc[i][2 * k + 1].x,
                               acc[i][2 * k + 1].y),
                   c[e]);
        }
    }
}

template <int BN_, int STAGES>
__global__ void __launch_bounds__(128, F32Cfg<BN_, STAGES>::MIN_BLOCKS)
    gemm_f32_kernel(const __grid_constant__ CUtensorMap tmap_a,
                    const __grid_constant__ CUtensorMap tmap_b,
                    const GemmArgs<float, float> args, const KernelCtx ctx) {
    using Cfg = F32Cfg<BN_, STAGES>;
    constexpr int G = Cfg::G;
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
        prefetch_tmap(&tmap_b);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        fence_barrier_init();
    }
    __syncthreads();

    // A stream-K tail grid behind this one may start once every block of this
    // grid has started: its blocks then take over the slots these free.
    grid_launch_dependents();
    // whole tiles follow the stream-K tiles [0, args.split_tiles)
    int m0, n0;
    tile_origin(static_cast<int>(blockIdx.x) + args.split_tiles, args.num_m_tiles,
                args.num_n_tiles, args.group_m, BM, BN, m0, n0);
    const int T = args.num_k_tiles;
    const bool producer = threadIdx.x == 0;

    // Issue the TMA copies of K-tile t into slot t % S.
    auto issue = [&](int t) {
        const int s = t % STAGES;
        mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
        tma_load_2d(sA + s * Cfg::A_BYTES, &tmap_a, &full[s], t * BK, m0);
        tma_load_2d(sB + s * Cfg::B_BYTES, &tmap_b, &full[s], n0, t * BK);
    };
    int next_load = 0;  // tiles [0, next_load) have been issued (producer lane only)
    if (producer) {
        // prologue: fill min(S, T) slots
        for (; next_load < T && next_load < STAGES; ++next_load) issue(next_load);
    }

    // ---------------- consumers ----------------
    const int wm = static_cast<int>(warp) >> 1;  // warp tile row (0..1)
    const int wn = static_cast<int>(warp) & 1;   // warp tile column (0..1)
    const int tr = static_cast<int>(lane) >> 2;  // 0..7
    const int tc = static_cast<int>(lane) & 3;   // 0..3

    constexpr int WN = BN / 2;
    AccTile<BN> acc;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 2 * G; ++j) acc[i][j] = make_float2(0.f, 0.f);

    // byte offsets inside a slot
    const uint32_t a_row0 = static_cast<uint32_t>((wm * 64 + tr) * 128);  // row 8*i+tr: + i*1024
    const uint32_t b_col0 = static_cast<uint32_t>((wn * WN + tc * 4) * 4);

    bool ok = true;
    for (int kt = 0; kt < T; ++kt) {
        if (producer) {
            // steady state: refill released slots, up to S tiles ahead of kt
            while (next_load < T && next_load < kt + STAGES) {
                const int prev = next_load - STAGES;  // last tile that used this slot
                uint64_t *e = &empty[next_load % STAGES];
                const uint32_t par = static_cast<uint32_t>(prev / STAGES) & 1u;
                if (!mbar_test_wait(e, par)) {
                    if (next_load > kt) break;  // not needed yet: try again next iteration
                    if (!mbar_wait(e, par, ctx, kSiteProducerEmpty)) break;
                }
                issue(next_load++);
            }
        }
        const uint32_t s = kt % STAGES, ph = (kt / STAGES) & 1u;
        if (!mbar_wait(&full[s], ph, ctx, kSiteConsumerFull)) {
            ok = false;
            break;
        }
        const uint32_t a_base = smem_u32(sA + s * Cfg::A_BYTES) + a_row0;
        const uint32_t b_base = smem_u32(sB + s * Cfg::B_BYTES) + b_col0;
        mma_ktile<BN, 0, BK / 4>(acc, a_base, b_base, tr);
        // Release the slot: this warp's reads of it are done.  The reads have
        // returned their values (the products above consumed them) and the
        // arrive orders them before the producer's acquiring wait, after
        // which its TMA overwrites the slot: a read-then-overwrite order
        // needs no proxy fence (measured: +0.4 % without one).
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
    }
    if (!ok) return;

    // ---------------- epilogue: alpha * acc + beta * C ----------------
    store_tile<BN>(args, acc, m0, n0, wm, wn, tr, tc);
}

// The stream-K tail (args.split_tiles = R > 0 output tiles, the tiles the
// full waves would leave over): the whole tiles [R, tiles), exactly full
// waves, run first in gemm_f32_kernel; this grid of G blocks, one per
// resident slot, is launched behind it with programmatic serialisation, so
// its blocks take over each SM slot a whole-tile block frees.  It deals the
// R * T K-iterations of tiles [0, R) out in equal contiguous ranges, block j
// taking [j * R * T / G, (j + 1) * R * T / G) (pieces of at most two tiles,
// since R < G): the leftover tiles cost R / G of a tile per slot instead of a
// whole extra wave.  (Run first instead, the two blocks sharing an SM end
// their equal shares at different times, and the whole tiles behind them
// end staggered by as much.)  A piece ends in an exchange: every
// piece stores its raw partial sums to its own slot in `partials`, counts
// itself on the tile's ticket in `counters` (after a fence), and the piece
// that takes the last ticket adds all pieces in slot order (so the result
// does not depend on timing) and writes C.  Nothing waits on another block.
struct F32Stream {
    int T, G, j, R;
    long long sk_a, sk_total;
    int sk_len, n_sk;

    __device__ __forceinline__ void init(const GemmArgs<float, float> &a) {
        T = a.num_k_tiles;
        G = static_cast<int>(gridDim.x);
        j = static_cast<int>(blockIdx.x);
        R = a.split_tiles;
        sk_total = static_cast<long long>(R) * T;
        sk_a = R > 0 ? j * sk_total / G : 0;
        sk_len = R > 0 ? static_cast<int>((j + 1) * sk_total / G - sk_a) : 0;
        n_sk = sk_len == 0 ? 0 : ((sk_a / T) == ((sk_a + sk_len - 1) / T) ? 1 : 2);
    }
    __device__ __forceinline__ int units() const { return n_sk; }
    __device__ __forceinline__ int iterations() const { return sk_len; }
    // piece u (0 or 1): its tile and K-tiles [kb, ke)
    __device__ __forceinline__ void unit(int u, int &tile, int &kb, int &ke) const {
        tile = static_cast<int>(sk_a / T) + u;
        const long long t0 = static_cast<long long>(tile) * T;
        const long long lo = sk_a > t0 ? sk_a : t0;
        const long long end = sk_a + sk_len, hi = end < t0 + T ? end : t0 + T;
        kb = static_cast<int>(lo - t0);
        ke = static_cast<int>(hi - t0);
    }
    // the slot holding stream-K iteration x
    __device__ __forceinline__ int slot_of(long long x) const {
        return static_cast<int>(((x + 1) * G - 1) / sk_total);
    }
};

template <int BN_, int STAGES>
__global__ void __launch_bounds__(128, F32Cfg<BN_, STAGES>::MIN_BLOCKS)
    gemm_f32_streamk_kernel(const __grid_constant__ CUtensorMap tmap_a,
                            const __grid_constant__ CUtensorMap tmap_b,
                            const GemmArgs<float, float> args, const KernelCtx ctx) {
    using Cfg = F32Cfg<BN_, STAGES>;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * Cfg::A_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFFSET);
    uint64_t *empty = full + STAGES;
    __shared__ int last_piece;
    // The schedule and the producer's cursor (the unit and K-tile of its next
    // load) live in shared memory: they are read once per unit or K-tile,
    // and registers are all taken by the 8 x 16 tile.
    __shared__ F32Stream ws;
    __shared__ int pc[6];  // unit, tile, next K-tile, end K-tile, m0, n0

    const uint32_t warp = warp_id_uniform();
    const uint32_t lane = lane_id();
    const int tid = static_cast<int>(threadIdx.x);

    if (threadIdx.x == 0) {
        prefetch_tmap(&tmap_a);
        prefetch_tmap(&tmap_b);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        fence_barrier_init();
        ws.init(args);
    }
    __syncthreads();

    const int total = ws.iterations();
    const int nunits = ws.units();
    const bool producer = threadIdx.x == 0;

    auto p_enter = [&](int u) {
        int tile, kb, ke, m0, n0;
        ws.unit(u, tile, kb, ke);
        tile_origin(tile, args.num_m_tiles, args.num_n_tiles, args.group_m, BM, BN, m0, n0);
        pc[0] = u;
        pc[1] = tile;
        pc[2] = kb;
        pc[3] = ke;
        pc[4] = m0;
        pc[5] = n0;
    };
    // Issue the TMA copies of the next iteration (number g) into slot g % S.
    auto issue = [&](int g) {
        while (pc[2] == pc[3]) p_enter(pc[0] + 1);
        const int s = g % STAGES, kt = pc[2];
        mbar_arrive_expect_tx(&full[s], Cfg::STAGE_BYTES);
        tma_load_2d(sA + s * Cfg::A_BYTES, &tmap_a, &full[s], kt * BK, pc[4]);
        tma_load_2d(sB + s * Cfg::B_BYTES, &tmap_b, &full[s], pc[5], kt * BK);
        pc[2] = kt + 1;
    };
    int next_load = 0;  // iterations [0, next_load) have been issued (producer lane only)
    if (producer && total > 0) {
        p_enter(0);
        // prologue: fill min(S, total) slots
        for (; next_load < total && next_load < STAGES; ++next_load) issue(next_load);
    }

    // ---------------- consumers ----------------
    const int wm = static_cast<int>(warp) >> 1;  // warp tile row (0..1)
    const int wn = static_cast<int>(warp) & 1;   // warp tile column (0..1)
    const int tr = static_cast<int>(lane) >> 2;  // 0..7
    const int tc = static_cast<int>(lane) & 3;   // 0..3

    constexpr int WN = BN / 2;
    // byte offsets inside a slot
    const uint32_t a_row0 = static_cast<uint32_t>((wm * 64 + tr) * 128);  // row 8*i+tr: + i*1024
    const uint32_t b_col0 = static_cast<uint32_t>((wn * WN + tc * 4) * 4);

    // A failed (timed-out) wait is recorded and the block keeps going
    // without waiting, so that every thread still meets every block barrier.
    bool ok = true;
    int g = 0;
    for (int u = 0; u < nunits; ++u) {
        int tile, kb, ke;
        ws.unit(u, tile, kb, ke);
        AccTile<BN> acc;
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int k = 0; k < BN / 16; ++k) acc[i][k] = make_float2(0.f, 0.f);
        for (int kt = kb; kt < ke; ++kt, ++g) {
            if (producer && ok) {
                // steady state: refill released slots, up to S iterations ahead of g
                while (next_load < total && next_load < g + STAGES) {
                    const int prev = next_load - STAGES;  // last iteration that used this slot
                    uint64_t *e = &empty[next_load % STAGES];
                    const uint32_t par = static_cast<uint32_t>(prev / STAGES) & 1u;
                    if (!mbar_test_wait(e, par)) {
                        if (next_load > g) break;  // not needed yet: try again next iteration
                        if (!mbar_wait(e, par, ctx, kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                    }
                    issue(next_load++);
                }
            }
            const uint32_t s = g % STAGES, ph = (g / STAGES) & 1u;
            if (ok && !mbar_wait(&full[s], ph, ctx, kSiteConsumerFull)) ok = false;
            const uint32_t a_base = smem_u32(sA + s * Cfg::A_BYTES) + a_row0;
            const uint32_t b_base = smem_u32(sB + s * Cfg::B_BYTES) + b_col0;
            mma_ktile<BN, 0, BK / 4>(acc, a_base, b_base, tr);
            // Release the slot (no proxy fence: see gemm_f32_kernel).
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }

        int m0, n0;
        tile_origin(tile, args.num_m_tiles, args.num_n_tiles, args.group_m, BM, BN, m0, n0);
        // a piece of `tile`: leave the partial sums, take a ticket
        const int first = ws.slot_of(static_cast<long long>(tile) * ws.T);
        const int last = ws.slot_of(static_cast<long long>(tile + 1) * ws.T - 1);
        float4 *mine = reinterpret_cast<float4 *>(args.partials) +
                       static_cast<long long>(ws.j * 2 + u) * (BM * BN / 4);
#pragma unroll
        for (int i = 0; i < 8; ++i)
#pragma unroll
            for (int k = 0; k < BN / 32; ++k)
                mine[(i * (BN / 32) + k) * 128 + tid] =
                    make_float4(acc[i][2 * k].x, acc[i][2 * k].y, acc[i][2 * k + 1].x,
                                acc[i][2 * k + 1].y);
        __threadfence();
        __syncthreads();
        if (tid == 0)
            last_piece = atomicAdd(&args.counters[tile], 1u) == static_cast<uint32_t>(last - first);
        __syncthreads();
        if (last_piece) {
            __threadfence();
            // Every piece is stored: add them in slot order straight into C
            // (float4 f of each piece holds the same elements of the tile),
            // eight float4 of C and of every piece in flight at once.
            constexpr int NF = 8 * (BN / 32);
            const bool read_c = args.beta != 0.f;
#pragma unroll 1
            for (int f0 = 0; f0 < NF; f0 += 8) {
                float4 c[8], sum[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    int row, col;
                    c4_coords<BN>(f0 + e, m0, n0, wm, wn, tr, tc, row, col);
                    c[e] = read_c ? load_c4(args, row, col) : make_float4(0.f, 0.f, 0.f, 0.f);
                }
                for (int q = first; q <= last; ++q) {
                    const int qunit = tile - static_cast<int>(
                                                 (static_cast<long long>(q) * ws.sk_total / ws.G) / ws.T);
                    const float4 *src = reinterpret_cast<const float4 *>(args.partials) +
                                        static_cast<long long>(q * 2 + qunit) * (BM * BN / 4) +
                                        f0 * 128 + tid;
                    float4 x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = __ldcg(src + e * 128);
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        if (q == first) {
                            sum[e] = x[e];
                        } else {
                            sum[e].x += x[e].x;
                            sum[e].y += x[e].y;
                            sum[e].z += x[e].z;
                            sum[e].w += x[e].w;
                        }
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    int row, col;
                    c4_coords<BN>(f0 + e, m0, n0, wm, wn, tr, tc, row, col);
                    if (ok) put_c4(args, row, col, sum[e], c[e]);
                }
            }
        }
        __syncthreads();  // last_piece is read by every thread before it is rewritten
    }
    // This grid runs beside the tail of the whole-tile grid launched before
    // it; it does not end before that grid has, so that later work on the
    // stream sees all of C.
    grid_dependency_wait();
}

// ------------------------------------------- register-staged comparator ---
// The same block tile, register tile and arithmetic with the producer of the
// pages' own kernels: no TMA and no mbarriers.  Every thread loads its share
// of K-tile t+1 from global memory into registers while the block computes
// tile t from one of two shared-memory buffers, then stores the registers
// into the other buffer (A with the same 128-byte swizzle TMA would apply,
// so the arithmetic reads both kernels' buffers identically); one block
// barrier per K-tile hands the buffers over ("Double Buffering: Software
// Pipelining the K-Loop", sections "The Kernel" and "Mechanics": the global
// loads at the top of the iteration, the shared stores at the bottom, the
// arithmetic in between covering their latency; "GPU-Kernel pipelinen",
// step 3, the LDG-register variant).  With two buffers the buffer written in
// iteration t was last read in iteration t-1, before that iteration's
// barrier, so the barrier the LDG-register listing places before the stores
// is not needed.  To fit beside the 8 x 16 register tile, the next tile is
// staged in PARTS pieces, each loaded before and stored after 1/PARTS of the
// current tile's arithmetic.
//
// Loads: A is 128 rows x 8 float4 (thread f: row f / 8 + 16 j, float4 f % 8),
// B is 32 rows x BN/4 float4; consecutive threads read consecutive 16-byte
// pieces of a row.  Out-of-range rows and columns read as zero (the TMA
// kernel's out-of-bounds fill), element by element at a ragged K or N edge.
template <int BN>
struct RegStage {
    static constexpr int A_F4 = 8;          // float4 of A per thread per K-tile
    static constexpr int B_ROW_F4 = BN / 4;  // float4 per B row
    static constexpr int B_ROWS_PER_PASS = 128 / B_ROW_F4;
    static constexpr int B_F4 = 32 / B_ROWS_PER_PASS;  // float4 of B per thread per K-tile
    static constexpr int PARTS = BN == 128 ? 4 : 2;     // register budget
    static constexpr int A_PART = A_F4 / PARTS, B_PART = B_F4 / PARTS;
    static_assert(A_F4 % PARTS == 0 && B_F4 % PARTS == 0 && 8 % PARTS == 0, "parts");
};

// One K iteration of the register-staged loop from part P on: load part P of
// the next tile, do part P of this tile's arithmetic, store part P.
template <int BN, int P, class Load, class Store, class RA, class RB>
__device__ __forceinline__ void regstage_parts(AccTile<BN> &acc, uint32_t a_base, uint32_t b_base,
                                               int tr, bool more, int t_next, int buf_next,
                                               const Load &load, const Store &store, RA &ra,
                                               RB &rb) {
    constexpr int PARTS = RegStage<BN>::PARTS;
    if constexpr (P < PARTS) {
        if (more) load(t_next, P, ra, rb);
        mma_ktile<BN, P * 8 / PARTS, (P + 1) * 8 / PARTS>(acc, a_base, b_base, tr);
        if (more) store(buf_next, P, ra, rb);
        regstage_parts<BN, P + 1>(acc, a_base, b_base, tr, more, t_next, buf_next, load, store,
                                  ra, rb);
    }
}

__device__ __forceinline__ float4 load_f4(const float *row, int col, int limit, bool row_ok) {
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (!row_ok || col >= limit) return v;
    if (col + 4 <= limit) return __ldg(reinterpret_cast<const float4 *>(row + col));
    v.x = row[col];
    if (col + 1 < limit) v.y = row[col + 1];
    if (col + 2 < limit) v.z = row[col + 2];
    return v;
}

__device__ __forceinline__ void sts_f4(uint32_t saddr, float4 v) {
    sts128(saddr, __float_as_uint(v.x), __float_as_uint(v.y), __float_as_uint(v.z),
           __float_as_uint(v.w));
}

template <int BN>
__global__ void __launch_bounds__(128, F32Cfg<BN, 2>::MIN_BLOCKS)
    gemm_f32_regstage_kernel(const float *__restrict__ A, long long lda,
                             const float *__restrict__ B, long long ldb,
                             const GemmArgs<float, float> args) {
    using Cfg = F32Cfg<BN, 2>;
    using RS = RegStage<BN>;
    constexpr int BM = Cfg::BM, BK = Cfg::BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    const uint32_t sA = smem_u32(smem);                       // [2][A_BYTES]
    const uint32_t sB = smem_u32(smem + 2 * Cfg::A_BYTES);    // [2][B_BYTES]

    const int tid = static_cast<int>(threadIdx.x);
    const uint32_t warp = warp_id_uniform();
    const uint32_t lane = lane_id();
    int m0, n0;
    tile_origin(blockIdx.x, args.num_m_tiles, args.num_n_tiles, args.group_m, BM, BN, m0, n0);
    const int T = args.num_k_tiles;

    // this thread's load coordinates
    const int a_row = tid >> 3, a_c4 = tid & 7;                // + 16 j rows
    const int b_row = tid / RS::B_ROW_F4, b_c4 = tid % RS::B_ROW_F4;  // + B_ROWS_PER_PASS j rows

    // load part h of K-tile t into registers
    auto load_part = [&](int t, int h, float4 (&ra)[RS::A_PART], float4 (&rb)[RS::B_PART]) {
        const int k0 = t * BK;
#pragma unroll
        for (int j = 0; j < RS::A_PART; ++j) {
            const int r = a_row + 16 * (h * RS::A_PART + j);
            const int m = m0 + r;
            ra[j] = load_f4(A + static_cast<long long>(m < args.M ? m : 0) * lda, k0 + 4 * a_c4,
                            args.K, m < args.M);
        }
#pragma unroll
        for (int j = 0; j < RS::B_PART; ++j) {
            const int r = b_row + RS::B_ROWS_PER_PASS * (h * RS::B_PART + j);
            const int k = k0 + r;
            rb[j] = load_f4(B + static_cast<long long>(k < args.K ? k : 0) * ldb, n0 + 4 * b_c4,
                            args.N, k < args.K);
        }
    };
    // store part h from registers into buffer `buf`
    auto store_part = [&](int buf, int h, const float4 (&ra)[RS::A_PART],
                          const float4 (&rb)[RS::B_PART]) {
        const uint32_t a_slot = sA + buf * Cfg::A_BYTES, b_slot = sB + buf * Cfg::B_BYTES;
#pragma unroll
        for (int j = 0; j < RS::A_PART; ++j) {
            const int r = a_row + 16 * (h * RS::A_PART + j);
            sts_f4(a_slot + r * 128 + ((a_c4 ^ (r & 7)) << 4), ra[j]);
        }
#pragma unroll
        for (int j = 0; j < RS::B_PART; ++j) {
            const int r = b_row + RS::B_ROWS_PER_PASS * (h * RS::B_PART + j);
            sts_f4(b_slot + r * (BN * 4) + b_c4 * 16, rb[j]);
        }
    };

    const int wm = static_cast<int>(warp) >> 1, wn = static_cast<int>(warp) & 1;
    const int tr = static_cast<int>(lane) >> 2, tc = static_cast<int>(lane) & 3;
    constexpr int WN = BN / 2;
    AccTile<BN> acc;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < BN / 16; ++j) acc[i][j] = make_float2(0.f, 0.f);
    const uint32_t a_row0 = static_cast<uint32_t>((wm * 64 + tr) * 128);
    const uint32_t b_col0 = static_cast<uint32_t>((wn * WN + tc * 4) * 4);

    float4 ra[RS::A_PART], rb[RS::B_PART];
    // prologue: K-tile 0 into buffer 0
    if (T > 0) {
#pragma unroll
        for (int h = 0; h < RS::PARTS; ++h) {
            load_part(0, h, ra, rb);
            store_part(0, h, ra, rb);
        }
    }
    __syncthreads();
    for (int kt = 0; kt < T; ++kt) {
        const int cur = kt & 1;
        const uint32_t a_base = sA + cur * Cfg::A_BYTES + a_row0;
        const uint32_t b_base = sB + cur * Cfg::B_BYTES + b_col0;
        regstage_parts<BN, 0>(acc, a_base, b_base, tr, kt + 1 < T, kt + 1, cur ^ 1, load_part,
                              store_part, ra, rb);
        __syncthreads();  // tile kt+1 is in place; tile kt's buffer may be refilled
    }
    store_tile<BN>(args, acc, m0, n0, wm, wn, tr, tc);
}

// ----------------------------------------------------------------- host ---
template <int BN, int STAGES>
static cudaError_t launch_f32_impl(const LaunchF32 &p, cudaStream_t stream) {
    using Cfg = F32Cfg<BN, STAGES>;
    GemmArgs<float, float> a{};
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
    a.split_tiles = static_cast<int>(p.sched.split_tiles);
    a.partials = p.sched.partials;
    a.counters = p.sched.counters;
    const long long tiles = static_cast<long long>(a.num_m_tiles) * a.num_n_tiles;
    if (tiles < 1) return cudaSuccess;
    // the whole tiles, one block each
    const long long whole = tiles - a.split_tiles;
    if (whole > 0) {
        gemm_f32_kernel<BN, STAGES><<<static_cast<unsigned>(whole), Cfg::THREADS,
                                      Cfg::SMEM_BYTES, stream>>>(*p.tmap_a, *p.tmap_b, a, p.ctx);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess || a.split_tiles == 0) return e;
    }
    // the stream-K tail: one block per resident slot, programmatically
    // serialised behind the whole tiles so that it fills the slots they free
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t lc{};
    lc.gridDim = dim3(static_cast<unsigned>(p.sched.sk_slots));
    lc.blockDim = dim3(Cfg::THREADS);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = attr;
    lc.numAttrs = whole > 0 ? 1 : 0;
    return cudaLaunchKernelEx(&lc, gemm_f32_streamk_kernel<BN, STAGES>, *p.tmap_a, *p.tmap_b, a,
                              p.ctx);
}

template <int BN, int STAGES>
static cudaError_t f32_slots(const LaunchCommon &p, int *slots) {
    *slots = p.sm_count * (p.blocks_per_sm > 0 ? p.blocks_per_sm : 1);
    return cudaSuccess;
}

template <int BN>
static cudaError_t launch_f32_regstage(const LaunchF32 &p, cudaStream_t stream) {
    using Cfg = F32Cfg<BN, 2>;
    GemmArgs<float, float> a{};
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
    gemm_f32_regstage_kernel<BN><<<tiles, Cfg::THREADS, 2 * Cfg::STAGE_BYTES + 1024, stream>>>(
        static_cast<const float *>(p.a_ptr), p.lda, static_cast<const float *>(p.b_ptr), p.ldb, a);
    return cudaGetLastError();
}

template <int BN>
static KernelInfo info_f32_regstage() {
    using Cfg = F32Cfg<BN, 2>;
    KernelInfo k;
    k.bm = Cfg::BM;
    k.bn = Cfg::BN;
    k.bk = Cfg::BK;
    k.stages = 2;
    k.threads = Cfg::THREADS;
    k.smem_bytes = 2 * Cfg::STAGE_BYTES + 1024;
    k.a_box_x = Cfg::BK;  // tensor maps are encoded but not used by this kernel
    k.a_box_y = Cfg::BM;
    k.b_box_x = Cfg::BN;
    k.b_box_y = Cfg::BK;
    k.a_swizzle128 = true;
    k.b_swizzle128 = false;
    k.producer = PGEMM_PRODUCER_REGISTERS;
    k.func = reinterpret_cast<const void *>(gemm_f32_regstage_kernel<BN>);
    k.launch_f32 = launch_f32_regstage<BN>;
    return k;
}

template <int BN, int STAGES>
static KernelInfo info_f32() {
    using Cfg = F32Cfg<BN, STAGES>;
    KernelInfo k;
    k.bm = Cfg::BM;
    k.bn = Cfg::BN;
    k.bk = Cfg::BK;
    k.stages = STAGES;
    k.threads = Cfg::THREADS;
    k.smem_bytes = Cfg::SMEM_BYTES;
    k.a_box_x = Cfg::BK;   // 32 floats = 128 bytes, swizzled
    k.a_box_y = Cfg::BM;
    k.b_box_x = Cfg::BN;   // BN floats (256 or 512 bytes), unswizzled
    k.b_box_y = Cfg::BK;
    k.a_swizzle128 = true;
    k.b_swizzle128 = false;
    k.stream_k = true;
    k.schedule_slots = f32_slots<BN, STAGES>;
    k.func = reinterpret_cast<const void *>(gemm_f32_kernel<BN, STAGES>);
    k.aux_func = reinterpret_cast<const void *>(gemm_f32_streamk_kernel<BN, STAGES>);
    k.launch_f32 = launch_f32_impl<BN, STAGES>;
    return k;
}

const KernelInfo *f32_kernels(int *count) {
    // S = 1 is the unpipelined comparator (load and compute strictly alternate)
    static const KernelInfo table[] = {
        info_f32<128, 2>(), info_f32<128, 3>(), info_f32<128, 4>(), info_f32<128, 5>(),
        info_f32<128, 6>(), info_f32<128, 1>(),
        // 128 x 64 tiles: 8 x 8 per thread, few enough registers for three blocks per SM
        info_f32<64, 2>(), info_f32<64, 3>(), info_f32<64, 4>(),
        // the register-staged double buffer (comparator: the pages' producer)
        info_f32_regstage<128>(), info_f32_regstage<64>()};
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace pg
