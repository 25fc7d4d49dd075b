// Shared definitions of the pipelined GEMM kernels: the argument block, the
// output-tile raster and the alpha/beta output update.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace pg {

// Sites recorded in the device status word when a bounded wait runs out.
enum WaitSite : uint32_t {
    kSiteProducerEmpty = 1,   // producer waiting for a stage to be released
    kSiteMmaAccEmpty = 2,     // MMA issuer waiting for the epilogue to free TMEM
    kSiteMmaFull = 3,         // MMA issuer waiting for a stage to land
    kSiteMmaDone = 4,         // MMA issuer draining its own MMAs before teardown
    kSiteEpilogueFull = 5,    // epilogue waiting for an accumulator
    kSiteConsumerFull = 6,    // FFMA consumer waiting for a stage to land
    kSiteConvertFull = 7,     // int8 widening warps waiting for a staged int8 tile
    kSiteConvertEmpty = 8,    // int8 widening warps waiting for a free fp16 slot
    kSiteSelfTest = 9,        // pgemm_selftest_wait_timeout
    kSiteSplitPartial = 10,   // last piece of a stream-K tile waiting for the others' partials
    kSiteWidenChunk = 11,     // TMA producer waiting for a K chunk widened inside the GEMM
};

// Problem description passed by value to every kernel.
template <typename Scalar, typename Out>
struct GemmArgs {
    int M, N, K;
    int num_m_tiles, num_n_tiles, num_k_tiles;
    int group_m;      // M-tiles per raster group (L2 reuse of B panels)
    Scalar alpha, beta;
    Out *C;           // row-major, leading dimension ldc
    long long ldc;
    int c_tma;        // 1: C is also described by a tensor map (TMA stores allowed)
    // Stream-K schedule of the persistent kernels: the K-iterations of the
    // first split_tiles output tiles (R tiles, R * T iterations laid end to
    // end) are dealt out to slots 0 .. sk_slots - 1, slot j taking
    // [j * R * T / sk_slots, (j + 1) * R * T / sk_slots): pieces of at most
    // two tiles.  The other tiles are whole units, tile R + j + i * G for
    // slot j of G.  The pieces of a tile meet through `partials` (raw partial
    // sums, one slab per slot and piece) and `counters` (zero at launch).
    // None: split_tiles = 0.  Alternatively the first half_tiles tiles are
    // each cut into two half-width units (the tile's left and right BN / 2
    // columns over all of K), on slots 0 .. 2 * half_tiles - 1: no exchange.
    int split_tiles, sk_slots;
    int half_tiles;
    uint32_t *partials;
    uint32_t *counters;
};

// Output tile `tile` -> (m0, n0).  Tiles are visited in groups of `group_m`
// M-tiles; inside a group the M index runs fastest, so the CTAs working at
// the same time share a few B column panels and a few A row panels in L2.
__device__ __forceinline__ void tile_origin(int tile, int num_m, int num_n, int group_m, int bm,
                                            int bn, int &m0, int &n0) {
    const int per_group = group_m * num_n;
    const int g = tile / per_group;
    const int first_m = g * group_m;
    const int gm = min(num_m - first_m, group_m);
    const int r = tile - g * per_group;
    m0 = (first_m + r % gm) * bm;
    n0 = (r / gm) * bn;
}

// out = alpha * acc + beta * c, with C not read when beta == 0.
__device__ __forceinline__ float axpby(float alpha, float acc, float beta, float c) {
    return fmaf(alpha, acc, beta * c);
}
__device__ __forceinline__ int32_t axpby(int32_t alpha, int32_t acc, int32_t beta, int32_t c) {
    // two's-complement arithmetic modulo 2^32
    return static_cast<int32_t>(static_cast<uint32_t>(alpha) * static_cast<uint32_t>(acc) +
                                static_cast<uint32_t>(beta) * static_cast<uint32_t>(c));
}

// One thread's output segment: row `row`, columns [col, col + 32), 32
// accumulator values held as 32-bit patterns.  Vector (16-byte) stores where
// the segment is in range and aligned, predicated scalar stores elsewhere.
template <typename Scalar, typename Out>
__device__ __forceinline__ void store_row32(const GemmArgs<Scalar, Out> &a, int row, int col,
                                            const uint32_t *acc, bool have_acc) {
    if (row >= a.M) return;
    Out *cp = a.C + static_cast<long long>(row) * a.ldc + col;
    const bool read_c = a.beta != Scalar(0);
    const bool full = (col + 32 <= a.N) && ((reinterpret_cast<uintptr_t>(cp) & 15u) == 0);
    if (full) {
#pragma unroll
        for (int v = 0; v < 8; ++v) {
            Out o[4];
            Out c[4] = {Out(0), Out(0), Out(0), Out(0)};
            if (read_c) {
                const uint4 cv = *reinterpret_cast<const uint4 *>(cp + 4 * v);
                c[0] = __builtin_bit_cast(Out, cv.x);
                c[1] = __builtin_bit_cast(Out, cv.y);
                c[2] = __builtin_bit_cast(Out, cv.z);
                c[3] = __builtin_bit_cast(Out, cv.w);
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const Out x = have_acc ? __builtin_bit_cast(Out, acc[4 * v + e]) : Out(0);
                o[e] = read_c ? axpby(a.alpha, x, a.beta, c[e]) : axpby(a.alpha, x, Scalar(0), Out(0));
            }
            uint4 ov;
            ov.x = __builtin_bit_cast(uint32_t, o[0]);
            ov.y = __builtin_bit_cast(uint32_t, o[1]);
            ov.z = __builtin_bit_cast(uint32_t, o[2]);
            ov.w = __builtin_bit_cast(uint32_t, o[3]);
            *reinterpret_cast<uint4 *>(cp + 4 * v) = ov;
        }
    } else {
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            if (col + e < a.N) {
                const Out x = have_acc ? __builtin_bit_cast(Out, acc[e]) : Out(0);
                cp[e] = read_c ? axpby(a.alpha, x, a.beta, cp[e]) : axpby(a.alpha, x, Scalar(0), Out(0));
            }
        }
    }
}

__device__ __forceinline__ uint8_t *align_1024(uint8_t *p) {
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

}  // namespace pg
