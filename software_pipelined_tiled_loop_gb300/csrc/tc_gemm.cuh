// Tensor-core GEMM kernel body shared by the bf16 and the exact-int8 paths:
// 16-bit operands (bf16, or fp16 holding widened int8), fp32 accumulators in
// tensor memory (tcgen05), fed by an S-stage TMA ring.
//
// The K-loop is the software pipeline of "Double Buffering: Software
// Pipelining the K-Loop" (sections "Two Stages, One Barrier" and "Mechanics")
// generalised to S stages and split across warps the way "Software pipelines
// and asynchronous copies" describes the state machine (sections "Prologue,
// steady state, and epilogue" and "Producer-consumer synchronization"):
//
//   warp 0 (one lane)  producer: for every K-tile t, wait empty[t % S], post
//                      the stage's byte count on full[t % S] and issue the TMA
//                      copies of the A and B panels.  The first S waits pass at
//                      once: that is the prologue, and it issues min(S, T)
//                      loads, never one beyond K.
//   warp 1 (one lane)  MMA issuer: wait full[t % S], issue BK/16 tcgen05.mma
//                      into a TMEM accumulator, then tcgen05.commit to
//                      empty[t % S] so the stage is refilled only after the
//                      tensor core has finished reading it (the reuse edge).
//                      After the last K-tile of an accumulation round it
//                      commits to acc_full (the drain).  Warp 1 owns TMEM.
//   warps 2..5         epilogue: wait acc_full, tcgen05.ld the accumulator
//                      (each warp reads its own 32-lane TMEM quadrant), then
//                      release acc_empty.
//
// An accumulation round is the whole K range of an output tile (bf16), or a
// chunk of KC K-tiles (exact int8: a chunk's fp32 partial sums of fp16
// products of int8 values stay integers of magnitude <= 2^24 and are exact;
// the epilogue converts each chunk to int32 and adds it into registers).
//
// The kernel is persistent (grid = resident blocks, each walking its own list
// of work units; the pipeline prologue is paid once per block, not once per
// tile) and TMEM holds two accumulators, so the epilogue of one round
// overlaps the main loop of the next.  A work unit is an output tile, or a
// stream-K piece of one of the tiles a partial last wave would leave over
// (GemmArgs, SlotPlan); a slot's pieces run first and meet the other pieces
// of their tiles through global memory (SplitSlab).  Stage index t % S
// and phase parity (t / S) & 1 come from a running counter, valid for any S
// (the page's XOR swap is valid for two stages only).
//
// Shared-memory layouts (both 128-byte swizzled, written by TMA):
//   A stage: BM = 128 rows (m) x 64 elements (k) -> K-major operand: rows of
//            128 B, 8-row groups 1024 B apart (SBO = 1024); K = 16 -> +32 B.
//   B stage: BN/64 boxes of 64 (n) x 64 (k) -> N-major operand: each box is
//            64 k-rows of 128 B, 8-k-row groups 1024 B apart (SBO = 1024),
//            boxes (64-column n blocks) BK*128 B apart (LBO); K = 16 -> +2048 B.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"
#include "widen.cuh"

namespace pg {

// BN: tile width; STAGES: ring depth; KC: K-tiles per accumulation round (0 =
// all of K); BF16: operand type (1 = bf16, 0 = fp16); INT_FOLD: exact-int8
// epilogue (fold fp32 chunk sums into int32 registers); EPI: epilogue warps
// (4: one per TMEM lane quadrant; 8: two per quadrant, each half the columns).
// CM: CTAs per cluster along M, CG: tcgen05 CTA group; either both 1, or both
// 2: a CTA pair computes a 256 x BN tile with one M = 256 MMA issued by the
// even CTA; each CTA loads and holds its 128 rows of A and half of B's
// columns (so a stage is a third smaller and the ring one to two stages
// deeper), and receives its 128 rows of the accumulator in its own TMEM.
// PROD: who fills the stage ring.  0: one lane of warp 0 issues TMA copies.
// 1: four producer warps (warps 0-3) load int8 A and B tiles from global
// memory into registers, widen them to fp16 there and store them into the
// swizzled stage; the separate widening pass disappears.  Then the
// epilogue warps are 4 .. 4 + EPI - 1 and the MMA issuer is warp 4 + EPI,
// and every role is a whole warpgroup, so that setmaxnreg can move
// registers from the producers and the MMA warpgroup to the epilogue.
// 2: the int8 tiles arrive by TMA in a second ring of S8 int8 stages (half
// the bytes of an fp16 stage), filled by one lane of warp 4 + EPI + 1; the
// four warps 0-3 widen each landed int8 stage into the fp16 stage the tensor
// core reads (shared memory to shared memory) in XG groups that take
// alternate K-tiles.  No widening pass, and the int8 operands cross L2 once
// at half the fp16 bytes.
// 3: the widening pass runs inside the GEMM: warps 0-3 of every CTA widen
// their share of A and B into the fp16 copies, one 64-wide K chunk after
// another, while one lane of warp 4 + EPI + 1 fills the ring by TMA from
// those copies as in 0, waiting for each K chunk to be complete in every
// CTA before it loads from it (FusedWiden).
// KSUB: 64-wide K sub-tiles per stage (1 or 2).  With two, a stage holds
// 128 K columns under one full / empty barrier pair and the MMA issuer issues
// eight MMAs per wait and commit instead of four: the per-stage bookkeeping
// of the issuer (barrier wait, commit, loop) is paid half as often.  The TMA
// boxes and the shared-memory layout of each sub-tile are those of a
// one-sub-tile stage.
template <int BN_, int STAGES_, int KC_, int BF16_, bool INT_FOLD_, int EPI_ = 4, int CM_ = 1,
          int CG_ = 1, int PROD_ = 0, int S8_ = 0, int XG_ = 1, int KSUB_ = 1>
struct TcCfg {
    static constexpr int BM = 128, BN = BN_, BK = 64, STAGES = STAGES_, KC = KC_, CM = CM_;
    static constexpr int KSUB = KSUB_;
    static constexpr int SBK = BK * KSUB;  // K columns per stage (a "K-tile" of the schedule)
    static constexpr int CG = CG_;
    static constexpr int B_COLS = BN / CG;  // B columns this CTA loads and holds
    static constexpr int BF16 = BF16_;
    static constexpr bool INT_FOLD = INT_FOLD_;
    static constexpr int EPI = EPI_;
    static constexpr int EPI_COLS = BN * 4 / EPI;  // columns per epilogue warp
    using Scalar = typename std::conditional<INT_FOLD, int32_t, float>::type;
    static constexpr int A_SUB = BM * BK * 2;      // one 64-wide sub-tile of A
    static constexpr int B_SUB = B_COLS * BK * 2;  // and of B
    static constexpr int A_BYTES = A_SUB * KSUB;
    static constexpr int B_BYTES = B_SUB * KSUB;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // per CTA
    static constexpr int TX_BYTES = STAGE_BYTES * CG;      // counted on the MMA's full barrier
    // a half-width unit (BN = 256 tiles: columns [128 h, 128 h + 128) only).
    // Not in the exact-int8 kernels: their epilogue holds 128 sums a thread,
    // and the half-width bookkeeping beside them raised the default int8
    // kernel's spills from 20 to 228 bytes of loads.
    static constexpr int STAGE_BYTES_HALF = A_BYTES + B_BYTES / 2;
    static constexpr int TX_BYTES_HALF = STAGE_BYTES_HALF * CG;
    static constexpr bool HALVES = BN_ == 256 && !INT_FOLD_ && PROD_ == 0;
    // PROD = 2: the int8 staging ring (A 128 x 64 bytes, then B as B_COLS/64
    // boxes of 64 k-rows x 64 bytes; 64-byte rows, unswizzled).
    // PROD = 3: the same ring holds the int8 boxes the widening warps convert
    // (four slots of 8 KB)
    static constexpr int S8 = PROD_ == 2 ? S8_ : (PROD_ == 3 ? 4 : 0);
    static constexpr int XG = PROD_ == 2 ? XG_ : 1;        // transform groups
    static constexpr int XG_WARPS = 4 / XG;                // warps per transform group
    static constexpr int A8_BYTES = BM * BK;               // int8
    static constexpr int STAGE8_BYTES = PROD_ == 3 ? 8192 : (BM + B_COLS) * BK;
    static constexpr int RING8_BYTES = S8 * STAGE8_BYTES;
    // Epilogue staging: one or two 32x32 fp32 blocks per epilogue warp (two
    // let a TMA store drain while the next block is staged), as many as fit.
    static constexpr int STAGE_BUFS = STAGES * STAGE_BYTES + RING8_BYTES + EPI * 2 * 4096 +
                                                  (2 * STAGES + 5 + 2 * S8) * 8 + 16 + 1024 <=
                                              232448
                                          ? 2
                                          : 1;
    static constexpr int STAGING_BYTES = EPI * STAGE_BUFS * 32 * 32 * 4;
    static constexpr int ACC_COLS = BN;        // fp32 accumulator: one TMEM column per n
    static constexpr int TMEM_COLS = 2 * BN;   // two accumulators
    static constexpr int PROD = PROD_;
    static constexpr int EPI_WARP0 = PROD ? 4 : 2;        // first epilogue warp
    static constexpr int MMA_WARP = PROD ? 4 + EPI : 1;   // MMA issuer, owns TMEM
    static constexpr int TMA8_WARP = MMA_WARP + 1;        // PROD = 2, 3: the TMA producer
    static constexpr int THREADS = PROD ? 32 * (4 + EPI + 4) : 64 + 32 * EPI;
    // arrivals that complete a stage's full barrier: the TMA producer's
    // expect_tx, or one per producer (transform) warp of each CTA
    static constexpr int FULL_ARRIVALS = PROD == 1 ? 4 * CG : (PROD == 2 ? XG_WARPS * CG : 1);
    // setmaxnreg shares of the PROD = 1 layout (launched at 65536 / THREADS)
    static constexpr int REGS_PRODUCER = 104, REGS_MMA = 48, REGS_EPILOGUE = 176;
    static constexpr int WIDEN_CHUNK = 256; // PROD = 3: K chunk (elements) published at once
    static constexpr int RING8_OFFSET = STAGES * STAGE_BYTES;
    static constexpr int STAGING_OFFSET = RING8_OFFSET + RING8_BYTES;
    static constexpr int BAR_OFFSET = STAGING_OFFSET + STAGING_BYTES;
    static constexpr int NUM_BARS = 2 * STAGES + 5 + 2 * S8;
    static constexpr int USED = BAR_OFFSET + NUM_BARS * 8 + 16;
    // TMEM has 512 columns per SM: at most 512 / TMEM_COLS blocks may share an
    // SM, or a block would stall in tcgen05.alloc.  The shared-memory request
    // is padded so that occupancy never exceeds that.
    static constexpr int MAX_BLOCKS = 512 / TMEM_COLS;
    static constexpr int SMEM_BYTES = smem_request(USED + 1024, MAX_BLOCKS);
    static_assert(BN % 64 == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(EPI == 4 || EPI == 8, "EPI");
    static_assert(EPI_COLS % 32 == 0, "epilogue column split");
    static_assert(!INT_FOLD || EPI_COLS == 128, "the int32 fold keeps 128 columns per thread");
    static_assert(!INT_FOLD || KC * SBK <= 1024, "a round's fp32 sum must stay below 2^24");
    static_assert(KSUB == 1 || (KSUB == 2 && (PROD_ == 0 || PROD_ == 3)),
                  "two sub-tiles a stage: TMA-fed kernels only");
    static_assert(USED + 1024 <= 232448, "shared memory");
    static_assert((CM == 1 && CG == 1) || (CM == 2 && CG == 2 && (BN / 64) % 2 == 0),
                  "a CTA pair is a cluster of two splitting B's columns in halves");
    static_assert(!PROD || (INT_FOLD && EPI == 8 && B_COLS % 128 == 0),
                  "register-staged producer: int8 operands, two epilogue warpgroups");
    static_assert(WIDEN_CHUNK % SBK == 0, "a K chunk holds whole K-tiles");
    static_assert(PROD != 2 || (S8 >= 2 && (XG == 1 || XG == 2) && B_COLS == 128),
                  "staged producer: an int8 ring of two or more stages, one or two groups");
    // Every use of an int8 slot must fall to the same transform group.  A
    // group waits on a slot's full barrier by phase parity; were the slot's
    // previous use another group's, this group could begin that wait while
    // the previous use's copy is still in flight (copies may land out of
    // order), two phases ahead of the barrier, and the parity would read the
    // phase before as complete.
    static_assert(PROD != 2 || S8 % XG == 0, "int8 ring depth a multiple of the groups");
    static_assert(!PROD || 128 * (REGS_PRODUCER + REGS_MMA) + 32 * EPI * REGS_EPILOGUE <=
                               65536, "setmaxnreg shares exceed the block's registers");
    static_assert(!PROD || THREADS == 512, "launched at 128 registers a thread");
};

// One warp writes a 32 x 32 block of C: rows [m_base, m_base + 32), columns
// [col, col + 32); lane t holds row m_base + t in vals[0..31] (raw
// accumulator values as 32-bit patterns; have_acc = false means zeros).  The
// block is staged in shared memory with the 128-byte swizzle (16-byte chunk
// j of row t at chunk j ^ (t % 8): conflict-free), then either
//   - written by one TMA bulk-tensor store (C describable by a tensor map and
//     beta == 0; the store clips rows/columns outside C), or
//   - written by 32 coalesced row stores (lane l writes column col + l),
//     predicated at the edges, reading C first when beta != 0.
// `buf` is this warp's staging buffer for this block: with NBUF = 2 buffers
// used in turn, the store issued into the other buffer may still be reading.
template <int NBUF, typename Scalar>
__device__ __forceinline__ void store_block32(const GemmArgs<Scalar, Scalar> &a,
                                              const CUtensorMap *tmap_c, uint8_t *buf,
                                              int m_base, int col, const uint32_t *vals,
                                              bool have_acc, bool tma_path) {
    const uint32_t lane = lane_id();
    const uint32_t sbuf = smem_u32(buf);
    if (tma_path) {
        // the store that last used this buffer must have finished reading it
        if (lane == 0) bulk_wait_read<NBUF - 1>();
        __syncwarp();
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            uint32_t o[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const Scalar x = have_acc ? __builtin_bit_cast(Scalar, vals[4 * j + e]) : Scalar(0);
                o[e] = __builtin_bit_cast(uint32_t, axpby(a.alpha, x, Scalar(0), Scalar(0)));
            }
            sts128(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(tmap_c, buf, col, m_base);
            bulk_commit();
        }
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t z = 0u;
            sts128(sbuf + lane * 128 + ((j ^ (lane & 7)) << 4), have_acc ? vals[4 * j] : z,
                   have_acc ? vals[4 * j + 1] : z, have_acc ? vals[4 * j + 2] : z,
                   have_acc ? vals[4 * j + 3] : z);
        }
        __syncwarp();
        // the block's rows inside C (none when m_base >= M) and this lane's column
        const int rows = a.M - m_base < 32 ? a.M - m_base : 32;
        const int c = col + static_cast<int>(lane);
        if (c < a.N) {
            Scalar *cp = a.C + static_cast<long long>(m_base) * a.ldc + c;
            const uint32_t rd = sbuf + (lane & 3) * 4;
            const uint32_t ch = lane >> 2;
            if (a.beta != Scalar(0)) {
#pragma unroll 4
                for (int r = 0; r < rows; ++r, cp += a.ldc) {
                    const uint32_t w = lds32(rd + r * 128 + ((ch ^ (r & 7)) << 4));
                    *cp = axpby(a.alpha, __builtin_bit_cast(Scalar, w), a.beta, *cp);
                }
            } else {
#pragma unroll 4
                for (int r = 0; r < rows; ++r, cp += a.ldc) {
                    const uint32_t w = lds32(rd + r * 128 + ((ch ^ (r & 7)) << 4));
                    *cp = axpby(a.alpha, __builtin_bit_cast(Scalar, w), Scalar(0), Scalar(0));
                }
            }
        }
        __syncwarp();
    }
}

// Hand an accumulator back to the MMA issuer: a local arrive, or with a CTA
// pair an arrive on the even CTA's barrier (remote from the odd CTA).
template <class Cfg>
__device__ __forceinline__ void release_acc(uint64_t *acc_empty_bar) {
    if constexpr (Cfg::CG == 2)
        mbar_arrive_cluster(mapa_shared(smem_u32(acc_empty_bar), 0));
    else
        mbar_arrive(acc_empty_bar);
}

// One work unit of the persistent schedule: an output tile (schedule index)
// and the K-tiles [kb, ke) it accumulates.  For a stream-K piece, part >= 0
// is its place among the `parts` slots sharing the tile, slab numbers its
// partial-sum slab (two per slot: slot * 2 + the piece's place in the slot's
// list) and slab0 the slab of the tile's piece 0.  Pieces 1, 2, ... start
// inside the tile, so each is its slot's first piece: slab (first slot + j)
// * 2; piece 0 is its slot's second piece when that slot began in the tile
// before.  half >= 0: a half-width unit, only the tile's columns
// [half * BN / 2, (half + 1) * BN / 2) over all of K.
struct WorkUnit {
    int tile, kb, ke, part, parts, slab, slab0, half;
};

// A slot's list of work units (GemmArgs: the schedule of the leftover
// tiles): first its stream-K pieces (at most two) or its half-width unit,
// then its whole tiles.  Producer, MMA issuer and epilogue walk the same
// list.  Held in shared memory and written once, with the pieces decoded in
// full there, so that walking the list costs no 64-bit divisions (and no
// registers) in the loops.
struct SlotPlan {
    int T, R, G, j;
    int n_sk, n_half, n_whole;
    WorkUnit piece[2];

    template <typename A>
    __device__ __forceinline__ void init(const A &a, int slot, int slots, int tiles) {
        T = a.num_k_tiles;
        // the leftover tiles [0, R) are split along K (stream-K pieces) or
        // along N (two half-width units each, on slots 0 .. 2R - 1); the
        // whole tiles are R + j, R + j + G, ...
        R = a.split_tiles + a.half_tiles;
        G = slots;
        j = slot;
        n_half = a.half_tiles > 0 && slot < 2 * a.half_tiles ? 1 : 0;
        const int Rk = a.split_tiles;
        const int Gs = a.sk_slots;
        const long long total = static_cast<long long>(Rk) * T;
        const bool in_sk = Rk > 0 && slot < Gs;
        const long long sk_a = in_sk ? slot * total / Gs : 0;
        const long long sk_end = in_sk ? (slot + 1) * total / Gs : 0;
        n_sk = sk_end == sk_a ? 0 : ((sk_a / T) == ((sk_end - 1) / T) ? 1 : 2);
        // the slot holding stream-K iteration x
        auto slot_of = [&](long long x) { return static_cast<int>(((x + 1) * Gs - 1) / total); };
        for (int u = 0; u < n_sk; ++u) {
            WorkUnit &w = piece[u];
            w.tile = static_cast<int>(sk_a / T) + u;
            const long long t0 = static_cast<long long>(w.tile) * T;
            const long long lo = sk_a > t0 ? sk_a : t0;
            const long long hi = sk_end < t0 + T ? sk_end : t0 + T;
            w.kb = static_cast<int>(lo - t0);
            w.ke = static_cast<int>(hi - t0);
            const int first = slot_of(t0), last = slot_of(t0 + T - 1);
            w.part = slot - first;
            w.parts = last - first + 1;
            w.slab = slot * 2 + u;
            w.slab0 = first * 2 + (first * total / Gs < t0 ? 1 : 0);
            w.half = -1;
        }
        const int whole = tiles - R;
        n_whole = slot < whole ? (whole - slot + slots - 1) / slots : 0;
    }
    __device__ __forceinline__ int units() const { return n_sk + n_half + n_whole; }
    __device__ __forceinline__ WorkUnit unit(int u) const {
        if (u < n_sk) return piece[u];
        WorkUnit w;
        w.kb = 0;
        w.ke = T;
        w.part = -1;
        w.parts = 1;
        w.slab = 0;
        w.slab0 = 0;
        w.half = -1;
        if (u < n_sk + n_half) {
            w.tile = j >> 1;
            w.half = j & 1;
            return w;
        }
        w.tile = R + j + (u - n_sk - n_half) * G;
        return w;
    }
};

// Accumulation rounds of a unit: chunks of KC K-tiles, or all of its K range.
template <class Cfg>
__device__ __forceinline__ int unit_round_tiles(const WorkUnit &w) {
    return Cfg::KC > 0 ? Cfg::KC : (w.ke > w.kb ? w.ke - w.kb : 1);
}
template <class Cfg>
__device__ __forceinline__ int unit_rounds(const WorkUnit &w) {
    const int kct = unit_round_tiles<Cfg>(w);
    return w.ke > w.kb ? (w.ke - w.kb + kct - 1) / kct : 0;
}

// Where the stream-K pieces of a tile meet, for one epilogue warp's part of
// the tile (32 rows x EPI_COLS columns): a slab of raw partial sums per
// piece (two slabs per slot, one for each of its pieces) and two counters per
// tile and warp (pieces arrived, partials written).  A warp arrives once its
// own sums are in registers.  Every piece but the last to arrive stores its
// partial into its slab and then counts it written (release); the last one
// waits until all the others are written (acquire) and adds them, in piece
// order (slot order), to its own before the alpha/beta update.  The pieces it
// waits for have arrived, so they are past every wait of their own: the
// exchange cannot deadlock whatever part of the grid is resident, and nobody
// waits on a piece that has not started.
//
// Slab layout: 16-byte group g (columns 4g .. 4g+3) of row r at word
// (g * 32 + r) * 4, so that each store or load of a warp covers 512
// consecutive bytes.
template <class Cfg>
struct SplitSlab {
    static constexpr int kSlabWords = 32 * Cfg::EPI_COLS;
    // Few registers: the int8 epilogue holds 128 sums beside this.  Pointers
    // are re-derived from the kernel arguments (WorkUnit: the slab numbers).
    int tile, part, parts, own, sub, slab0;  // sub: crank * EPI + e, this warp's share
    bool last;

    __device__ __forceinline__ SplitSlab()
        : tile(0), part(0), parts(1), own(0), sub(0), slab0(0), last(true) {}

    template <typename A>
    __device__ __forceinline__ SplitSlab(const A &a, const SlotPlan &sp, const WorkUnit &w,
                                         uint32_t crank, uint32_t e)
        : tile(w.tile), part(w.part), parts(w.parts), own(w.slab),
          sub(static_cast<int>(crank) * Cfg::EPI + static_cast<int>(e)), slab0(w.slab0) {
        uint32_t old = 0;
        if (lane_id() == 0) old = atomicAdd(counters(a), 1u);
        old = __shfl_sync(0xffffffffu, old, 0);
        last = old == static_cast<uint32_t>(parts - 1);
    }

    // [0] pieces arrived, [1] partials written
    template <typename A>
    __device__ __forceinline__ uint32_t *counters(const A &a) const {
        return a.counters + 2 * (static_cast<long long>(tile) * Cfg::CM * Cfg::EPI + sub);
    }
    template <typename A>
    __device__ __forceinline__ uint32_t *slab(const A &a, int s) const {
        return a.partials + (static_cast<long long>(s) * Cfg::CM * Cfg::EPI + sub) * kSlabWords;
    }

    // The last piece: wait until every other piece's partial is written.
    template <typename A>
    __device__ __forceinline__ bool wait_others(const A &a, const KernelCtx &ctx) const {
        bool ok = true;
        if (lane_id() == 0)
            ok = wait_counter(counters(a) + 1, static_cast<uint32_t>(parts - 1), ctx,
                              kSiteSplitPartial);
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        __syncwarp();
        __threadfence();
        return ok;
    }

    // Store 32 columns [c, c + 32) of this lane's row as this piece's partial.
    template <typename A>
    __device__ __forceinline__ void put(const A &a, int c, const uint32_t *v) const {
        uint4 *dst = reinterpret_cast<uint4 *>(slab(a, own)) + (c / 4) * 32 + lane_id();
#pragma unroll
        for (int g = 0; g < 8; ++g)
            dst[g * 32] = make_uint4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    }

    // After the last put: count this partial as written.
    template <typename A>
    __device__ __forceinline__ void publish(const A &a) const {
        __threadfence();
        __syncwarp();
        if (lane_id() == 0) red_release_add(counters(a) + 1, 1u);
    }

    // Piece j's 32 columns [c, c + 32) of this lane's row (j != part): the
    // piece of slot (this slot - part + j).
    template <typename A>
    __device__ __forceinline__ void get(const A &a, const SlotPlan &sp, int j, int c,
                                        uint32_t *v) const {
        const int s = j == 0 ? slab0 : (sp.j - part + j) * 2;
        const uint4 *src = reinterpret_cast<const uint4 *>(slab(a, s)) + (c / 4) * 32 + lane_id();
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            const uint4 x = __ldcg(src + g * 32);
            v[4 * g] = x.x;
            v[4 * g + 1] = x.y;
            v[4 * g + 2] = x.z;
            v[4 * g + 3] = x.w;
        }
    }

    // v <- the sum over all pieces of columns [c, c + 32), v holding this
    // piece's own values on entry.  fp32: added in piece order, P0 + P1 + ...,
    // whichever piece arrived last, so the result does not depend on timing.
    template <typename A>
    __device__ __forceinline__ void reduce_f32(const A &a, const SlotPlan &sp, int c,
                                               uint32_t *v) const {
        float sum[32];
        uint32_t t[32];
        for (int j = 0; j < parts; ++j) {
            if (j != part) get(a, sp, j, c, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float x = __uint_as_float(j == part ? v[i] : t[i]);
                sum[i] = j == 0 ? x : sum[i] + x;
            }
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(sum[i]);
    }

    // int32: v += every other piece's values, modulo 2^32 (order-free).
    template <typename A>
    __device__ __forceinline__ void reduce_i32(const A &a, const SlotPlan &sp, int c,
                                               uint32_t *v) const {
        uint32_t t[32];
        for (int j = 0; j < parts; ++j) {
            if (j == part) continue;
            get(a, sp, j, c, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] += t[i];
        }
    }
};

// The int8 operands as stored by the caller, for the register-staged
// producer and the in-kernel widening: row-major, pitches in elements
// (bytes), rows 16-byte aligned.  In-kernel widening (PROD = 3) also: the
// fp16 copies it writes (the TMA maps' sources) and the per-chunk counters.
struct TcOperands {
    const int8_t *A;
    const int8_t *B;
    long long lda, ldb;
    __half *A16, *B16;
    long long lda16, ldb16;
    uint32_t *ready;  // one per 64-wide K chunk, zero at launch
};

// In-kernel widening (PROD = 3).  K chunk c is A's columns [KW c, KW c + KW)
// and B's rows [KW c, KW c + KW) (KW = WIDEN_CHUNK, the last chunk possibly
// narrower), cut into 8 KB int8 boxes: A boxes of 128 rows x 64 columns
// (bytes), then B boxes of 64 rows x 128 columns.  The boxes of a chunk are
// dealt to the CTAs round-robin (box b to CTA b mod G); every CTA walks its
// boxes chunk by chunk.  One lane TMA-loads them into a four-slot int8 ring;
// the 128 threads of warps 0-3 convert each landed box to fp16 and store it
// into the fp16 copies (thread t: 16-byte pieces t, t + 128, ... of the box,
// so a warp reads 512 consecutive bytes of the box and writes whole 128-byte
// lines), release the slot, and after their last box of a chunk publish it:
// a fence (the thread's own stores; no load of the thread is in flight, the
// copies being the TMA's), then a release add on the chunk's counter by each
// warp.  The chunk is complete at 4 * gridDim.x.
struct WidenBoxes {
    int M, N, K, KW, nchunks, mb, nb;  // row blocks of A (128), column blocks of B (128)

    __device__ __forceinline__ WidenBoxes(int M_, int N_, int K_, int KW_)
        : M(M_), N(N_), K(K_), KW(KW_), nchunks((K_ + KW_ - 1) / KW_), mb((M_ + 127) / 128),
          nb((N_ + 127) / 128) {}
    // 64-wide K blocks of chunk c
    __device__ __forceinline__ int kblocks(int c) const {
        const int w = min(KW, K - c * KW);
        return (w + 63) / 64;
    }
    __device__ __forceinline__ int boxes(int c) const { return kblocks(c) * (mb + nb); }
    // box b of chunk c: operand (A or B) and the box's origin
    __device__ __forceinline__ void decode(int c, int b, bool &is_a, int &x, int &y) const {
        const int na = kblocks(c) * mb;
        is_a = b < na;
        if (is_a) {  // A: x = K column (bytes), y = row
            x = c * KW + (b % kblocks(c)) * 64;
            y = (b / kblocks(c)) * 128;
        } else {     // B: x = N column, y = K row
            const int bb = b - na;
            x = (bb % nb) * 128;
            y = c * KW + (bb / nb) * 64;
        }
    }
};

// Convert one landed 8 KB int8 box in shared memory (`box`) to fp16 in the
// destination copy, skipping the pieces beyond the matrix (K and N are
// multiples of 16, so every 16-byte piece is wholly inside or outside).
__device__ __forceinline__ void widen_box(const TcOperands &op, const WidenBoxes &wb, bool is_a,
                                          int x, int y, uint32_t box, uint32_t t) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t p = t + 128u * j;  // 16-byte piece of the box
        int r, cx;                        // row and column (bytes) of the piece in the matrix
        if (is_a) {  // 128 rows of 64 bytes: 4 pieces a row
            r = y + static_cast<int>(p >> 2);
            cx = x + static_cast<int>(p & 3u) * 16;
        } else {     // 64 rows of 128 bytes: 8 pieces a row
            r = y + static_cast<int>(p >> 3);
            cx = x + static_cast<int>(p & 7u) * 16;
        }
        const uint4 v = lds_u4(box + p * 16);
        const bool in = is_a ? (r < wb.M && cx < wb.K) : (r < wb.K && cx < wb.N);
        if (!in) continue;
        uint32_t o[8];
        widen16(v, o);
        __half *dst = is_a ? op.A16 + static_cast<long long>(r) * op.lda16 + cx
                           : op.B16 + static_cast<long long>(r) * op.ldb16 + cx;
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        d[0] = make_uint4(o[0], o[1], o[2], o[3]);
        d[1] = make_uint4(o[4], o[5], o[6], o[7]);
    }
}

// Register-staged int8 producer (PROD = 1), run by the 128 threads of warps
// 0-3 of each CTA.  For every K-tile of the slot's units it loads this CTA's
// 128 x 64 slice of A and 64 x B_COLS slice of B from global memory (16-byte
// vectors, zero outside the matrices), widens the bytes to fp16 exactly in
// registers and stores them into the stage with the same 128-byte swizzle a
// TMA copy would produce, so the MMA issuer's descriptors are unchanged.  The
// loads of the next K-tile are issued before the current one is converted
// (the register double buffer of the pages' LDG-to-register prefetch), and
// the stage ring in front of the MMA issuer is S deep as before.  Each warp
// fences its stores into the async proxy and arrives once on the stage's full
// barrier (with a CTA pair: the even CTA's, released at cluster scope).
//
// Thread t's share of a K-tile, chosen so that each 8-lane phase of a
// 16-byte shared store covers 32 distinct banks and each warp load covers
// whole 64-byte row segments:
//   A: rows (t >> 2) + 32 p, p < 4, byte chunk t & 3 of the row's 64 bytes;
//   B: rows 16 r + 4 w + ((l >> 2) & 1) + 2 ((l >> 4) & 1), r < 4, of the
//      column panel 2 h + ((l >> 3) & 1), h < B_COLS / 128, byte chunk l & 3
//      of the panel's 64 bytes (w = t >> 5, l = t & 31).
// v with its bytes n .. 15 cleared (0 < n < 16): a vector that straddles the
// end of a row (the padding of a relaid-out operand holds no values).
__device__ __forceinline__ uint4 keep_bytes(uint4 v, int n) {
    auto m = [n](int i) -> uint32_t {
        const int k = n - 4 * i;
        return k >= 4 ? 0xffffffffu : (k <= 0 ? 0u : (1u << (8 * k)) - 1u);
    };
    v.x &= m(0);
    v.y &= m(1);
    v.z &= m(2);
    v.w &= m(3);
    return v;
}

template <class Cfg>
struct RegProducer {
    static constexpr int BK = Cfg::BK, BM = Cfg::BM;
    static constexpr int NB = 4 * (Cfg::B_COLS / 128);  // B vectors per thread per K-tile
    // One K-tile's vectors as loaded, and how many bytes of each A vector and
    // of each B panel pair's vectors lie inside the matrix (the bytes past the
    // end are cleared when the tile is stored, not when it is loaded, so that
    // nothing waits for a load before the tile is needed).
    struct Tile {
        uint4 a[4], b[NB];
        int an, bn[NB / 4];
    };

    int a_row, a_col, b_row, b_col;   // this thread's base coordinates within a tile
    uint32_t a_soff, b_soff;          // its swizzled byte offsets within a stage (chunk 2q)
    uint32_t a_x, b_x;                // the row's swizzle (row & 7)

    __device__ __forceinline__ explicit RegProducer(uint32_t t) {
        const uint32_t w = t >> 5, l = t & 31u;
        a_row = static_cast<int>(t >> 2);
        a_col = static_cast<int>(t & 3u) * 16;
        a_x = (t >> 2) & 7u;
        a_soff = (t >> 2) * 128u;
        b_row = static_cast<int>(4 * w + ((l >> 2) & 1u) + 2 * ((l >> 4) & 1u));
        b_col = static_cast<int>(((l >> 3) & 1u) * 64 + (l & 3u) * 16);
        b_x = static_cast<uint32_t>(b_row) & 7u;
        b_soff = ((l >> 3) & 1u) * (BK * 128) + static_cast<uint32_t>(b_row) * 128u;
    }

    // Issue the loads of K-tile kt for the tile whose A rows start at m0 and
    // whose B columns (this CTA's share) start at nb.  Rows are 16-byte
    // aligned and padded to a multiple of 16 bytes, so a vector that starts
    // inside a row is readable whole.  Vectors outside the matrix are zero.
    __device__ __forceinline__ void load(Tile &t, const TcOperands &op, int M, int N, int K,
                                         int m0, int nb, int kt) const {
        const int k0 = kt * BK;
        t.an = K - (k0 + a_col);  // bytes of A's vectors inside the K range
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int r = m0 + a_row + 32 * p;
            t.a[p] = make_uint4(0u, 0u, 0u, 0u);
            if (r < M && t.an > 0)
                t.a[p] = ldg_nc_v4(op.A + static_cast<long long>(r) * op.lda + (k0 + a_col));
        }
#pragma unroll
        for (int h = 0; h < NB / 4; ++h) t.bn[h] = N - (nb + b_col + 128 * h);
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            const int kr = k0 + b_row + 16 * (i & 3);
            const int c = nb + b_col + 128 * (i >> 2);
            t.b[i] = make_uint4(0u, 0u, 0u, 0u);
            if (kr < K && c < N) t.b[i] = ldg_nc_v4(op.B + static_cast<long long>(kr) * op.ldb + c);
        }
    }

    // Widen and store the loaded K-tile into the stage at shared addresses
    // sa (A) and sb (B).
    __device__ __forceinline__ void store(const Tile &t, uint32_t sa, uint32_t sb) const {
        const uint32_t qa = static_cast<uint32_t>(a_col) >> 3;         // 2 q
        const uint32_t qb = (static_cast<uint32_t>(b_col) & 63u) >> 3;  // 2 q within the panel
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            uint32_t o[8];
            widen16(t.an < 16 && t.an > 0 ? keep_bytes(t.a[p], t.an) : t.a[p], o);
            const uint32_t base = sa + a_soff + 4096u * p;
            sts128(base + ((qa ^ a_x) << 4), o[0], o[1], o[2], o[3]);
            sts128(base + (((qa + 1) ^ a_x) << 4), o[4], o[5], o[6], o[7]);
        }
#pragma unroll
        for (int i = 0; i < NB; ++i) {
            uint32_t o[8];
            const int bn = t.bn[i >> 2];
            widen16(bn < 16 && bn > 0 ? keep_bytes(t.b[i], bn) : t.b[i], o);
            const uint32_t base = sb + b_soff + 2048u * (i & 3) + 2u * BK * 128u * (i >> 2);
            sts128(base + ((qb ^ b_x) << 4), o[0], o[1], o[2], o[3]);
            sts128(base + (((qb + 1) ^ b_x) << 4), o[4], o[5], o[6], o[7]);
        }
    }
};

template <class Cfg>
__global__ void __launch_bounds__(Cfg::THREADS, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmap_a,
                   const __grid_constant__ CUtensorMap tmap_b,
                   const __grid_constant__ CUtensorMap tmap_c,
                   const __grid_constant__ CUtensorMap tmap_a8,
                   const __grid_constant__ CUtensorMap tmap_b8,
                   const GemmArgs<typename Cfg::Scalar, typename Cfg::Scalar> args,
                   const TcOperands ops, const KernelCtx ctx) {
    using Scalar = typename Cfg::Scalar;
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK, STAGES = Cfg::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = align_1024(smem_raw);
    uint8_t *sA = smem;
    uint8_t *sB = smem + STAGES * Cfg::A_BYTES;
    uint8_t *sRing8 = smem + Cfg::RING8_OFFSET;  // PROD = 2: int8 stages
    uint8_t *sStage = smem + Cfg::STAGING_OFFSET;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::BAR_OFFSET);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;  // [2]
    uint64_t *acc_empty = acc_full + 2;   // [2]
    uint64_t *mma_done = acc_empty + 2;
    uint64_t *full8 = mma_done + 1;       // [S8]: an int8 stage has landed
    uint64_t *empty8 = full8 + Cfg::S8;   // [S8]: an int8 stage has been widened
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(empty8 + Cfg::S8);
    __shared__ SlotPlan sp;  // this slot's list of work units

    const uint32_t warp = warp_id_uniform();
    const uint32_t lane = lane_id();
    // Cluster geometry: with a CTA pair a "tile" of the schedule is a 2 x 1
    // stack of 128-row tiles; this CTA computes the one at its cluster rank.
    const int num_m_sched = (args.num_m_tiles + Cfg::CM - 1) / Cfg::CM;

    if (warp == 0 && lane == 0) {
        sp.init(args, static_cast<int>(blockIdx.x) / Cfg::CM, static_cast<int>(gridDim.x) / Cfg::CM,
                num_m_sched * args.num_n_tiles);
        if constexpr (Cfg::PROD != 1) {
            prefetch_tmap(&tmap_a);
            prefetch_tmap(&tmap_b);
        }
        if (args.c_tma) prefetch_tmap(&tmap_c);
        if constexpr (Cfg::PROD == 3) {
            prefetch_tmap(&tmap_a8);
            prefetch_tmap(&tmap_b8);
        }
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], Cfg::FULL_ARRIVALS);
            // released by the MMA issuer (with a CTA pair: the even CTA's, whose
            // MMAs read this CTA's stage too)
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            // with a CTA pair the even CTA's barrier counts both CTAs' epilogues
            mbar_init(&acc_empty[b], Cfg::EPI * Cfg::CG);
        }
        mbar_init(mma_done, 1);
        for (int s = 0; s < Cfg::S8; ++s) {
            mbar_init(&full8[s], 1);                 // the int8 producer's expect_tx
            mbar_init(&empty8[s], Cfg::XG_WARPS);    // the warps of the group that widens it
        }
        // (PROD = 3: XG_WARPS = 4, the four widening warps release each box)
        fence_barrier_init();
    }
    if (warp == Cfg::MMA_WARP) {
        if constexpr (Cfg::CG == 2) {
            tmem_alloc_pair(tmem_slot, Cfg::TMEM_COLS);  // both CTAs; same address in each
            tmem_relinquish_pair();
        } else {
            tmem_alloc(tmem_slot, Cfg::TMEM_COLS);
            tmem_relinquish();
        }
    }
    tc_fence_before();
    __syncwarp();
    if constexpr (Cfg::CM > 1)
        cluster_sync();  // the peer's barriers exist before anything reaches them
    else
        __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touched only on-chip state; global memory may still be
    // being written by a pre-pass launched just before (widening, repack).
    grid_dependency_wait();

    const uint32_t crank = Cfg::CM > 1 ? cluster_ctarank() : 0u;
    const int num_units = sp.units();

    // ---------------- producer: TMA into the stage ring ----------------
    // One lane runs it: warp 0 (PROD = 0), or warp MMA_WARP + 1 (PROD = 3),
    // where chunk_ready(kt) first waits until K chunk kt of the operands has
    // been widened by every CTA.
    auto tma_producer = [&](auto &&chunk_ready) {
        uint32_t it = 0;
        bool ok = true;
        for (int u = 0; ok && u < num_units; ++u) {
            const WorkUnit w = sp.unit(u);
            int m0, n0;
            tile_origin(w.tile, num_m_sched, args.num_n_tiles, args.group_m, BM * Cfg::CM, BN, m0,
                        n0);
            m0 += static_cast<int>(crank) * BM;
            for (int kt = w.kb; kt < w.ke; ++kt, ++it) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteProducerEmpty) || !chunk_ready(kt)) {
                    ok = false;
                    break;
                }
                // a half-width unit loads half of this CTA's B columns: those
                // of the unit's half of the tile
                const bool hf = Cfg::HALVES && w.half >= 0;
                const int b_cols = hf ? Cfg::B_COLS / 2 : Cfg::B_COLS;
                const int nb = n0 + (hf ? w.half * (BN / 2) : 0) + static_cast<int>(crank) * b_cols;
                if constexpr (Cfg::CG == 2) {
                    // Both CTAs load their A rows and B columns into their own
                    // shared memory; the bytes are counted on the even CTA's
                    // full barrier, which its producer arms for both.
                    const uint32_t full_lead = mapa_shared(smem_u32(&full[s]), 0);
                    if (crank == 0)
                        mbar_arrive_expect_tx(&full[s], hf ? Cfg::TX_BYTES_HALF : Cfg::TX_BYTES);
#pragma unroll
                    for (int q = 0; q < Cfg::KSUB; ++q) {
                        const int k0 = kt * Cfg::SBK + q * BK;
                        tma_load_2d_pair(sA + s * Cfg::A_BYTES + q * Cfg::A_SUB, &tmap_a, full_lead,
                                         k0, m0);
                        for (int j = 0; j < b_cols / 64; ++j)
                            tma_load_2d_pair(sB + s * Cfg::B_BYTES + q * Cfg::B_SUB + j * (BK * 128),
                                             &tmap_b, full_lead, nb + j * 64, k0);
                    }
                    continue;
                }
                mbar_arrive_expect_tx(&full[s], hf ? Cfg::STAGE_BYTES_HALF : Cfg::STAGE_BYTES);
#pragma unroll
                for (int q = 0; q < Cfg::KSUB; ++q) {
                    const int k0 = kt * Cfg::SBK + q * BK;
                    tma_load_2d(sA + s * Cfg::A_BYTES + q * Cfg::A_SUB, &tmap_a, &full[s], k0, m0);
                    for (int j = 0; j < b_cols / 64; ++j)
                        tma_load_2d(sB + s * Cfg::B_BYTES + q * Cfg::B_SUB + j * (BK * 128), &tmap_b,
                                    &full[s], nb + j * 64, k0);
                }
            }
        }
        if constexpr (Cfg::CM > 1) {
            // Producer tail: wait for the last release of every stage.  Those
            // are the pair MMA issuer's multicast arrivals on this CTA's
            // barriers, so none can land after the cluster has been left.
            for (int i = 0; ok && i < STAGES; ++i, ++it) {
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                ok = mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteProducerEmpty);
            }
        }
    };


    if (Cfg::PROD ? warp < 4 : warp == 0) {
        if constexpr (Cfg::PROD == 3) {
            // ------- the widening pass, inside the GEMM (warps 0-3) -------
            setmaxnreg_dec<Cfg::REGS_PRODUCER>();
            const WidenBoxes wb(args.M, args.N, args.K, Cfg::WIDEN_CHUNK);
            const int G = static_cast<int>(gridDim.x);
            uint32_t it = 0;  // this CTA's boxes so far (ring position)
            bool ok = true;
            for (int c = 0; c < wb.nchunks; ++c) {
                const int nbx = wb.boxes(c);
                for (int b = static_cast<int>(blockIdx.x); ok && b < nbx; b += G, ++it) {
                    const uint32_t s8 = it % Cfg::S8, ph8 = (it / Cfg::S8) & 1u;
                    if (!mbar_wait(&full8[s8], ph8, ctx, kSiteConvertFull)) {
                        ok = false;
                        break;
                    }
                    bool is_a;
                    int x, y;
                    wb.decode(c, b, is_a, x, y);
                    widen_box(ops, wb, is_a, x, y, smem_u32(sRing8 + s8 * Cfg::STAGE8_BYTES),
                              threadIdx.x);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty8[s8]);  // the box has been read
                }
                if (!ok) break;
                // this warp's share of chunk c is written: publish it
                __threadfence();
                fence_proxy_async_global();
                __syncwarp();
                if (lane == 0) red_release_add(ops.ready + c, 1u);
            }
        } else if constexpr (Cfg::PROD == 2) {
            // ------- int8 stages widened into fp16 stages (warps 0-3) -------
            // Group g of XG takes the slot's K-tiles g, g + XG, ...  For each:
            // wait until its int8 stage has landed and its fp16 slot has been
            // read by the tensor core, widen the stage's 64-byte rows (A's 128,
            // then B's 64-row boxes) into the fp16 slot's 128-byte rows with
            // the 128-byte swizzle TMA would write, fence the stores into the
            // async proxy, then release the int8 stage and arrive once per
            // warp on the MMA issuer's full barrier (with a CTA pair the even
            // CTA's, at cluster scope).  Thread t of a group takes the stage's
            // 16-byte chunks t, t + TG, ...: each warp load reads 512
            // consecutive bytes, and every 8-lane phase of a 16-byte store
            // covers rows r and r + 1 of one 8-row swizzle group, 32 distinct
            // banks.
            setmaxnreg_dec<Cfg::REGS_PRODUCER>();
            constexpr int TG = Cfg::XG_WARPS * 32;             // threads per group
            constexpr int PER = Cfg::STAGE8_BYTES / 16 / TG;   // chunks per thread
            static_assert(PER % 8 == 0, "chunks per thread");
            const uint32_t g = warp / Cfg::XG_WARPS;
            const uint32_t tg = (warp % Cfg::XG_WARPS) * 32u + lane;
            const uint32_t x = (tg >> 2) & 7u;  // the swizzle of every row this thread writes
            const uint32_t c2 = (tg & 3u) * 2u; // fp16 chunks c2, c2 + 1 of the row
            const uint32_t lo_off = (c2 ^ x) << 4, hi_off = ((c2 + 1u) ^ x) << 4;
            int total = 0;  // K-tiles of this slot
            for (int u = 0; u < num_units; ++u) {
                const WorkUnit w = sp.unit(u);
                total += w.ke - w.kb;
            }
            bool ok = true;
            for (int it = static_cast<int>(g); it < total; it += Cfg::XG) {
                const uint32_t s8 = it % Cfg::S8, ph8 = (it / Cfg::S8) & 1u;
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                // every lane observes the int8 stage's completion (TMA bytes)
                if (!mbar_wait(&full8[s8], ph8, ctx, kSiteConvertFull)) {
                    ok = false;
                    break;
                }
                bool fr = true;
                if (lane == 0) fr = mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteConvertEmpty);
                if (__shfl_sync(0xffffffffu, fr ? 1 : 0, 0) == 0) {
                    ok = false;
                    break;
                }
                const uint32_t src = smem_u32(sRing8 + s8 * Cfg::STAGE8_BYTES) + tg * 16u;
                const uint32_t dA = smem_u32(sA + s * Cfg::A_BYTES);
                const uint32_t dB = smem_u32(sB + s * Cfg::B_BYTES);
#pragma unroll
                for (int h = 0; h < PER; h += 8) {
                    uint4 v[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) v[j] = lds_u4(src + (h + j) * TG * 16);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t r = (tg >> 2) + (h + j) * (TG / 4);  // 64-byte row
                        const uint32_t row = r < BM ? dA + r * 128u : dB + (r - BM) * 128u;
                        uint32_t o[8];
                        widen16(v[j], o);
                        sts128(row + lo_off, o[0], o[1], o[2], o[3]);
                        sts128(row + hi_off, o[4], o[5], o[6], o[7]);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&empty8[s8]);
                    if constexpr (Cfg::CG == 2)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&full[s]), 0));
                    else
                        mbar_arrive(&full[s]);
                }
            }
            if constexpr (Cfg::CM > 1) {
                // the last multicast releases of the fp16 ring land before the exit
                if (threadIdx.x == 0)
                    for (int i = 0; ok && i < STAGES; ++i) {
                        const int t2 = total + i;
                        ok = mbar_wait(&empty[t2 % STAGES], ((t2 / STAGES) & 1u) ^ 1u, ctx,
                                       kSiteConvertEmpty);
                    }
            }
        } else if constexpr (Cfg::PROD == 1) {
            // ------- producer: int8 loads widened in registers (warps 0-3) -------
            setmaxnreg_dec<Cfg::REGS_PRODUCER>();
            const RegProducer<Cfg> rp(threadIdx.x);
            using Tile = typename RegProducer<Cfg>::Tile;
            Tile x, y;  // two K-tiles in registers, used in turn
            // The slot's K-tiles in order: unit u, K-tile kt < ke, and the
            // unit's A row and B column origins for this CTA.
            int u = -1, kt = -1, ke = 0, m0 = 0, nb = 0;
            auto advance = [&](int &uu, int &k, int &kend, int &m, int &n) -> bool {
                ++k;
                while (k >= kend) {
                    if (++uu >= num_units) return false;
                    const WorkUnit w = sp.unit(uu);
                    k = w.kb;
                    kend = w.ke;
                    tile_origin(w.tile, num_m_sched, args.num_n_tiles, args.group_m,
                                BM * Cfg::CM, BN, m, n);
                    m += static_cast<int>(crank) * BM;
                    n += static_cast<int>(crank) * Cfg::B_COLS;
                }
                return true;
            };
            uint32_t it = 0;
            bool ok = true;
            // Store the K-tile held in `now` into the next stage; before that,
            // issue the loads of the one after it into `next`.  Returns
            // whether there is a next one.
            auto step = [&](Tile &now, Tile &next) -> bool {
                int u2 = u, kt2 = kt, ke2 = ke, m2 = m0, n2 = nb;
                const bool have2 = advance(u2, kt2, ke2, m2, n2);
                if (have2) rp.load(next, ops, args.M, args.N, args.K, m2, n2, kt2);
                const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteProducerEmpty);
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                if (!ok) return false;
                rp.store(now, smem_u32(sA + s * Cfg::A_BYTES), smem_u32(sB + s * Cfg::B_BYTES));
                // the stores become visible to the tensor core's reads, then
                // one arrival per warp
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (Cfg::CG == 2)
                        mbar_arrive_cluster(mapa_shared(smem_u32(&full[s]), 0));
                    else
                        mbar_arrive(&full[s]);
                }
                ++it;
                u = u2;
                kt = kt2;
                ke = ke2;
                m0 = m2;
                nb = n2;
                return have2;
            };
            bool have = advance(u, kt, ke, m0, nb);
            if (have) rp.load(x, ops, args.M, args.N, args.K, m0, nb, kt);
            while (have && step(x, y)) have = step(y, x);
            if constexpr (Cfg::CM > 1) {
                // as below: the last multicast releases land before the exit
                if (threadIdx.x == 0)
                    for (int i = 0; ok && i < STAGES; ++i, ++it) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        ok = mbar_wait(&empty[s], ph ^ 1u, ctx, kSiteProducerEmpty);
                    }
            }
        } else if (lane == 0) {
            tma_producer([](int) { return true; });
        }
    } else if (Cfg::PROD ? warp >= static_cast<uint32_t>(Cfg::MMA_WARP) : warp == 1) {
        if constexpr (Cfg::PROD) setmaxnreg_dec<Cfg::REGS_MMA>();  // the MMA warpgroup
        if constexpr (Cfg::PROD == 3) {
            if (warp == Cfg::TMA8_WARP + 1 && lane == 0) {
                // ------- the widening's int8 boxes by TMA into the int8 ring -------
                const WidenBoxes wb(args.M, args.N, args.K, Cfg::WIDEN_CHUNK);
                const int G = static_cast<int>(gridDim.x);
                uint32_t it = 0;
                bool ok = true;
                for (int c = 0; ok && c < wb.nchunks; ++c) {
                    const int nbx = wb.boxes(c);
                    for (int b = static_cast<int>(blockIdx.x); b < nbx; b += G, ++it) {
                        const uint32_t s8 = it % Cfg::S8, ph8 = (it / Cfg::S8) & 1u;
                        if (!mbar_wait(&empty8[s8], ph8 ^ 1u, ctx, kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        bool is_a;
                        int x, y;
                        wb.decode(c, b, is_a, x, y);
                        mbar_arrive_expect_tx(&full8[s8], Cfg::STAGE8_BYTES);
                        tma_load_2d(sRing8 + s8 * Cfg::STAGE8_BYTES, is_a ? &tmap_a8 : &tmap_b8,
                                    &full8[s8], x, y);
                    }
                }
            }
            if (warp == Cfg::TMA8_WARP && lane == 0) {
                // K chunks complete in order for every warp that widens, so
                // chunk kt complete means every chunk before it is too
                int ready_upto = 0;
                const uint32_t target = 4u * gridDim.x;
                tma_producer([&](int kt) -> bool {
                    const int c = kt * Cfg::SBK / Cfg::WIDEN_CHUNK;  // the K chunk holding K-tile kt
                    if (c < ready_upto) return true;
                    if (!wait_counter(ops.ready + c, target, ctx, kSiteWidenChunk)) return false;
                    fence_proxy_async_global();  // the TMA copies below read what was published
                    ready_upto = c + 1;
                    return true;
                });
            }
        }
        if constexpr (Cfg::PROD == 2) {
            if (warp == Cfg::TMA8_WARP && lane == 0) {
                // ---------------- producer: int8 tiles by TMA into the int8 ring ----------------
                // Each CTA loads its own 128 rows of A and B_COLS columns of B
                // (two 64-byte-wide boxes) into its own int8 stage, counted on
                // its own barrier; the bytes outside the matrices arrive as zeros.
                uint32_t it = 0;
                bool ok = true;
                for (int u = 0; ok && u < num_units; ++u) {
                    const WorkUnit w = sp.unit(u);
                    int m0, n0;
                    tile_origin(w.tile, num_m_sched, args.num_n_tiles, args.group_m, BM * Cfg::CM,
                                BN, m0, n0);
                    m0 += static_cast<int>(crank) * BM;
                    const int nb = n0 + static_cast<int>(crank) * Cfg::B_COLS;
                    for (int kt = w.kb; kt < w.ke; ++kt, ++it) {
                        const uint32_t s8 = it % Cfg::S8, ph8 = (it / Cfg::S8) & 1u;
                        if (!mbar_wait(&empty8[s8], ph8 ^ 1u, ctx, kSiteProducerEmpty)) {
                            ok = false;
                            break;
                        }
                        uint8_t *dst = sRing8 + s8 * Cfg::STAGE8_BYTES;
                        mbar_arrive_expect_tx(&full8[s8], Cfg::STAGE8_BYTES);
                        tma_load_2d(dst, &tmap_a, &full8[s8], kt * BK, m0);
#pragma unroll
                        for (int j = 0; j < Cfg::B_COLS / 64; ++j)
                            tma_load_2d(dst + Cfg::A8_BYTES + j * (64 * BK), &tmap_b, &full8[s8],
                                        nb + j * 64, kt * BK);
                    }
                }
            }
        }
        // with a CTA pair only the even CTA issues (its MMAs cover both CTAs)
        if (warp == Cfg::MMA_WARP && lane == 0 && (Cfg::CG == 1 || crank == 0)) {
            // ---------------- MMA issuer ----------------
            constexpr uint32_t idesc_full = idesc_f16(BM * Cfg::CG, BN, Cfg::BF16, /*A K-major*/ 0,
                                                      /*B N-major*/ 1);
            constexpr uint32_t idesc_half = idesc_f16(BM * Cfg::CG, BN / 2, Cfg::BF16, 0, 1);
            constexpr uint16_t kPair = 3;  // both CTAs of the pair
            uint32_t it = 0, gr = 0;
            bool ok = true;
            for (int u = 0; ok && u < num_units; ++u) {
                const WorkUnit w = sp.unit(u);
                const int kct = unit_round_tiles<Cfg>(w);
                const int rounds = unit_rounds<Cfg>(w);
                // a half-width unit: N = BN / 2 into the accumulator's first columns
                const uint32_t idesc = (Cfg::HALVES && w.half >= 0) ? idesc_half : idesc_full;
                for (int r = 0; ok && r < rounds; ++r, ++gr) {
                    const uint32_t ab = gr & 1u, aph = (gr >> 1) & 1u;
                    if (!mbar_wait(&acc_empty[ab], aph ^ 1u, ctx, kSiteMmaAccEmpty)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + ab * Cfg::ACC_COLS;
                    const int k_begin = w.kb + r * kct;
                    const int k_end = min(w.ke, k_begin + kct);
                    for (int kt = k_begin; kt < k_end; ++kt, ++it) {
                        const uint32_t s = it % STAGES, ph = (it / STAGES) & 1u;
                        // register-staged stages of a pair: the odd CTA's warps
                        // released their stores at cluster scope
                        const bool landed = (Cfg::PROD && Cfg::CG == 2)
                                                ? mbar_wait_cluster(&full[s], ph, ctx, kSiteMmaFull)
                                                : mbar_wait(&full[s], ph, ctx, kSiteMmaFull);
                        if (!landed) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const bool first = kt == k_begin;
#pragma unroll
                        for (int q = 0; q < Cfg::KSUB; ++q) {
                            // a sub-tile wholly beyond K holds only zero fill
                            if (q > 0 && kt * Cfg::SBK + q * BK >= args.K) break;
                            const uint32_t a_addr = smem_u32(sA + s * Cfg::A_BYTES + q * Cfg::A_SUB);
                            const uint32_t b_addr = smem_u32(sB + s * Cfg::B_BYTES + q * Cfg::B_SUB);
#pragma unroll
                            for (int k = 0; k < BK / 16; ++k) {
                                const uint64_t ad = smem_desc_sw128(a_addr + k * 32, 16, 1024);
                                const uint64_t bd =
                                    smem_desc_sw128(b_addr + k * 2048, BK * 128, 1024);
                                const uint32_t acc = (first && q == 0 && k == 0) ? 0u : 1u;
                                if constexpr (Cfg::CG == 2)
                                    umma_f16_ss_pair(d_tmem, ad, bd, idesc, acc);
                                else
                                    umma_f16_ss(d_tmem, ad, bd, idesc, acc);
                            }
                        }
                        // stage s is free once these MMAs have read it (in both CTAs
                        // of a pair)
                        if constexpr (Cfg::CG == 2)
                            umma_commit_pair_multicast(&empty[s], kPair);
                        else
                            umma_commit(&empty[s]);
                    }
                    // round complete -> epilogue (of both CTAs, with a pair)
                    if (ok) {
                        if constexpr (Cfg::CG == 2)
                            umma_commit_pair_multicast(&acc_full[ab], kPair);
                        else
                            umma_commit(&acc_full[ab]);
                    }
                }
            }
            if constexpr (Cfg::CG == 2)
                umma_commit_pair_multicast(mma_done, 1);  // this CTA's barrier only
            else
                umma_commit(mma_done);
            mbar_wait(mma_done, 0, ctx, kSiteMmaDone);
        }
    } else {
        // ---------------- epilogue warps ----------------
        if constexpr (Cfg::PROD) setmaxnreg_inc<Cfg::REGS_EPILOGUE>();
        const uint32_t e = warp - Cfg::EPI_WARP0;  // epilogue warp index
        const uint32_t q = warp & 3u;           // the TMEM lane quadrant this warp may read
        const int col0 = static_cast<int>(e >> 2) * Cfg::EPI_COLS;  // its column range
        uint8_t *wbuf = sStage + e * (Cfg::STAGE_BUFS * 32 * 32 * 4);  // this warp's buffers
        uint32_t nstore = 0;  // blocks this warp has stored (selects the buffer)
        auto next_buf = [&]() -> uint8_t * {
            return wbuf + (nstore++ % Cfg::STAGE_BUFS) * (32 * 32 * 4);
        };
        const bool tma_path = args.c_tma && args.beta == Scalar(0);
        uint32_t gr = 0;
        bool ok = true;
        // The unit's place in C: rows [m_base, m_base + 32) of this warp's
        // quadrant, columns from n0 (rows below C take no part, and a
        // stream-K piece there exchanges nothing: the same for every piece).
        // A half-width unit's accumulator columns [0, BN / 2) are C's columns
        // from n0 + half * BN / 2; warps whose columns lie beyond BN / 2 have
        // nothing of it (idle()), but still pass each accumulator back.
        auto place = [&](const WorkUnit &w, int &m_base, int &n0, bool &in_range, bool &split) {
            int m0;
            tile_origin(w.tile, num_m_sched, args.num_n_tiles, args.group_m, BM * Cfg::CM, BN, m0, n0);
            if (Cfg::HALVES && w.half >= 0) n0 += w.half * (BN / 2);
            m0 += static_cast<int>(crank) * BM;
            in_range = m0 < args.M;  // the second tile of a pair may lie below C
            m_base = m0 + static_cast<int>(q * 32);
            split = w.part >= 0 && in_range;
        };
        auto idle = [&](const WorkUnit &w) { return Cfg::HALVES && w.half >= 0 && col0 >= BN / 2; };
        for (int u = 0; ok && u < num_units; ++u) {
            if constexpr (Cfg::INT_FOLD) {
                const int rounds = unit_rounds<Cfg>(sp.unit(u));
                const bool no_cols = idle(sp.unit(u));
                // Exact int8: sum the rounds' integer-valued fp32 partials in
                // int32.  Rounds of at most 256 products (|x| <= 2^22) convert
                // with one FADD: for an integer-valued x with |x| <= 2^22,
                // x + 1.5*2^23 is exact and its bit pattern is 0x4B400000 + x
                // (the 0x4B400000 of every round is subtracted once at the
                // end).  Longer rounds (up to 1024 products, |x| <= 2^24) use
                // the exact float-to-int conversion, which is slower per value
                // but needed 4x less often.
                constexpr bool kMagicFold = Cfg::KC * Cfg::SBK <= 256;
                constexpr float kMagic = 12582912.0f;  // 1.5 * 2^23
                uint32_t acc[Cfg::EPI_COLS];
#pragma unroll
                for (int j = 0; j < Cfg::EPI_COLS; ++j) acc[j] = 0u;
                for (int r = 0; r < rounds; ++r, ++gr) {
                    const uint32_t ab = gr & 1u, aph = (gr >> 1) & 1u;
                    if (!mbar_wait(&acc_full[ab], aph, ctx, kSiteEpilogueFull)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t t_row =
                        tmem_base + ((q * 32u) << 16) + ab * Cfg::ACC_COLS + col0;
                    if (!no_cols) {
#pragma unroll
                        for (int c = 0; c < Cfg::EPI_COLS; c += 16) {
                            uint32_t v[16];
                            tmem_ld_32x32b_x16(t_row + c, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                if constexpr (kMagicFold)
                                    acc[c + j] += __float_as_uint(__uint_as_float(v[j]) + kMagic);
                                else
                                    acc[c + j] +=
                                        static_cast<uint32_t>(__float2int_rn(__uint_as_float(v[j])));
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) release_acc<Cfg>(&acc_empty[ab]);
                }
                if (!ok) break;
                const uint32_t bias =
                    kMagicFold ? static_cast<uint32_t>(rounds) * 0x4B400000u : 0u;  // mod 2^32
#pragma unroll
                for (int j = 0; j < Cfg::EPI_COLS; ++j) acc[j] -= bias;
                // the unit again, from the shared plan: nothing of it stays in
                // registers while the 128 sums are built
                const WorkUnit w = sp.unit(u);
                int m_base, n0;
                bool in_range, split;
                place(w, m_base, n0, in_range, split);
                if (no_cols) continue;
                if (split) {
                    const SplitSlab<Cfg> slab(args, sp, w, crank, e);
                    if (!slab.last) {
#pragma unroll
                        for (int c = 0; c < Cfg::EPI_COLS; c += 32) slab.put(args, c, acc + c);
                        slab.publish(args);
                        continue;
                    }
                    if (!slab.wait_others(args, ctx)) break;
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_COLS; c += 32) slab.reduce_i32(args, sp, c, acc + c);
                }
                if (in_range) {
#pragma unroll
                    for (int c = 0; c < Cfg::EPI_COLS; c += 32)
                        store_block32<Cfg::STAGE_BUFS>(args, &tmap_c, next_buf(), m_base, n0 + col0 + c, acc + c,
                                      rounds > 0, tma_path);
                }
            } else {
                const WorkUnit w = sp.unit(u);
                const int rounds = unit_rounds<Cfg>(w);
                int m_base, n0;
                bool in_range, split;
                place(w, m_base, n0, in_range, split);
                if (rounds > 0) {
                    const uint32_t ab = gr & 1u, aph = (gr >> 1) & 1u;
                    if (!mbar_wait(&acc_full[ab], aph, ctx, kSiteEpilogueFull)) break;
                    tc_fence_after();
                    if (idle(w)) {
                        // none of this half-width unit's columns is this warp's
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) release_acc<Cfg>(&acc_empty[ab]);
                        ++gr;
                        continue;
                    }
                    const uint32_t t_row =
                        tmem_base + ((q * 32u) << 16) + ab * Cfg::ACC_COLS + col0;
                    // role in a stream-K tile: store a partial, or add them all
                    int role = 0;  // 0: whole tile, 1: store partial, 2: reduce
                    SplitSlab<Cfg> slab = split ? SplitSlab<Cfg>(args, sp, w, crank, e) : SplitSlab<Cfg>();
                    if (split) {
                        role = slab.last ? 2 : 1;
                        if (role == 2 && !slab.wait_others(args, ctx)) ok = false;
                    }
#pragma unroll 1
                    for (int c = 0; c < Cfg::EPI_COLS; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(t_row + c, v);
                        tmem_ld_wait();
                        if (c + 32 >= Cfg::EPI_COLS) {
                            // last TMEM read of this accumulator: hand it back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0) release_acc<Cfg>(&acc_empty[ab]);
                        }
                        if (!ok) continue;
                        if (role == 1) {
                            slab.put(args, c, v);
                            continue;
                        }
                        if (role == 2) slab.reduce_f32(args, sp, c, v);
                        if (in_range)
                            store_block32<Cfg::STAGE_BUFS>(args, &tmap_c, next_buf(), m_base, n0 + col0 + c, v, true,
                                          tma_path);
                    }
                    if (role == 1) slab.publish(args);
                    ++gr;
                } else if (!idle(w)) {
                    // K == 0: C = beta * C, tensor memory is never read
                    uint32_t zero[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) zero[j] = 0u;
#pragma unroll 1
                    for (int c = 0; in_range && c < Cfg::EPI_COLS; c += 32)
                        store_block32<Cfg::STAGE_BUFS>(args, &tmap_c, next_buf(), m_base, n0 + col0 + c, zero, false,
                                      tma_path);
                }
            }
        }
        if (lane == 0) bulk_wait_all();  // this warp's C stores have landed
        __syncwarp();
    }

    // ---------------- teardown ----------------
    tc_fence_before();
    __syncwarp();
    if constexpr (Cfg::CM > 1)
        cluster_sync();  // no CTA leaves while its peer may still signal it
    else
        __syncthreads();
    if (warp == Cfg::MMA_WARP) {
        __syncwarp();
        tc_fence_after();
        if constexpr (Cfg::CG == 2)
            tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
        else
            tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
}

// ----------------------------------------------------------------- host ---
template <class Cfg, class P>
static cudaError_t launch_tc(const P &p, cudaStream_t stream) {
    GemmArgs<typename Cfg::Scalar, typename Cfg::Scalar> a{};
    a.M = p.M;
    a.N = p.N;
    a.K = p.K;
    a.num_m_tiles = (p.M + Cfg::BM - 1) / Cfg::BM;
    a.num_n_tiles = (p.N + Cfg::BN - 1) / Cfg::BN;
    a.num_k_tiles = (p.K + Cfg::SBK - 1) / Cfg::SBK;
    // Raster groups of 16 tile rows up to K = 4096, else 8.  On the pair
    // with 128-column stages: int8 4096^3 100.1-100.4 us with 16 against
    // 101.1-102.0 with 8, bf16 4096^3 86.0-87.1 against 86.9-88.1; bf16
    // 4096^2 x 16384 304.2-306.2 us with 8 against 309.3-310.5 with 16 (a
    // group of 16 pair rows then holds 128 MiB of A); bf16 8192^3 the same
    // time with 8 or 16 and 1063 against 1253 MB read from DRAM with 8.
    a.group_m = p.group_m > 0 ? p.group_m : (p.K <= 4096 ? 16 : 8);
    a.alpha = p.alpha;
    a.beta = p.beta;
    a.C = p.C;
    a.ldc = p.ldc;
    a.c_tma = p.tmap_c != nullptr ? 1 : 0;
    const TileSchedule &sc = p.sched;
    a.split_tiles = static_cast<int>(sc.split_tiles);
    a.half_tiles = static_cast<int>(sc.half_tiles);
    a.sk_slots = sc.sk_slots;
    a.partials = sc.partials;
    a.counters = sc.counters;
    const CUtensorMap &tc = p.tmap_c != nullptr ? *p.tmap_c : *p.tmap_a;
    // After a pre-pass of this call, launch with programmatic stream
    // serialisation: the prologue overlaps the pre-pass's tail, and every
    // thread waits for it (grid_dependency_wait) before touching memory.
    cudaLaunchAttribute attr[3];
    int nattr = 0;
    if (p.after_prepass) {
        attr[nattr].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[nattr].val.programmaticStreamSerializationAllowed = 1;
        ++nattr;
    }
    cudaLaunchConfig_t lc{};
    lc.blockDim = dim3(Cfg::THREADS);
    lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
    lc.stream = stream;
    lc.attrs = attr;
    // one CTA (or CTA pair) per schedule slot, at most one per work unit
    // every slot when pieces are dealt out (the plan is made for sc.slots),
    // else at most one slot per tile
    const long long units = sc.split_tiles > 0 ? sc.slots : sc.tiles + sc.half_tiles;
    const int grid_units = static_cast<int>(units < sc.slots ? units : sc.slots);
    if (grid_units < 1) return cudaSuccess;
    lc.gridDim = dim3(Cfg::CM * grid_units);
    if constexpr (Cfg::CM > 1) {
        attr[nattr].id = cudaLaunchAttributeClusterDimension;
        attr[nattr].val.clusterDim.x = Cfg::CM;
        attr[nattr].val.clusterDim.y = 1;
        attr[nattr].val.clusterDim.z = 1;
        ++nattr;
    }
    lc.numAttrs = nattr;
    TcOperands ops{};
    if constexpr (Cfg::PROD != 0) {
        // setmaxnreg.inc waits until the block's pool can grant the
        // registers, and the pool is what the kernel was launched with:
        // launch only if the shares fit it, so that no warpgroup can wait
        // for registers that will never come.
        static const bool regs_fit = [] {
            cudaFuncAttributes fa{};
            return cudaFuncGetAttributes(&fa, tc_gemm_kernel<Cfg>) == cudaSuccess &&
                   fa.numRegs * Cfg::THREADS >= 128 * (Cfg::REGS_PRODUCER + Cfg::REGS_MMA) +
                                                    32 * Cfg::EPI * Cfg::REGS_EPILOGUE;
        }();
        if (!regs_fit) return cudaErrorInvalidConfiguration;
    }
    if constexpr (Cfg::PROD == 3) {
        // every CTA's widening feeds every CTA's loads: all must be resident
        attr[nattr].id = cudaLaunchAttributeCooperative;
        attr[nattr].val.cooperative = 1;
        ++nattr;
        lc.numAttrs = nattr;
        ops.A = static_cast<const int8_t *>(p.widen_src_a);
        ops.B = static_cast<const int8_t *>(p.widen_src_b);
        ops.lda = p.widen_lda;
        ops.ldb = p.widen_ldb;
        ops.A16 = static_cast<__half *>(const_cast<void *>(p.a_ptr));
        ops.B16 = static_cast<__half *>(const_cast<void *>(p.b_ptr));
        ops.lda16 = p.lda;
        ops.ldb16 = p.ldb;
        ops.ready = p.widen_ready;
    }
    if constexpr (Cfg::PROD == 1) {
        ops.A = static_cast<const int8_t *>(p.a_ptr);
        ops.B = static_cast<const int8_t *>(p.b_ptr);
        ops.lda = p.lda;
        ops.ldb = p.ldb;
    }
    // the widening's int8 maps (PROD = 3); any valid map for the others
    const CUtensorMap &ta8 = p.tmap_a8 != nullptr ? *p.tmap_a8 : *p.tmap_a;
    const CUtensorMap &tb8 = p.tmap_b8 != nullptr ? *p.tmap_b8 : *p.tmap_b;
    return cudaLaunchKernelEx(&lc, tc_gemm_kernel<Cfg>, *p.tmap_a, *p.tmap_b, tc, ta8, tb8, a, ops,
                              p.ctx);
}

// Schedule slots of a persistent launch: resident CTAs (at most MAX_BLOCKS per
// SM, the TMEM limit), or resident clusters for a CTA pair.
template <class Cfg>
static cudaError_t tc_slots(const LaunchCommon &p, int *slots) {
    if constexpr (Cfg::CM == 1) {
        const int per_sm = p.blocks_per_sm < Cfg::MAX_BLOCKS ? p.blocks_per_sm : Cfg::MAX_BLOCKS;
        *slots = p.sm_count * (per_sm > 0 ? per_sm : 1);
        return cudaSuccess;
    } else {
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = Cfg::CM;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cudaLaunchConfig_t lc{};
        lc.blockDim = dim3(Cfg::THREADS);
        lc.dynamicSmemBytes = Cfg::SMEM_BYTES;
        lc.gridDim = dim3(Cfg::CM * p.sm_count);
        lc.attrs = attr;
        lc.numAttrs = 1;
        int clusters = 0;
        cudaError_t e = cudaOccupancyMaxActiveClusters(&clusters, tc_gemm_kernel<Cfg>, &lc);
        if (e != cudaSuccess) return e;
        if (clusters < 1) return cudaErrorInvalidConfiguration;
        *slots = clusters;
        return cudaSuccess;
    }
}

template <class Cfg>
static KernelInfo tc_info() {
    KernelInfo k;
    k.bm = Cfg::BM * Cfg::CM;  // the tile a cluster computes
    k.bn = Cfg::BN;
    k.bk = Cfg::SBK;  // K columns per stage
    k.stages = Cfg::STAGES;
    k.threads = Cfg::THREADS;
    k.smem_bytes = Cfg::SMEM_BYTES;
    k.a_box_x = Cfg::BK;
    k.a_box_y = Cfg::BM;
    k.b_box_x = 64;
    k.b_box_y = Cfg::BK;
    // fp16 / bf16 boxes of 64 elements (128 bytes) land 128-byte swizzled;
    // the staged producer's int8 boxes (64 bytes wide) land as plain rows
    k.a_swizzle128 = k.b_swizzle128 = Cfg::PROD != 2;
    k.c_tma = true;
    k.kc = Cfg::KC;
    k.slabs_per_tile = Cfg::CM * Cfg::EPI;
    k.producer = Cfg::PROD == 1   ? PGEMM_PRODUCER_REGISTERS
                 : Cfg::PROD == 2 ? PGEMM_PRODUCER_STAGED
                 : Cfg::PROD == 3 ? PGEMM_PRODUCER_WIDEN_IN_KERNEL
                                  : PGEMM_PRODUCER_TMA;
    k.schedule_slots = tc_slots<Cfg>;
    k.halves = Cfg::HALVES;
    k.func = reinterpret_cast<const void *>(tc_gemm_kernel<Cfg>);
    return k;
}

}  // namespace pg
