/*
 * pgemm -- software-pipelined dense GEMM for one GB300 GPU (sm_103a).
 *
 * Every gemm_* call computes
 *
 *     C <- alpha * A * B + beta * C
 *
 * with row-major operands: A is M x K (leading dimension K), B is K x N
 * (leading dimension N), C is M x N (leading dimension N).  This is the
 * argument list, the operand walk and the alpha/beta output update of the
 * double-buffered SGEMM in "Double Buffering: Software Pipelining the K-Loop"
 * (section "The Kernel"), extended with a CUDA stream.  Its K-loop is
 * software-pipelined over an S-stage shared-memory ring with a prologue, a
 * circular steady state and a drain ("Software pipelines and asynchronous
 * copies", sections "Prologue, steady state, and epilogue" and
 * "Producer-consumer synchronization"): TMA bulk-tensor copies fill a stage
 * and complete on its "full" mbarrier (readiness edge); the consumers release
 * it through its "empty" mbarrier (reuse edge).
 *
 * Common rules for all gemm_* entry points:
 *   - A, B and C are DEVICE pointers owned by the caller; the library keeps no
 *     reference after the call returns.  C is read (when beta != 0) and
 *     written in place.  A and C, or B and C, must not overlap.
 *   - The call is asynchronous on `stream` (NULL = the legacy default
 *     stream): it enqueues work and returns; the caller synchronises.  The
 *     library may enqueue a small repack kernel and stream-ordered scratch
 *     on the same stream when a leading dimension is not a multiple of 16
 *     bytes (int8: its widened operands), and stream-ordered scratch for
 *     partial sums when tiles are split along K (see
 *     pgemm_config.max_k_parts), whose counters a cudaMemsetAsync zeroes
 *     (int8: its widening kernel does).  Scratch comes from a memory pool
 *     the library owns per device (cudaMallocFromPoolAsync /
 *     cudaFreeAsync) that keeps the memory it has mapped, so that calls
 *     with synchronisations between them do not map it again;
 *     pgemm_trim_scratch() gives it back.
 *   - M, N, K >= 0.  M == 0 or N == 0: nothing is done.  K == 0: C <- beta*C
 *     (C is not read when beta == 0, so a NaN in C does not survive).
 *   - beta == 0: C is not read (BLAS convention).
 *   - Errors are returned synchronously: PGEMM_ERR_INVALID_VALUE (negative
 *     dimension, NULL pointer with a non-empty operand, bad config),
 *     PGEMM_ERR_MISALIGNED (a base pointer not 16-byte aligned),
 *     PGEMM_ERR_UNSUPPORTED_DEVICE (the current device is not sm_103),
 *     PGEMM_ERR_CUDA (a launch or runtime failure; the CUDA error is also
 *     left for cudaGetLastError).  A device-side wait that ran past its time
 *     limit is not visible here; pgemm_get_device_status() reports it.
 *   - Thread safety: calls may come from several host threads; the first
 *     call on a device does a one-time set-up.
 */
#ifndef PGEMM_H
#define PGEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define PGEMM_API __attribute__((visibility("default")))
#else
#define PGEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* The same type as cudaStream_t (a pointer to the runtime's stream object). */
typedef struct CUstream_st *pgemm_stream_t;

typedef enum {
    PGEMM_OK = 0,
    PGEMM_ERR_INVALID_VALUE = 1,
    PGEMM_ERR_MISALIGNED = 2,
    PGEMM_ERR_UNSUPPORTED_DEVICE = 3,
    PGEMM_ERR_CUDA = 4,
    PGEMM_ERR_TIMEOUT = 5,
    PGEMM_ERR_UNSUPPORTED_CONFIG = 6,
    PGEMM_ERR_TOO_LARGE = 7
} pgemm_status;

/* Data types, for the introspection calls. */
typedef enum { PGEMM_F32 = 0, PGEMM_BF16 = 1, PGEMM_I8 = 2 } pgemm_dtype;

/* Who fills the shared-memory stages (pgemm_config.producer).
 *   PGEMM_PRODUCER_TMA: TMA bulk-tensor copies into an S-stage ring guarded by
 *     full / empty mbarriers, issued by one producer thread (every dtype; the
 *     default).
 *   PGEMM_PRODUCER_REGISTERS: the comparator of "GPU-Kernel pipelinen"
 *     (step 3, the LDG-register variant) and of the double-buffered SGEMM of
 *     "Double Buffering: Software Pipelining the K-Loop" (section "The
 *     Kernel"), threads loading the next K-tile into registers:
 *     - fp32 (128 x 128 and 128 x 64, stages = 2): every thread of the block
 *       loads its share of K-tile t+1 while the block computes tile t from
 *       one of two shared-memory buffers, then stores the registers into the
 *       other buffer, and one block barrier per K-tile hands the buffers
 *       over.  Same tile, register tile and arithmetic as the TMA kernel;
 *       only the producer differs.
 *     - int8 (CTA pair 256 x 256, stages 4..6): four producer warps per CTA
 *       load the int8 tiles, widen them exactly to fp16 in registers and
 *       store them into the S-stage ring the tensor core reads, so no
 *       widening pass runs; the MMA issuer and the exact-round epilogue are
 *       the default kernel's.
 *   PGEMM_PRODUCER_STAGED (int8, CTA pair 256 x 256): TMA copies the int8
 *     tiles as they are into a ring of `stages` int8 stages (16 KB each per
 *     CTA, half an fp16 stage), and four warps per CTA widen each landed
 *     stage exactly to fp16 into a short ring of fp16 stages that the tensor
 *     core reads (shared memory to shared memory).  No widening pass runs and
 *     the operands cross L2 as int8; the MMA issuer and the exact-round
 *     epilogue are the default kernel's.
 *   PGEMM_PRODUCER_WIDEN_IN_KERNEL (int8, CTA pair 256 x 256): the TMA ring of
 *     PGEMM_PRODUCER_TMA, but the int8 -> fp16 widening of A and B runs inside
 *     the GEMM instead of as a pass before it: four warps per CTA widen the
 *     operands into the fp16 scratch one 64-wide K chunk after another, and
 *     the TMA producer loads from a chunk once every CTA has published its
 *     share of it, so the widening overlaps the main loop of the first tiles.
 *     Needs K and N multiples of 16 (int8 rows 16-byte aligned); launched
 *     cooperatively (every CTA resident). */
typedef enum {
    PGEMM_PRODUCER_TMA = 0,
    PGEMM_PRODUCER_REGISTERS = 1,
    PGEMM_PRODUCER_STAGED = 2,
    PGEMM_PRODUCER_WIDEN_IN_KERNEL = 3
} pgemm_producer;

/* Which multiply-accumulate consumes the stages (pgemm_config.engine).
 *   PGEMM_ENGINE_DEFAULT: FFMA register tiles (fp32), tcgen05.mma into
 *     tensor memory (bf16; int8 as exact fp16 products).
 *   PGEMM_ENGINE_MMA_SYNC (int8 only): the alternative exact int8 route,
 *     warp-level mma.sync.m16n8k32 s8 x s8 -> s32 on the int8 operands
 *     themselves, 128 x 128 tiles, K-tiles of 128, on the same TMA ring (a
 *     pre-pass writes B transposed, K-major, as the MMA's column operand
 *     wants it).  Same results as the default, bit for bit. */
typedef enum { PGEMM_ENGINE_DEFAULT = 0, PGEMM_ENGINE_MMA_SYNC = 1 } pgemm_engine;

/* A kernel configuration: output tile bm x bn, K-tile bk (elements), and the
 * number of pipeline stages (shared-memory ring slots).  Stage count trades
 * latency coverage against shared memory and resident blocks ("Software
 * pipelines and asynchronous copies", section "Selecting the number of
 * stages").  Zero fields mean "library default for this shape"; bk = 0 with
 * the other fields set means "whichever built K-tile matches".  The CTA pair
 * (bm = bn = 256) is built with 64-column stages (S = 4..6) and with 128-column
 * stages (bk = 128, S = 2 or 3: two 64-column sub-tiles landed under one
 * barrier, the default for bf16 and int8 pairs).
 *
 * max_k_parts (the pages have no counterpart): stream-K against wave
 * quantisation (pgemm_stream_k_plan).  The tiles a partial last wave would
 * hold have their K-iterations dealt out to every resident CTA (or CTA pair);
 * the persistent tensor-core kernels run a slot's pieces before its whole
 * tiles, fp32 runs them as a second grid behind the whole tiles.  The last
 * piece of a tile to finish adds the others' partial sums (fp32 sums in slot
 * order, so the result does not depend on timing; int8: exact int32) before
 * the alpha/beta update.  max_k_parts = 0: the library's choice (at most 2
 * pieces a tile for the tensor-core kernels, whose exchange is slower than
 * the fp32 kernels'; none for fp32); 1: off; n > 1: at most n pieces a tile. */
/* group_m (the pages have no counterpart): the order in which output tiles
 * are handed out.  Tiles go down group_m tile rows (tile pairs for a CTA
 * pair), then one tile column to the right, and so on across C, then the
 * next group of rows: the CTAs running at once share A row panels and B
 * column panels through L2, and group_m sets the shape of that working set.
 * 0: the library's choice (fp32: 8; bf16 and int8: 16 for K <= 4096, else
 * 8). */
typedef struct {
    int bm, bn, bk, stages;
    int max_k_parts;
    int producer; /* a pgemm_producer */
    int engine;   /* a pgemm_engine */
    int group_m;  /* raster group of the tile order (0: the library's choice) */
} pgemm_config;

/* fp32: FFMA register-tiled consumers on the pipelined ring.  Semantics are
 * plain fp32 multiply-add (no TF32).  Alignment: A, B, C 16-byte aligned.
 * Any M, N, K (tails and unaligned leading dimensions are handled). */
PGEMM_API pgemm_status gemm_f32(int M, int N, int K, float alpha, const float *A, const float *B,
                      float beta, float *C, pgemm_stream_t stream);

/* bf16: A and B hold bf16 bit patterns (uint16); products are accumulated in
 * fp32 in tensor memory (tcgen05.mma kind::f16) and C is fp32.  alpha and
 * beta are fp32. */
PGEMM_API pgemm_status gemm_bf16(int M, int N, int K, float alpha, const uint16_t *A, const uint16_t *B,
                       float beta, float *C, pgemm_stream_t stream);

/* int8: A, B int8; the exact integer dot products are accumulated modulo 2^32
 * into int32; C <- alpha*acc + beta*C in int32 arithmetic modulo 2^32 (two's
 * complement wrap-around).  The products run on the tensor cores as fp16
 * values (exact for |v| <= 128) with exact fp32 partial sums over K chunks of
 * at most 1024, folded into int32. */
PGEMM_API pgemm_status gemm_i8(int M, int N, int K, int32_t alpha, const int8_t *A, const int8_t *B,
                     int32_t beta, int32_t *C, pgemm_stream_t stream);

/* Size of the fixed device scratch array that gemm_i8_noalloc uses. */
#define PGEMM_NOALLOC_SCRATCH_BYTES (32u << 20)

/* gemm_i8 for callers that must not have the library allocate device memory.
 * The pages have no counterpart: this is a deployment variant of gemm_i8.
 *
 * Some callers cannot allocate: a program that has handed all of the GPU's
 * memory to its own allocator or runs under a fixed memory budget, or code on
 * a path where an allocation call is not allowed or could block (cudaFree can
 * synchronise the whole device).  gemm_i8 widens A and B to fp16 in
 * stream-ordered scratch it allocates per call; this entry point instead
 * widens them into one file-scope device array of PGEMM_NOALLOC_SCRATCH_BYTES
 * (32 MiB), which every GPU that loads the library holds until the process
 * exits.  It calls no cudaMalloc, cudaMallocAsync or cudaFree.
 *
 * Same arguments, semantics and results as gemm_i8 (bit-identical).  Limit:
 * 2 * (M * round_up(K, 8) + K * round_up(N, 8)) bytes, each operand rounded
 * up to 256 bytes, must fit in the array; larger problems return
 * PGEMM_ERR_TOO_LARGE without doing anything.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  All calls share the one array and it keeps the
 * last call's contents (no byte of it needs to start at zero: every byte a
 * call reads it has written first), so calls whose work overlaps on the GPU
 * (different streams without ordering between them) race and give wrong
 * results: order them on one stream, or with events. */
PGEMM_API pgemm_status gemm_i8_noalloc(int M, int N, int K, int32_t alpha, const int8_t *A,
                                       const int8_t *B, int32_t beta, int32_t *C,
                                       pgemm_stream_t stream);

/* The same three operations with an explicit configuration (cfg may be NULL
 * for the default).  Returns PGEMM_ERR_UNSUPPORTED_CONFIG for a configuration
 * the library was not built with (pgemm_list_configs enumerates them). */
PGEMM_API pgemm_status gemm_f32_ex(int M, int N, int K, float alpha, const float *A, const float *B,
                         float beta, float *C, const pgemm_config *cfg, pgemm_stream_t stream);
PGEMM_API pgemm_status gemm_bf16_ex(int M, int N, int K, float alpha, const uint16_t *A,
                          const uint16_t *B, float beta, float *C, const pgemm_config *cfg,
                          pgemm_stream_t stream);
PGEMM_API pgemm_status gemm_i8_ex(int M, int N, int K, int32_t alpha, const int8_t *A, const int8_t *B,
                        int32_t beta, int32_t *C, const pgemm_config *cfg, pgemm_stream_t stream);

/* The configuration the library picks for a shape (the per-shape table). */
PGEMM_API pgemm_status pgemm_default_config(pgemm_dtype dtype, int M, int N, int K, pgemm_config *out);

/* Up to `cap` built configurations of a dtype written to `out`; returns how
 * many exist (call with cap = 0 to count). */
PGEMM_API int pgemm_list_configs(pgemm_dtype dtype, pgemm_config *out, int cap);

/* Resource figures of one configuration's kernel on the current device:
 * dynamic shared memory per block (bytes), registers per thread, threads per
 * block and resident blocks per SM.  Any output pointer may be NULL. */
PGEMM_API pgemm_status pgemm_kernel_attrs(pgemm_dtype dtype, const pgemm_config *cfg, int *smem_bytes,
                                int *regs_per_thread, int *threads_per_block,
                                int *blocks_per_sm);

/* The schedule a call with these arguments would use on the current device
 * (cfg NULL = default configuration): output tiles (a CTA pair's 256-row tile
 * counts once), schedule slots (units that run at once), tiles split along K
 * and their parts (0 and 1 when nothing is split; for fp32, the stream-K
 * tiles and the most pieces one of them is spread over), and tiles run as two
 * half-width units each (the 256-wide tensor-core tiles of a partial last
 * wave, cut along N when they fit twice on the slots; then nothing is split
 * along K).  No GPU work is enqueued.  Any output pointer may be NULL. */
PGEMM_API pgemm_status pgemm_schedule(pgemm_dtype dtype, const pgemm_config *cfg, int M, int N,
                                      int K, long long *tiles, int *slots,
                                      long long *split_tiles, int *parts,
                                      long long *half_tiles);

/* The stream-K rule, a pure host computation (no device needed; the pages
 * have no counterpart).  `tiles` output tiles on `slots` schedule slots
 * (resident blocks, or CTA pairs) with K of `k_tiles` K-tiles: the
 * R = tiles % slots tiles of the partial last wave have their R * k_tiles
 * K-iterations laid end to end and dealt out to Gs slots, slot j taking
 * [j * R * k_tiles / Gs, (j + 1) * R * k_tiles / Gs) -- pieces of at most
 * two tiles -- and every slot then takes whole tiles R + j, R + j + slots, ...
 * Gs = slots, unless max_parts = n > 1 and some tile would be spread over
 * more than n slots: then Gs = R * p with p = min(n, slots / R), and every
 * tile is exactly p pieces.  Used only when every slot gets at least 8
 * K-iterations and the longest share is at most 7/8 of k_tiles; max_parts = 1
 * turns it off.  The pieces of a tile each leave their partial sums; one adds
 * them in slot order (so results do not depend on timing) and writes C.
 * Outputs: R (0 when unused), Gs, the most slots one tile is spread over (1
 * when unused) and the K-iterations per slot.  The library calls it with
 * pgemm_config.max_k_parts, or with 2 (tensor-core kernels) and 0 (fp32) when
 * that is 0. */
PGEMM_API pgemm_status pgemm_stream_k_plan(long long tiles, int slots, int k_tiles, int max_parts,
                                           long long *sk_tiles, int *sk_slots, int *max_pieces,
                                           long long *share);

/* The stage-reuse hazard experiment of "Software pipelines and asynchronous
 * copies" (section "Practice"): a two-stage copy-and-reduce over the rows of
 * X (rows x cols fp32, row-major, cols a multiple of 4, at most 8192).  One
 * producer thread per block copies row perm[r] into stage (t % 2) with a bulk
 * copy; four consumer warps each sum a quarter of the stage and atomically add
 * it to out[r] (the caller zeroes out; rows r = block, block + grid, ...).
 * check_reuse != 0: the producer waits until every consumer warp has finished
 * the tile that last used a stage before overwriting it (the consume-before-
 * reuse edge).  check_reuse == 0: that one wait is skipped.  delay_warp (0..3,
 * or -1 for none) sleeps delay_ns before reading each tile.  trace (device,
 * may be NULL): trace[0] counts events of block 0, then up to trace_cap pairs
 * {globaltimer ns, event << 56 | stage << 48 | warp << 40 | tile}; events 1
 * load issued, 2 load landed, 3 reuse wait begins, 4 reuse allowed, 5 read
 * begins, 6 read ends.  All pointers are device pointers; asynchronous on
 * `stream`; every wait is bounded (see pgemm_get_device_status). */
PGEMM_API pgemm_status pgemm_stage_reuse_demo(const float *X, int rows, int cols, const int *perm,
                                              float *out, int check_reuse, int delay_warp,
                                              unsigned delay_ns, unsigned long long *trace,
                                              int trace_cap, pgemm_stream_t stream);

/* Synchronises `stream`, then reads and clears the library's device status
 * word of the current device: PGEMM_OK, or PGEMM_ERR_TIMEOUT if a kernel's
 * bounded mbarrier wait ran out (the kernel then skipped the rest of its work
 * and returned; its output is undefined).  PGEMM_ERR_CUDA on a CUDA error. */
PGEMM_API pgemm_status pgemm_get_device_status(pgemm_stream_t stream);

/* A self-test of the bounded-wait path: launches one block that waits, with a
 * time limit of `limit_us` microseconds, on an mbarrier that nothing will
 * ever arrive on, and returns what pgemm_get_device_status then reports
 * (PGEMM_ERR_TIMEOUT when the wait path works).  The kernel never hangs and
 * never faults; the context stays usable. */
PGEMM_API pgemm_status pgemm_selftest_wait_timeout(int limit_us, pgemm_stream_t stream);

/* A static description of a status code. */
PGEMM_API const char *pgemm_status_string(pgemm_status status);

/* Synchronises the current device, then returns all unused memory of the
 * library's scratch pool on it to the system (the pool keeps what it has
 * mapped between calls otherwise).  PGEMM_ERR_CUDA on a CUDA error. */
PGEMM_API pgemm_status pgemm_trim_scratch(void);

/* Library version, major * 10000 + minor * 100 + patch. */
PGEMM_API int pgemm_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PGEMM_H */
