// Host dispatch for the pipelined GEMMs: argument validation, the per-shape
// (tile, stages) table, operand repacking for leading dimensions that TMA
// cannot describe, tensor-map encoding and the launch on the caller's stream.
//
// The entry points follow the kernel signature (M, N, K, alpha, A, B, beta, C)
// of "Double Buffering: Software Pipelining the K-Loop" (section "The
// Kernel") plus a stream; the stage-count choice follows "Software pipelines
// and asynchronous copies" (section "Selecting the number of stages"): a
// deeper ring hides more latency but costs shared memory and resident blocks,
// so the default table is per shape and every built configuration can be
// selected explicitly for a sweep.
#include <cuda.h>
#include <cuda_runtime.h>

#include <functional>
#include <mutex>
#include <unordered_map>

#include "pgemm.h"
#include "common.cuh"
#include "kernels.h"

namespace pg {

// The device status word of each device (one instance per device context).
__device__ uint32_t g_status_word = 0;

constexpr uint64_t kDefaultWaitLimitNs = 2000000000ull;  // 2 s per mbarrier wait

constexpr int kMaxDevices = 64;

struct KernelState {
    bool ready = false;
    int blocks_per_sm = 0;
    int slots = 0;  // schedule slots of a persistent launch (0: not persistent)
};

struct DeviceState {
    bool init = false;
    pgemm_status init_status = PGEMM_OK;
    int sm_count = 0;
    uint32_t *status = nullptr;
    // Stream-ordered scratch comes from this pool, which keeps what it has
    // mapped when streams synchronise (the default pool's release threshold
    // of zero would hand it back at every synchronisation, and the next call
    // would map it again: ~60 us for 29 MB of stream-K partial sums).
    cudaMemPool_t pool = nullptr;
    std::unordered_map<const void *, KernelState> kernels;
};

// Guards the one-time set-up of a device and of each kernel on it (and the
// table of kernels already set up).  Everything after that set-up -- the
// choice of configuration, scratch allocation, tensor-map encoding and the
// launches -- runs without it, so host threads calling on their own streams
// enqueue concurrently.
static std::mutex g_mu;
static DeviceState g_dev[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
static EncodeTiledFn g_encode = nullptr;

// One-time set-up of the current device (under g_mu).
static pgemm_status device_setup(int *dev_out, DeviceState **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PGEMM_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PGEMM_ERR_UNSUPPORTED_DEVICE;
    // Make the device's primary context current in this host thread: the
    // tensor-map encoder is a driver call and needs one, and a thread whose
    // first CUDA work is this call (a worker thread of the caller) may not
    // have one yet.
    if (cudaSetDevice(dev) != cudaSuccess) return PGEMM_ERR_CUDA;
    DeviceState &d = g_dev[dev];
    if (!d.init) {
        d.init = true;
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            d.init_status = PGEMM_ERR_CUDA;
        } else if (major != 10 || minor != 3) {
            // the library carries sm_103a code only
            d.init_status = PGEMM_ERR_UNSUPPORTED_DEVICE;
        } else if (cudaGetSymbolAddress(reinterpret_cast<void **>(&d.status), g_status_word) !=
                   cudaSuccess) {
            d.init_status = PGEMM_ERR_CUDA;
        } else if (!g_encode) {
            cudaDriverEntryPointQueryResult q{};
            void *fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                d.init_status = PGEMM_ERR_CUDA;
            else
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        if (d.init_status == PGEMM_OK) {
            cudaMemPoolProps props{};
            props.allocType = cudaMemAllocationTypePinned;
            props.handleTypes = cudaMemHandleTypeNone;
            props.location.type = cudaMemLocationTypeDevice;
            props.location.id = dev;
            cuuint64_t keep = ~cuuint64_t(0);
            if (cudaMemPoolCreate(&d.pool, &props) != cudaSuccess ||
                cudaMemPoolSetAttribute(d.pool, cudaMemPoolAttrReleaseThreshold, &keep) !=
                    cudaSuccess)
                d.init_status = PGEMM_ERR_CUDA;
        }
    }
    *dev_out = dev;
    *out = &d;
    return d.init_status;
}

// One-time set-up of a kernel on a device (under g_mu): shared-memory
// attributes, resident blocks per SM and, for the persistent kernels, the
// number of schedule slots of a launch.
static pgemm_status kernel_setup(DeviceState &d, const KernelInfo &k, int *blocks_per_sm,
                                 int *slots = nullptr) {
    KernelState &ks = d.kernels[k.func];
    if (!ks.ready) {
        if (cudaFuncSetAttribute(k.func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 k.smem_bytes) != cudaSuccess)
            return PGEMM_ERR_CUDA;
        // all of the unified L1/shared storage as shared memory, so that the
        // occupancy the shared-memory request was sized for is reachable
        if (cudaFuncSetAttribute(k.func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 cudaSharedmemCarveoutMaxShared) != cudaSuccess)
            return PGEMM_ERR_CUDA;
        if (k.aux_func != nullptr &&
            (cudaFuncSetAttribute(k.aux_func, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  k.smem_bytes) != cudaSuccess ||
             cudaFuncSetAttribute(k.aux_func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  cudaSharedmemCarveoutMaxShared) != cudaSuccess))
            return PGEMM_ERR_CUDA;
        int n = 0;
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k.func, k.threads, k.smem_bytes) !=
            cudaSuccess)
            return PGEMM_ERR_CUDA;
        if (n < 1) return PGEMM_ERR_UNSUPPORTED_CONFIG;
        if (k.schedule_slots != nullptr) {
            LaunchCommon q{};
            q.sm_count = d.sm_count;
            q.blocks_per_sm = n;
            if (k.schedule_slots(q, &ks.slots) != cudaSuccess) return PGEMM_ERR_CUDA;
        }
        ks.blocks_per_sm = n;
        ks.ready = true;
    }
    *blocks_per_sm = ks.blocks_per_sm;
    if (slots) *slots = ks.slots;
    return PGEMM_OK;
}

static const KernelInfo *table_of(pgemm_dtype dt, int *count) {
    switch (dt) {
        case PGEMM_F32: return f32_kernels(count);
        case PGEMM_BF16: return bf16_kernels(count);
        case PGEMM_I8: return i8_kernels(count);
    }
    *count = 0;
    return nullptr;
}

// The per-shape default (tile, stages) table, read off the stage sweep:
//  * fp32: 128 x 128 tiles with three stages (two blocks per SM; four or more
//    stages drop to one block per SM and lose 16 %); 128 x 64 tiles when the
//    128 x 128 grid would leave SMs without two blocks each.
//  * bf16 and int8, short K (bf16 K <= 384, int8 K <= 512) when 128 x 256
//    tiles fill at least three waves: 128 x 256 tiles, three stages up to
//    K = 128, else four.  There the call is bound by writing C and by each
//    tile's fixed hand-offs (load, MMA, accumulator, epilogue), and the wider
//    tile halves the hand-offs for the same C bytes per SM (4096^2, mean of
//    200 calls: bf16 K = 32 16.4 against 18.4 us with 128 x 128, K = 64 16.5
//    against 16.8, K = 192 18.7 against 22.5 with the pair, K = 256 20.6
//    against 22.6, K = 384 level; int8 K = 32 27.6 against 32.8, K = 256
//    29.7 against 33.7, K = 512 32.8 against 35.9).  With fewer waves the
//    last wave's larger stores cost more than that (bf16 2048 x 4096 x 32:
//    12.4 against 12.9 us for 128 x 128).
//  * otherwise 256 x 256 tiles on a CTA pair (cta_group::2) when the
//    pairs cover half the SMs (bf16 8192^3 +12 %, int8 4096^3 +10 % over
//    128 x 256), with three stages of 128 K columns, each landed as two
//    64-column sub-tiles under one barrier: the MMA warp then waits, commits
//    and loops once per 8 MMAs instead of 4 (against six 64-column stages in
//    the same shared memory: bf16 4096^2 x 512 -8 %, x 2048 -4 %, 8192^3
//    -1 %, int8 4096^3 -1 %); else 128 x 128 with four stages.
static pgemm_config default_config(pgemm_dtype dt, int M, int N, int K, int sm_count) {
    pgemm_config c{128, 128, 0, 4};
    if (dt == PGEMM_F32) {
        const long long tiles128 = (long long)((M + 127) / 128) * ((N + 127) / 128);
        c.bn = tiles128 >= 2LL * sm_count ? 128 : 64;
        c.stages = 3;
        return c;
    }
    const long long wide_tiles = (long long)((M + 127) / 128) * ((N + 255) / 256);
    const int wide_max_k = dt == PGEMM_I8 ? 512 : 384;
    if (K <= wide_max_k && wide_tiles >= 3LL * sm_count) {
        c.bn = 256;
        c.stages = K <= 128 ? 3 : 4;
        return c;
    }
    const long long pairs = (long long)((M + 255) / 256) * ((N + 255) / 256);
    if (K <= 128) return c;  // 128 x 128, four stages
    if (pairs >= sm_count / 2) {
        c.bm = 256;
        c.bn = 256;
        c.bk = 128;
        c.stages = 3;
    }
    return c;
}

// Stream-K against wave quantisation.  A persistent grid of G slots runs
// `tiles` output tiles in ceil(tiles / G) waves; the R = tiles % G tiles of
// the partial last wave instead have their R * T K-iterations dealt out in
// equal contiguous ranges to Gs slots (pgemm_stream_k_plan), so that the
// extra wave costs about R / Gs of a tile.  The persistent tensor-core
// kernels run these pieces first, each slot's pieces before its whole tiles,
// so that the exchange of partial sums overlaps whole-tile work; the fp32
// kernels run them as a second grid behind the whole tiles.  The tensor-core
// kernels cap a tile at kTcMaxPieces pieces by default (equal halves, on
// R * 2 slots): their last piece waits for the others' partial sums and adds
// them in an epilogue warp, one 16 KB slab at a time, and with more pieces
// that exchange costs more than the shorter shares save (int8 4096^3: 132.5
// us with up to four pieces, 107.8 with halves, 110.5 without; bf16
// 2048^2 x 8192, where every slot would share: 65.0 against 57.3 without).
constexpr int kTcMaxPieces = 2;

// Half-width units instead (kernels with 256-wide tiles fed by TMA, the
// library's default up to kHalvesMaxK K columns): when the R leftover
// tiles fit twice on the slots, each is cut along N into its left and right
// 128 columns, 2R units of the full K range that exchange nothing (no
// partial-sum memory, no counters), so the wave after them is never held up
// by an exchange.  The limit is in K columns (kHalvesMaxK), whatever the
// kernel's K-tile width.  A half-width unit's N = 128 MMAs read A in full for half
// the products, so per K-tile it costs more than half a whole tile; with
// long K that outweighs the exchange it saves (bf16 4096^2: K = 512 24.6
// against 26.6 us without a split, K = 2048 53.2 against 55.9 us with K
// halves; K = 16384 328.7 against 311.8 us, and int8 4096^3 108.8 against
// 106.2 us).  An explicit max_k_parts > 1 asks for stream-K pieces.
// allow_k_split = false: a call that may not allocate (no exchange memory).
constexpr int kHalvesMaxK = 2048;
static TileSchedule plan_schedule(const KernelInfo &k, int M, int N, int K, int slots,
                                  int max_parts, bool allow_k_split = true) {
    TileSchedule s;
    s.tiles = static_cast<long long>((M + k.bm - 1) / k.bm) * ((N + k.bn - 1) / k.bn);
    s.slots = slots;
    if (k.schedule_slots == nullptr) return s;
    const int T = (K + k.bk - 1) / k.bk;
    if (k.halves && max_parts == 0 && K > 0 && K <= kHalvesMaxK) {
        const long long rem = s.tiles % slots;
        if (rem > 0 && 2 * rem <= slots) {
            s.half_tiles = rem;
            return s;
        }
    }
    if (!allow_k_split) return s;
    const int cap = max_parts > 0 ? max_parts : (k.stream_k ? 0 : kTcMaxPieces);
    long long share = 0;
    if (pgemm_stream_k_plan(s.tiles, slots, T, cap, &s.split_tiles, &s.sk_slots, &s.parts,
                            &share) != PGEMM_OK)
        return s;
    if (s.split_tiles > 0) {
        // a slab of partial sums for each of a slot's (at most two) pieces
        s.partial_words = 2LL * s.sk_slots * k.bm * k.bn;
        s.counter_words = k.stream_k ? s.split_tiles : s.split_tiles * k.slabs_per_tile * 2;
    }
    return s;
}

static const KernelInfo *find_kernel(pgemm_dtype dt, const pgemm_config &c) {
    int n = 0;
    const KernelInfo *t = table_of(dt, &n);
    for (int i = 0; i < n; ++i)
        if (t[i].bm == c.bm && t[i].bn == c.bn && t[i].stages == c.stages &&
            (c.bk == 0 || c.bk == t[i].bk) && t[i].producer == c.producer &&
            t[i].engine == c.engine)
            return &t[i];
    return nullptr;
}

static bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static pgemm_status encode_2d(CUtensorMap *map, CUtensorMapDataType type, int elem_bytes,
                              const void *base, long long inner, long long outer, long long ld,
                              int box_x, int box_y, bool swizzle128) {
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * elem_bytes};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_x), static_cast<cuuint32_t>(box_y)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(map, type, 2, const_cast<void *>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE,
                          swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PGEMM_OK : PGEMM_ERR_CUDA;
}

// Copies rows [0, rows) x [0, cols) of a row-major matrix with pitch `sld` to a
// new pitch `dld` (both in elements of `eb` bytes, 2 or 4; the destination rows
// start on 16-byte boundaries).  One block walks a row at a time; every
// 16-byte destination chunk is assembled from the one or two aligned 16-byte
// source chunks that cover it (a byte shift by the row's misalignment, which
// is even), so every store is a full 16-byte vector.  A chunk whose source
// window would reach past the end of the source matrix is copied in 2-byte
// units instead, as is the row's tail shorter than 16 bytes.
__device__ __forceinline__ uint4 shift_bytes(uint4 lo, uint4 hi, uint32_t off) {
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
    const uint32_t q = off >> 2, sh = (off & 3u) * 8u;  // sh is 0 or 16: offsets are even
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t a = w[(q + i) & 7], b = w[(q + i + 1) & 7];
        o[i] = sh ? __funnelshift_r(a, b, sh) : a;
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}

struct RepackJob {
    const uint8_t *src;
    long long sld;
    uint8_t *dst;
    long long dld;
    int rows, cols;
};

// blockIdx.y selects the operand: both repacks of a call in one launch.
__global__ void repack_rows_kernel(RepackJob j0, RepackJob j1, int eb) {
    const RepackJob &j = blockIdx.y == 0 ? j0 : j1;
    const uint8_t *__restrict__ src = j.src;
    uint8_t *__restrict__ dst = j.dst;
    const long long sld = j.sld, dld = j.dld;
    const int rows = j.rows, cols = j.cols;
    const long long row_bytes = static_cast<long long>(cols) * eb;
    const uint8_t *src_end = src + (static_cast<long long>(rows - 1) * sld + cols) * eb;
    for (int r = blockIdx.x; r < rows; r += gridDim.x) {
        const uint8_t *s = src + static_cast<long long>(r) * sld * eb;
        uint8_t *d = dst + static_cast<long long>(r) * dld * eb;
        const uint32_t off = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(s) & 15u);
        const uint4 *sa = reinterpret_cast<const uint4 *>(s - off);  // aligned down
        const long long nchunks = row_bytes / 16;
        for (long long j = threadIdx.x; j < nchunks; j += blockDim.x) {
            const uint8_t *win_end = reinterpret_cast<const uint8_t *>(sa + j) + (off ? 32 : 16);
            if (win_end <= src_end) {
                const uint4 lo = sa[j];
                reinterpret_cast<uint4 *>(d)[j] = off ? shift_bytes(lo, sa[j + 1], off) : lo;
            } else {
#pragma unroll
                for (int b = 0; b < 16; b += 2)
                    *reinterpret_cast<uint16_t *>(d + 16 * j + b) =
                        *reinterpret_cast<const uint16_t *>(s + 16 * j + b);
            }
        }
        for (long long b = nchunks * 16 + 2 * threadIdx.x; b < row_bytes; b += 2 * blockDim.x)
            *reinterpret_cast<uint16_t *>(d + b) = *reinterpret_cast<const uint16_t *>(s + b);
    }
    grid_launch_dependents();  // this block's rows are written
}

// Repack one or two operands (rows = 0: none) in a single launch.
static cudaError_t launch_repack(const void *src0, long long sld0, void *dst0, long long dld0,
                                 int rows0, int cols0, const void *src1, long long sld1,
                                 void *dst1, long long dld1, int rows1, int cols1, int eb,
                                 int sm_count, cudaStream_t s) {
    if (cols0 <= 0) rows0 = 0;
    if (cols1 <= 0) rows1 = 0;
    const RepackJob j0{static_cast<const uint8_t *>(src0), sld0, static_cast<uint8_t *>(dst0),
                       dld0, rows0, cols0};
    const RepackJob j1{static_cast<const uint8_t *>(src1), sld1, static_cast<uint8_t *>(dst1),
                       dld1, rows1, cols1};
    // operand 0 only, operand 1 only (as y = 0), or both
    const RepackJob &a = rows0 > 0 ? j0 : j1;
    const int ny = (rows0 > 0 && rows1 > 0) ? 2 : ((rows0 > 0 || rows1 > 0) ? 1 : 0);
    if (ny == 0) return cudaSuccess;
    const int most = rows0 > rows1 ? rows0 : rows1;
    const int blocks = most < sm_count * 8 ? most : sm_count * 8;
    repack_rows_kernel<<<dim3(blocks, ny), 256, 0, s>>>(a, j1, eb);
    return cudaGetLastError();
}

static long long round_up(long long v, long long m) { return (v + m - 1) / m * m; }

// Stream-ordered scratch owned by one call.
struct Scratch {
    void *p = nullptr;
    cudaStream_t s = nullptr;
    ~Scratch() {
        if (p) cudaFreeAsync(p, s);
    }
};

enum class Kind { F32, BF16, I8 };

// fixed_scratch (FixedScratchFn, kernels.h): when given, operand repacking / widening uses the buffer it
// provides instead of stream-ordered allocations, a problem that does not
// fit is rejected with PGEMM_ERR_TOO_LARGE, and no tile is split (the
// stream-K exchange would need memory too).
template <Kind KIND, typename In, typename Sc, typename Out>
static pgemm_status gemm_impl(int M, int N, int K, Sc alpha, const In *A, const In *B, Sc beta,
                              Out *C, const pgemm_config *cfg_in, cudaStream_t stream,
                              FixedScratchFn fixed_scratch = nullptr) {
    if (M < 0 || N < 0 || K < 0) return PGEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return PGEMM_OK;
    if (C == nullptr || (K > 0 && (A == nullptr || B == nullptr))) return PGEMM_ERR_INVALID_VALUE;
    if (!aligned16(C) || (K > 0 && (!aligned16(A) || !aligned16(B)))) return PGEMM_ERR_MISALIGNED;
    if (cfg_in && (cfg_in->max_k_parts < 0 || cfg_in->group_m < 0)) return PGEMM_ERR_INVALID_VALUE;
    constexpr pgemm_dtype DT =
        KIND == Kind::F32 ? PGEMM_F32 : (KIND == Kind::BF16 ? PGEMM_BF16 : PGEMM_I8);

    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_config c{};
    const KernelInfo *k = nullptr;
    int blocks_per_sm = 0, slots = 0;
    {
        // one-time set-up only; the rest of the call runs unlocked
        std::lock_guard<std::mutex> lock(g_mu);
        pgemm_status st = device_setup(&dev, &d);
        if (st != PGEMM_OK) return st;
        c = (cfg_in && cfg_in->stages > 0) ? *cfg_in : default_config(DT, M, N, K, d->sm_count);
        if (c.bm == 0) c.bm = 128;
        if (cfg_in) {
            c.max_k_parts = cfg_in->max_k_parts;
            if (cfg_in->group_m > 0) c.group_m = cfg_in->group_m;
        }
        // a call with fixed scratch widens by the pass: the in-kernel
        // widening's chunk counters would need memory of their own
        if (fixed_scratch != nullptr && c.producer == PGEMM_PRODUCER_WIDEN_IN_KERNEL)
            c.producer = PGEMM_PRODUCER_TMA;
        k = find_kernel(DT, c);
        if (!k) return PGEMM_ERR_UNSUPPORTED_CONFIG;
        st = kernel_setup(*d, *k, &blocks_per_sm, &slots);
        if (st != PGEMM_OK) return st;
    }
    pgemm_status st = PGEMM_OK;

    // The persistent schedule (tensor-core kernels).  A call with a fixed
    // scratch buffer does not split: the exchange area would need memory.
    TileSchedule sched;
    if (k->schedule_slots != nullptr)
        sched = plan_schedule(*k, M, N, K, slots, c.max_k_parts, fixed_scratch == nullptr);

    // Operands as the kernels read them: element type, pitch, base pointer.
    // int8 is widened to fp16 by a pre-pass, except for the mma.sync engine,
    // which reads the int8 values with B transposed (N rows of K), and the
    // register-staged and staged producers, which read them as they are
    // (rows relaid out to 16-byte pitches when K or N is not a multiple of 16).
    const bool imma = KIND == Kind::I8 && k->engine == PGEMM_ENGINE_MMA_SYNC;
    const bool rp = KIND == Kind::I8 && !imma && k->producer == PGEMM_PRODUCER_REGISTERS;
    // the staged producer's TMA copies the int8 operands as they are
    const bool staged = KIND == Kind::I8 && !imma && k->producer == PGEMM_PRODUCER_STAGED;
    const bool raw_i8 = rp || staged;  // the kernel reads int8 (no widening pass)
    // widening inside the GEMM: fp16 scratch as for the pass, no pass
    const bool fused = KIND == Kind::I8 && !imma && k->producer == PGEMM_PRODUCER_WIDEN_IN_KERNEL;
    if (fused && (K % 16 != 0 || N % 16 != 0)) return PGEMM_ERR_UNSUPPORTED_CONFIG;
    const bool widen_pass = KIND == Kind::I8 && !imma && !raw_i8 && !fused && K > 0;
    const long long widen_chunks = fused ? (K + 63) / 64 : 0;  // at most this many K chunks
    uint32_t *chunk_ready = nullptr;
    const int in_bytes = KIND == Kind::F32 ? 4 : ((imma || raw_i8) ? 1 : 2);
    const long long lda = K, ldb = N;
    const void *a_op = A;
    const void *b_op = B;
    long long a_ld = lda, b_ld = ldb;
    Scratch scratch;
    scratch.s = stream;
    Scratch split_area;  // partial sums and counters of stream-K tiles
    split_area.s = stream;
    if (sched.split_tiles > 0 || widen_chunks > 0) {
        // [partial sums][stream-K counters][K-chunk counters of in-kernel widening]
        const long long pbytes = round_up(sched.partial_words * 4, 256);
        const long long cbytes = round_up((sched.counter_words + widen_chunks) * 4, 256);
        if (cudaMallocFromPoolAsync(&split_area.p, pbytes + cbytes, d->pool, stream) != cudaSuccess)
            return PGEMM_ERR_CUDA;
        uint32_t *counters =
            reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(split_area.p) + pbytes);
        if (sched.split_tiles > 0) {
            sched.partials = static_cast<uint32_t *>(split_area.p);
            sched.counters = counters;
        }
        if (widen_chunks > 0) chunk_ready = counters + sched.counter_words;
        // The counters start at zero: the int8 widening pass (which the GEMM
        // waits for) zeroes them; otherwise a memset before any pre-pass does,
        // so that a programmatic launch after the pre-pass still finds them zero.
        if (!widen_pass && cudaMemsetAsync(counters, 0, cbytes, stream) != cudaSuccess)
            return PGEMM_ERR_CUDA;
    }
    std::function<cudaError_t()> prepass;  // repack / widening launch, if any
    if (K > 0) {
        // Rows of a relaid-out 16- or 32-bit operand start on 128-byte
        // boundaries, so that each row of a TMA box is whole cache lines (at
        // a 16-byte-aligned pitch such as 8208 bytes every row of a box
        // straddles two lines: bf16 4096 x 4104 x 4096 took 97.6 us against
        // 90.1 for 4352 columns, the same tiles at a 128-byte pitch).  int8
        // relayouts, and the array of gemm_i8_noalloc, whose capacity is
        // stated for pitches rounded up to 16 bytes, keep 16.
        const long long pitch_bytes = (in_bytes >= 2 && fixed_scratch == nullptr) ? 128 : 16;
        const long long align_elems = pitch_bytes / in_bytes;
        const bool widen = KIND == Kind::I8 && !imma && !raw_i8;
        const bool a_repack = widen || (lda * in_bytes) % 16 != 0;
        const bool b_repack = widen || imma || (ldb * in_bytes) % 16 != 0;
        if (a_repack || b_repack) {
            const long long a_ld2 = a_repack ? round_up(K, align_elems) : lda;
            const long long b_ld2 = imma ? round_up(K, align_elems)
                                         : (b_repack ? round_up(N, align_elems) : ldb);
            const long long b_rows = imma ? N : K;
            const long long a_bytes = a_repack ? round_up(a_ld2 * M * in_bytes, 256) : 0;
            const long long b_bytes = b_repack ? round_up(b_ld2 * b_rows * in_bytes, 256) : 0;
            uint8_t *base = nullptr;
            if (fixed_scratch != nullptr) {
                void *fp = nullptr;
                long long fbytes = 0;
                st = fixed_scratch(&fp, &fbytes);
                if (st != PGEMM_OK) return st;
                if (a_bytes + b_bytes > fbytes) return PGEMM_ERR_TOO_LARGE;
                base = static_cast<uint8_t *>(fp);
            } else {
                if (cudaMallocFromPoolAsync(&scratch.p, a_bytes + b_bytes, d->pool, stream) !=
                    cudaSuccess)
                    return PGEMM_ERR_CUDA;
                base = static_cast<uint8_t *>(scratch.p);
            }
            // The pre-pass is launched below, after every tensor map is encoded,
            // so that the GEMM launch follows it with no host work in between.
            // With the widening inside the GEMM there is none.
            if (!fused) prepass = [=, &d]() -> cudaError_t {
                if (imma || raw_i8) {  // int8 to 16-byte pitches as needed; mma.sync: B -> B^T
                    cudaError_t e = cudaSuccess;
                    if (a_repack)
                        e = launch_i8_relayout(reinterpret_cast<const int8_t *>(A), lda, base,
                                               a_ld2, M, K, false, d->sm_count, stream);
                    if (e == cudaSuccess && b_repack)
                        e = launch_i8_relayout(reinterpret_cast<const int8_t *>(B), ldb,
                                               base + a_bytes, b_ld2, K, N, imma, d->sm_count,
                                               stream);
                    return e;
                }
                if (widen)  // int8 -> fp16 of both operands in one launch
                    return launch_widen_i8_pair(reinterpret_cast<const int8_t *>(A), lda, base,
                                                a_ld2, M, K, reinterpret_cast<const int8_t *>(B),
                                                ldb, base + a_bytes, b_ld2, K, N,
                                                sched.counters,
                                                static_cast<int>(sched.counter_words),
                                                d->sm_count, stream);
                return launch_repack(A, lda, base, a_ld2, a_repack ? M : 0, K, B, ldb,
                                     base + a_bytes, b_ld2, b_repack ? K : 0, N, in_bytes,
                                     d->sm_count, stream);
            };
            if (a_repack) {
                a_op = base;
                a_ld = a_ld2;
            }
            if (b_repack) {
                b_op = base + a_bytes;
                b_ld = b_ld2;
            }
        }
    }

    // Tensor maps.  With K == 0 nothing is ever loaded, nor by the
    // register-staged producer; the maps then describe a 1 x 1 region of C so
    // that they are still valid objects.
    alignas(64) CUtensorMap ta, tb;
    const CUtensorMapDataType tmt = KIND == Kind::F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                    : KIND == Kind::BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : (imma || raw_i8)   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (K > 0 && imma) {
        st = encode_2d(&ta, tmt, 1, a_op, K, M, a_ld, k->a_box_x, k->a_box_y, k->a_swizzle128);
        if (st == PGEMM_OK)  // B^T: N rows of K
            st = encode_2d(&tb, tmt, 1, b_op, K, N, b_ld, k->b_box_x, k->b_box_y, k->b_swizzle128);
    } else if (K > 0 && !rp) {
        st = encode_2d(&ta, tmt, in_bytes, a_op, K, M, a_ld, k->a_box_x, k->a_box_y, k->a_swizzle128);
        if (st == PGEMM_OK)
            st = encode_2d(&tb, tmt, in_bytes, b_op, N, K, b_ld, k->b_box_x, k->b_box_y,
                           k->b_swizzle128);
    } else {
        st = encode_2d(&ta, tmt, in_bytes, C, 1, 1, 16 / in_bytes, k->a_box_x, k->a_box_y,
                       k->a_swizzle128);
        if (st == PGEMM_OK)
            st = encode_2d(&tb, tmt, in_bytes, C, 1, 1, 16 / in_bytes, k->b_box_x, k->b_box_y,
                           k->b_swizzle128);
    }
    if (st != PGEMM_OK) return st;

    // The in-kernel widening reads the caller's int8 operands by TMA.
    alignas(64) CUtensorMap ta8, tb8;
    if (fused && K > 0) {
        st = encode_2d(&ta8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, K, M, lda, 64, 128, false);
        if (st == PGEMM_OK)
            st = encode_2d(&tb8, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, N, K, ldb, 128, 64, false);
        if (st != PGEMM_OK) return st;
    }

    // C as a tensor map (32 x 32 boxes, 128-byte swizzle) when its rows are
    // 16-byte aligned, so that the tensor-core epilogue can store by TMA.
    alignas(64) CUtensorMap tc_map;
    const CUtensorMap *tmap_c = nullptr;
    if (k->c_tma && aligned16(C) && (static_cast<long long>(N) * 4) % 16 == 0) {
        const CUtensorMapDataType ct =
            KIND == Kind::I8 ? CU_TENSOR_MAP_DATA_TYPE_INT32 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
        if (encode_2d(&tc_map, ct, 4, C, N, M, N, 32, 32, true) == PGEMM_OK) tmap_c = &tc_map;
    }

    const bool after_prepass = static_cast<bool>(prepass);
    cudaError_t e = prepass ? prepass() : cudaSuccess;
    if (e != cudaSuccess) return PGEMM_ERR_CUDA;
    KernelCtx ctx{d->status, kDefaultWaitLimitNs};
    if constexpr (KIND == Kind::F32) {
        LaunchF32 p{};
        p.M = M; p.N = N; p.K = K; p.ldc = N; p.group_m = c.group_m;
        p.sm_count = d->sm_count; p.blocks_per_sm = blocks_per_sm;
        p.tmap_a = &ta; p.tmap_b = &tb; p.tmap_c = tmap_c; p.ctx = ctx;
        p.a_ptr = a_op; p.b_ptr = b_op; p.lda = a_ld; p.ldb = b_ld;
        p.after_prepass = after_prepass;
        p.sched = sched;
        p.alpha = alpha; p.beta = beta; p.C = C;
        e = k->launch_f32(p, stream);
    } else if constexpr (KIND == Kind::BF16) {
        LaunchBf16 p{};
        p.M = M; p.N = N; p.K = K; p.ldc = N; p.group_m = c.group_m;
        p.sm_count = d->sm_count; p.blocks_per_sm = blocks_per_sm;
        p.tmap_a = &ta; p.tmap_b = &tb; p.tmap_c = tmap_c; p.ctx = ctx;
        p.a_ptr = a_op; p.b_ptr = b_op; p.lda = a_ld; p.ldb = b_ld;
        p.after_prepass = after_prepass;
        p.sched = sched;
        p.alpha = alpha; p.beta = beta; p.C = C;
        e = k->launch_bf16(p, stream);
    } else {
        LaunchI8 p{};
        p.M = M; p.N = N; p.K = K; p.ldc = N; p.group_m = c.group_m;
        p.sm_count = d->sm_count; p.blocks_per_sm = blocks_per_sm;
        p.tmap_a = &ta; p.tmap_b = &tb; p.tmap_c = tmap_c; p.ctx = ctx;
        p.a_ptr = a_op; p.b_ptr = b_op; p.lda = a_ld; p.ldb = b_ld;
        p.widen_src_a = A; p.widen_src_b = B; p.widen_lda = lda; p.widen_ldb = ldb;
        p.widen_ready = chunk_ready;
        p.tmap_a8 = (fused && K > 0) ? &ta8 : nullptr;
        p.tmap_b8 = (fused && K > 0) ? &tb8 : nullptr;
        p.after_prepass = after_prepass;
        p.sched = sched;
        p.alpha = alpha; p.beta = beta; p.C = C;
        e = k->launch_i8(p, stream);
    }
    return e == cudaSuccess ? PGEMM_OK : PGEMM_ERR_CUDA;
}

// A block that waits, with a short limit, on an mbarrier nothing arrives on.
__global__ void selftest_wait_kernel(KernelCtx ctx) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0, ctx, kSiteSelfTest);
}

// The int8 GEMM with its widened operands placed in the fixed device buffer
// that `scratch` provides (no allocation); used by the no-allocation entry
// point.
pgemm_status gemm_i8_fixed_scratch(int M, int N, int K, int32_t alpha, const int8_t *A,
                                   const int8_t *B, int32_t beta, int32_t *C,
                                   FixedScratchFn scratch, cudaStream_t stream) {
    return gemm_impl<Kind::I8>(M, N, K, alpha, A, B, beta, C, nullptr, stream, scratch);
}

}  // namespace pg

using namespace pg;

extern "C" {

pgemm_status gemm_f32(int M, int N, int K, float alpha, const float *A, const float *B, float beta,
                      float *C, pgemm_stream_t stream) {
    return gemm_impl<Kind::F32>(M, N, K, alpha, A, B, beta, C, nullptr, stream);
}

pgemm_status gemm_bf16(int M, int N, int K, float alpha, const uint16_t *A, const uint16_t *B,
                       float beta, float *C, pgemm_stream_t stream) {
    return gemm_impl<Kind::BF16>(M, N, K, alpha, A, B, beta, C, nullptr, stream);
}

pgemm_status gemm_i8(int M, int N, int K, int32_t alpha, const int8_t *A, const int8_t *B,
                     int32_t beta, int32_t *C, pgemm_stream_t stream) {
    return gemm_impl<Kind::I8>(M, N, K, alpha, A, B, beta, C, nullptr, stream);
}

pgemm_status gemm_f32_ex(int M, int N, int K, float alpha, const float *A, const float *B,
                         float beta, float *C, const pgemm_config *cfg, pgemm_stream_t stream) {
    return gemm_impl<Kind::F32>(M, N, K, alpha, A, B, beta, C, cfg, stream);
}

pgemm_status gemm_bf16_ex(int M, int N, int K, float alpha, const uint16_t *A, const uint16_t *B,
                          float beta, float *C, const pgemm_config *cfg, pgemm_stream_t stream) {
    return gemm_impl<Kind::BF16>(M, N, K, alpha, A, B, beta, C, cfg, stream);
}

pgemm_status gemm_i8_ex(int M, int N, int K, int32_t alpha, const int8_t *A, const int8_t *B,
                        int32_t beta, int32_t *C, const pgemm_config *cfg, pgemm_stream_t stream) {
    return gemm_impl<Kind::I8>(M, N, K, alpha, A, B, beta, C, cfg, stream);
}

pgemm_status pgemm_default_config(pgemm_dtype dtype, int M, int N, int K, pgemm_config *out) {
    if (!out || M < 0 || N < 0 || K < 0) return PGEMM_ERR_INVALID_VALUE;
    if (dtype != PGEMM_F32 && dtype != PGEMM_BF16 && dtype != PGEMM_I8) return PGEMM_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    *out = default_config(dtype, M, N, K, d->sm_count);
    const KernelInfo *k = find_kernel(dtype, *out);
    if (k) out->bk = k->bk;
    return PGEMM_OK;
}

int pgemm_list_configs(pgemm_dtype dtype, pgemm_config *out, int cap) {
    int n = 0;
    const KernelInfo *t = table_of(dtype, &n);
    for (int i = 0; i < n && i < cap && out; ++i) out[i] = pgemm_config{t[i].bm, t[i].bn, t[i].bk, t[i].stages, 0, t[i].producer, t[i].engine, 0};
    return n;
}

pgemm_status pgemm_kernel_attrs(pgemm_dtype dtype, const pgemm_config *cfg, int *smem_bytes,
                                int *regs_per_thread, int *threads_per_block, int *blocks_per_sm) {
    if (!cfg) return PGEMM_ERR_INVALID_VALUE;
    pgemm_config c = *cfg;
    if (c.bm == 0) c.bm = 128;
    const KernelInfo *k = find_kernel(dtype, c);
    if (!k) return PGEMM_ERR_UNSUPPORTED_CONFIG;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    int bps = 0;
    st = kernel_setup(*d, *k, &bps);
    if (st != PGEMM_OK) return st;
    cudaFuncAttributes fa{};
    if (cudaFuncGetAttributes(&fa, k->func) != cudaSuccess) return PGEMM_ERR_CUDA;
    if (smem_bytes) *smem_bytes = k->smem_bytes;
    if (regs_per_thread) *regs_per_thread = fa.numRegs;
    if (threads_per_block) *threads_per_block = k->threads;
    if (blocks_per_sm) *blocks_per_sm = bps;
    return PGEMM_OK;
}

// A piece of a tile is at least kMinStreamKIters K-tiles, below which its
// exchange would cost about what it saves; stream-K is used only when the
// longest share is at most 7/8 of a tile.
constexpr long long kMinStreamKIters = 8;

pgemm_status pgemm_stream_k_plan(long long tiles, int slots, int k_tiles, int max_parts,
                                 long long *sk_tiles, int *sk_slots, int *max_pieces,
                                 long long *share) {
    if (tiles < 0 || slots < 1 || k_tiles < 0 || max_parts < 0 || !sk_tiles || !sk_slots ||
        !max_pieces || !share)
        return PGEMM_ERR_INVALID_VALUE;
    *sk_tiles = 0;
    *sk_slots = 0;
    *max_pieces = 1;
    *share = 0;
    if (max_parts == 1 || k_tiles == 0 || slots < 2) return PGEMM_OK;
    const long long rem = tiles % slots;
    if (rem == 0) return PGEMM_OK;
    const long long total = rem * k_tiles;
    // the most slots one of the R tiles is spread over, with g slots taking part
    auto most_pieces = [&](long long g) {
        // slot holding iteration x: the largest j with j * total / g <= x
        auto slot_of = [&](long long x) { return ((x + 1) * g - 1) / total; };
        long long most = 1;
        for (long long r = 0; r < rem; ++r) {
            const long long p = slot_of((r + 1) * k_tiles - 1) - slot_of(r * k_tiles) + 1;
            if (p > most) most = p;
        }
        return most;
    };
    long long g = slots;
    long long most = most_pieces(g);
    if (max_parts > 1 && most > max_parts) {
        // capped: g = R * p slots, p = min(cap, G / R), so that every tile is
        // exactly p pieces (slot r * p starts tile r)
        long long p = slots / rem;
        if (p > max_parts) p = max_parts;
        if (p < 2) return PGEMM_OK;
        g = rem * p;
        most = p;
    }
    if (total / g < kMinStreamKIters) return PGEMM_OK;
    // worth it only if the longest share saves at least an eighth of a tile
    // over the extra wave it replaces
    const long long longest = (total + g - 1) / g;
    if (longest * 8 > static_cast<long long>(k_tiles) * 7) return PGEMM_OK;
    *sk_tiles = rem;
    *sk_slots = static_cast<int>(g);
    *max_pieces = static_cast<int>(most);
    *share = total / g;
    return PGEMM_OK;
}

pgemm_status pgemm_schedule(pgemm_dtype dtype, const pgemm_config *cfg, int M, int N, int K,
                            long long *tiles, int *slots, long long *split_tiles, int *parts,
                            long long *half_tiles) {
    if (M < 0 || N < 0 || K < 0) return PGEMM_ERR_INVALID_VALUE;
    if (dtype != PGEMM_F32 && dtype != PGEMM_BF16 && dtype != PGEMM_I8) return PGEMM_ERR_INVALID_VALUE;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    pgemm_config c = (cfg && cfg->stages > 0) ? *cfg : default_config(dtype, M, N, K, d->sm_count);
    if (c.bm == 0) c.bm = 128;
    if (cfg) c.max_k_parts = cfg->max_k_parts;
    if (c.max_k_parts < 0) return PGEMM_ERR_INVALID_VALUE;
    const KernelInfo *k = find_kernel(dtype, c);
    if (!k) return PGEMM_ERR_UNSUPPORTED_CONFIG;
    int bps = 0, n = 0;
    st = kernel_setup(*d, *k, &bps, &n);
    if (st != PGEMM_OK) return st;
    TileSchedule s;
    if (k->schedule_slots != nullptr) {
        s = plan_schedule(*k, M, N, K, n, c.max_k_parts);
    } else {
        s.tiles = static_cast<long long>((M + k->bm - 1) / k->bm) * ((N + k->bn - 1) / k->bn);
        s.slots = d->sm_count * bps;
    }
    if (tiles) *tiles = s.tiles;
    if (slots) *slots = s.slots;
    if (split_tiles) *split_tiles = s.split_tiles;
    if (parts) *parts = s.parts;
    if (half_tiles) *half_tiles = s.half_tiles;
    return PGEMM_OK;
}

pgemm_status pgemm_get_device_status(pgemm_stream_t stream) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return PGEMM_ERR_CUDA;
    uint32_t v = 0;
    if (cudaMemcpy(&v, d->status, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess)
        return PGEMM_ERR_CUDA;
    if (v == 0) return PGEMM_OK;
    const uint32_t zero = 0;
    if (cudaMemcpy(d->status, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
        return PGEMM_ERR_CUDA;
    return (v & 0xF0000000u) == kStatusTimeout ? PGEMM_ERR_TIMEOUT : PGEMM_ERR_CUDA;
}

pgemm_status pgemm_selftest_wait_timeout(int limit_us, pgemm_stream_t stream) {
    if (limit_us <= 0 || limit_us > 5000000) return PGEMM_ERR_INVALID_VALUE;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        int dev = 0;
        DeviceState *d = nullptr;
        pgemm_status st = device_setup(&dev, &d);
        if (st != PGEMM_OK) return st;
        KernelCtx ctx{d->status, static_cast<uint64_t>(limit_us) * 1000ull};
        selftest_wait_kernel<<<1, 32, 0, stream>>>(ctx);
        if (cudaGetLastError() != cudaSuccess) return PGEMM_ERR_CUDA;
    }
    return pgemm_get_device_status(stream);
}

pgemm_status pgemm_stage_reuse_demo(const float *X, int rows, int cols, const int *perm,
                                    float *out, int check_reuse, int delay_warp,
                                    unsigned delay_ns, unsigned long long *trace, int trace_cap,
                                    pgemm_stream_t stream) {
    if (rows < 0 || cols <= 0 || cols % 4 != 0 || cols > 8192 || trace_cap < 0 ||
        delay_warp < -1 || delay_warp > 3)
        return PGEMM_ERR_INVALID_VALUE;
    if (rows == 0) return PGEMM_OK;
    if (!X || !perm || !out) return PGEMM_ERR_INVALID_VALUE;
    if (!aligned16(X)) return PGEMM_ERR_MISALIGNED;
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    KernelCtx ctx{d->status, kDefaultWaitLimitNs};
    const int blocks = rows < d->sm_count ? rows : d->sm_count;
    return launch_stage_reuse(X, rows, cols, perm, out, check_reuse, delay_warp, delay_ns, trace,
                              trace_cap, blocks, ctx, stream) == cudaSuccess
               ? PGEMM_OK
               : PGEMM_ERR_CUDA;
}

const char *pgemm_status_string(pgemm_status status) {
    switch (status) {
        case PGEMM_OK: return "ok";
        case PGEMM_ERR_INVALID_VALUE: return "invalid value";
        case PGEMM_ERR_MISALIGNED: return "pointer not 16-byte aligned";
        case PGEMM_ERR_UNSUPPORTED_DEVICE: return "unsupported device (needs sm_103)";
        case PGEMM_ERR_CUDA: return "CUDA error";
        case PGEMM_ERR_TIMEOUT: return "device wait timed out";
        case PGEMM_ERR_UNSUPPORTED_CONFIG: return "configuration not built";
        case PGEMM_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of gemm_i8_noalloc";
    }
    return "unknown status";
}

pgemm_status pgemm_trim_scratch(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    DeviceState *d = nullptr;
    pgemm_status st = device_setup(&dev, &d);
    if (st != PGEMM_OK) return st;
    if (cudaDeviceSynchronize() != cudaSuccess) return PGEMM_ERR_CUDA;
    return cudaMemPoolTrimTo(d->pool, 0) == cudaSuccess ? PGEMM_OK : PGEMM_ERR_CUDA;
}

int pgemm_version(void) { return 100; }

}  // extern "C"
