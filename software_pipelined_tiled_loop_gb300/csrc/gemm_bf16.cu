// bf16 GEMM: C (fp32) = alpha * A (bf16) * B (bf16) + beta * C, products
// accumulated in fp32 in tensor memory by tcgen05.mma kind::f16.  The kernel
// body, its pipeline and its shared-memory layouts are in tc_gemm.cuh.
#include "tc_gemm.cuh"

namespace pg {

// Eight epilogue warps (two per TMEM lane quadrant, each half the columns),
// so a tile's epilogue takes half as long as with four: at short K the calls
// are bound by the epilogue (a warp stages and stores its 32-column blocks
// one after another).  128-wide tiles with one or two stages keep four,
// which leaves room for two resident blocks per SM.
// CM = CG = 2: a CTA pair computes a 256 x BN tile with one M = 256 MMA (each
// CTA holds half of A's rows and half of B's columns), listed as bm = 256.
// KSUB = 2: stages of 128 K columns (two 64-wide sub-tiles under one barrier
// pair), listed as bk = 128.
template <int BN, int STAGES, int CM = 1, int KSUB = 1>
using Bf16Cfg = TcCfg<BN, STAGES, /*KC=*/0, /*BF16=*/1, /*INT_FOLD=*/false,
                      (BN == 256 || STAGES >= 3) ? 8 : 4, CM, CM, 0, 0, 1, KSUB>;

template <int BN, int STAGES, int CM = 1, int KSUB = 1>
static KernelInfo info_bf16() {
    KernelInfo k = tc_info<Bf16Cfg<BN, STAGES, CM, KSUB>>();
    k.launch_bf16 = launch_tc<Bf16Cfg<BN, STAGES, CM, KSUB>, LaunchBf16>;
    return k;
}

const KernelInfo *bf16_kernels(int *count) {
    static const KernelInfo table[] = {
        info_bf16<256, 2>(), info_bf16<256, 3>(), info_bf16<256, 4>(),
        info_bf16<128, 2>(), info_bf16<128, 3>(), info_bf16<128, 4>(),
        info_bf16<128, 5>(), info_bf16<128, 6>(),
        // S = 1: one slot, load and compute strictly alternate (the unpipelined
        // comparator: "kernel 10" of the SGEMM page)
        info_bf16<256, 1>(), info_bf16<128, 1>(),
        info_bf16<256, 4, 2>(), info_bf16<256, 5, 2>(), info_bf16<256, 6, 2>(),
        // the CTA pair with 128-column stages (three = the bytes of six 64-wide ones)
        info_bf16<256, 2, 2, 2>(), info_bf16<256, 3, 2, 2>(),
    };
    *count = static_cast<int>(sizeof(table) / sizeof(table[0]));
    return table;
}

}  // namespace pg
