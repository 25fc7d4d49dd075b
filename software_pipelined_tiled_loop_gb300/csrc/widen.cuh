// Exact int8 -> fp16 widening of packed bytes, shared by the widening pass
// and the tensor-core kernel's register-staged int8 producer.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace pg {

// Four packed int8 values -> two half2 (elements 0, 1 and 2, 3).  Bias each
// byte to b = x + 128, place it under the fp16 exponent 0x64 (the fp16 value
// 1024 + b, exact), and subtract 1152 with one half2 op: 1024 + x + 128 -
// 1152 = x, exact.
__device__ __forceinline__ void widen4(uint32_t w, __half2 &lo, __half2 &hi) {
    const uint32_t b = w ^ 0x80808080u;                    // x + 128 per byte
    const uint32_t l = __byte_perm(b, 0x64646464u, 0x4140);  // [0x64 b1 | 0x64 b0]
    const uint32_t h = __byte_perm(b, 0x64646464u, 0x4342);  // [0x64 b3 | 0x64 b2]
    const __half2 bias = __half2half2(__ushort_as_half(0x6480));  // 1152.0
    lo = __hsub2(*reinterpret_cast<const __half2 *>(&l), bias);
    hi = __hsub2(*reinterpret_cast<const __half2 *>(&h), bias);
}

// Sixteen packed int8 values (one 16-byte vector) -> sixteen fp16 values as
// eight 32-bit words: o[0..3] hold elements 0..7, o[4..7] elements 8..15.
__device__ __forceinline__ void widen16(const uint4 v, uint32_t (&o)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        __half2 lo, hi;
        widen4(w[i], lo, hi);
        o[2 * i] = *reinterpret_cast<const uint32_t *>(&lo);
        o[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&hi);
    }
}

}  // namespace pg
