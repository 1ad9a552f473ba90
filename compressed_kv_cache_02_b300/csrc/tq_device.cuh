// Device helpers shared by the libtq kernels.
#pragma once

#include <cuda_fp16.h>
#include <cstdint>

#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ void set_error(int* err, int bits) { atomicOr(err, bits); }

__device__ __forceinline__ float half_bits_to_float(uint16_t h) {
    return __half2float(__ushort_as_half(h));
}

__device__ __forceinline__ uint16_t float_to_half_bits(float x) {
    return __half_as_ushort(__float2half_rn(x));
}

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ float4 f4_add(float4 a, float4 b) {
    return make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w);
}
__device__ __forceinline__ float4 f4_fma(float s, float4 a, float4 c) {
    return make_float4(fmaf(s, a.x, c.x), fmaf(s, a.y, c.y), fmaf(s, a.z, c.z), fmaf(s, a.w, c.w));
}
__device__ __forceinline__ float4 f4_scale(float s, float4 a) {
    return make_float4(s * a.x, s * a.y, s * a.z, s * a.w);
}

// Clamp a cache length read from device memory; flag values outside [0, cap].
__device__ __forceinline__ int checked_len(const int32_t* len, int b, int64_t cap, int* err) {
    int L = len[b];
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && err) set_error(err, TQ_DEVERR_LEN_RANGE);
        L = L < 0 ? 0 : static_cast<int>(cap);
    }
    return L;
}

}  // namespace tq
