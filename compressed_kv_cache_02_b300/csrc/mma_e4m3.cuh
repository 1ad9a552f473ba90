// e4m3 helpers shared by the tensor-core kernels: rounding to e4m3, the exact value of an e4m3
// byte (a value is split into pieces b0 + b1/16 + b2/256 + b3/4096 by rounding the scaled
// remainder again), and the per-column exponent that scales a family of values into range.
#pragma once

#include <cuda_fp8.h>

#include "tq_device.cuh"

namespace tq {
namespace {

__host__ __device__ constexpr int odd_mask(int t) { return (2 * t) | (((t ^ (t >> 1) ^ (t >> 2)) & 1) ^ 1); }

__device__ __forceinline__ uint32_t to_e4m3(float x) {
    return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
// exact value of an e4m3 byte
__device__ __forceinline__ float from_e4m3(uint32_t b) {
    const uint32_t e = (b >> 3) & 15u, m = b & 7u;
    float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : (float)m * 0.001953125f;
    return (b & 0x80u) ? -v : v;
}
// Column exponent e0 for a family whose largest scaled magnitude is mx: mx 2^e0 in [128, 256).
__device__ __forceinline__ int column_exponent(float mx) {
    int E = 0;
    frexpf(mx, &E);
    return mx > 0.f ? 8 - E : 0;
}

}  // namespace
}  // namespace tq
