// e4m3 tensor-core helpers shared by the logits and search kernels: exact query splitting
// into e4m3 pieces, bit-plane to e4m3 fragment extraction, and mma.sync m16n8k32.
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
// piece pc of v * 2^e0 (pieces b0 + b1/16 + b2/256 + b3/4096)
__device__ __forceinline__ uint32_t piece(float v, int e0, int pc) {
    float x = ldexpf(v, e0);
    uint32_t b = to_e4m3(x);
    for (int p = 0; p < pc; ++p) {
        x = (x - from_e4m3(b)) * 16.f;
        b = to_e4m3(x);
    }
    return b;
}
// bits q, q+8, q+16, q+24 of x as e4m3 bytes 0 / 2^-6
__device__ __forceinline__ uint32_t ext(uint32_t x, int q) {
    return (q <= 3 ? (x << (3 - q)) : (x >> (q - 3))) & 0x08080808u;
}

__device__ __forceinline__ void mma_e4m3(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint2 b) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.f32.e4m3.e4m3.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b.x), "r"(b.y));
}

// bits 4t..4t+3 of x (t = 0..3) as e4m3 bytes 0 / 2^-6, in order (byte i <- bit 4t + i)
__device__ __forceinline__ uint32_t ext_nibble(uint32_t x, int t) {
    return (((x >> (4 * t)) & 15u) * (0x00204081u << 3)) & 0x08080808u;
}

// Column exponent e0 for a family whose largest scaled magnitude is mx: mx 2^e0 in [128, 256).
__device__ __forceinline__ int column_exponent(float mx) {
    int E = 0;
    frexpf(mx, &E);
    return mx > 0.f ? 8 - E : 0;
}

}  // namespace
}  // namespace tq
