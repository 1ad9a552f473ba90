// Device helpers shared by the attention kernels: packed fp32 pairs, the odd-subset masks of the
// Walsh form, the lane-rotated byte tables of the 4 query heads and the per-key scorer over them,
// and the warp reductions of the online softmax.
//
// The byte tables (lut.cuh) are stored here as T[v][k] (entry v of byte group k at v * 16 + k,
// 16 groups of 8 bits at d = 128).  At step j a thread looks up group k = (j + r) mod 16,
// r = lane mod 8, so the 8 lanes of each quarter-warp always hit 8 different bank slots whatever
// their byte values; each thread first rotates its 128-bit code vectors right by r bytes so the
// byte positions stay static.
#pragma once

#include <cuda_runtime.h>

#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

using u64 = unsigned long long;
__device__ __forceinline__ u64 pk2(float x, float y) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 upk2(u64 r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// The t-th positive integer with an odd number of set bits (t < 8): 2t + 1 - parity(t).  For
// t < 2^(P-1) these are the odd-size subsets of P bits in increasing order.  Plain arithmetic,
// so it folds to a constant once the loop over t is unrolled.
__host__ __device__ constexpr int odd_mask(int t) { return (2 * t) | (((t ^ (t >> 1) ^ (t >> 2)) & 1) ^ 1); }
static_assert(odd_mask(0) == 1 && odd_mask(1) == 2 && odd_mask(2) == 4 && odd_mask(3) == 7 && odd_mask(4) == 8 &&
                  odd_mask(5) == 11 && odd_mask(6) == 13 && odd_mask(7) == 14,
              "odd-size subsets of 4 bits");
template <int P> struct OddMasks {
    static constexpr int n = 1 << (P - 1);
};


__device__ __forceinline__ void build_tables_vk(float4* T, const float* a, int stride) {
    if (threadIdx.x < 16) T[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    for (int i = 0; i < 8; ++i) {
        const int half = 1 << i;
        for (int e = threadIdx.x; e < (16 << i); e += blockDim.x) {
            const int k = e & 15;
            const int v = half + (e >> 4);
            const int j = 8 * k + i;
            const float4 add = make_float4(a[j], a[stride + j], a[2 * stride + j], a[3 * stride + j]);
            T[v * 16 + k] = f4_add(T[(v - half) * 16 + k], add);
        }
        __syncthreads();
    }
}

// x rotated right by r bytes (0 <= r < 8) as a 128-bit little-endian vector.
__device__ __forceinline__ void rot_bytes(const uint32_t (&x)[4], int r, uint32_t (&y)[4]) {
    const bool w1 = r >= 4;
    const uint32_t a0 = w1 ? x[1] : x[0], a1 = w1 ? x[2] : x[1], a2 = w1 ? x[3] : x[2], a3 = w1 ? x[0] : x[3];
    const int sh = 8 * (r & 3);
    y[0] = __funnelshift_r(a0, a1, sh);
    y[1] = __funnelshift_r(a1, a2, sh);
    y[2] = __funnelshift_r(a2, a3, sh);
    y[3] = __funnelshift_r(a3, a0, sh);
}

template <int P>
__device__ __forceinline__ float4 score_key(const float4* __restrict__ Tq, const float4* __restrict__ Tu,
                                            const uint32_t (&pl)[P][4], const uint32_t (&sg)[4], float n, float rho,
                                            int r, const float* kap, float4 cq, float4 cu, float kq2, bool qjl) {
    constexpr int NT = OddMasks<P>::n;
    uint32_t y[P][4];
#pragma unroll
    for (int p = 0; p < P; ++p) rot_bytes(pl[p], r, y[p]);
    uint32_t ys[4];
    if (qjl) rot_bytes(sg, r, ys);
    float4 m[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) m[t] = make_float4(0.f, 0.f, 0.f, 0.f);
    float4 u = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int k = (j + r) & 15;
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            uint32_t x = 0u;
#pragma unroll
            for (int p = 0; p < P; ++p)
                if ((odd_mask(t) >> p) & 1) x ^= y[p][j >> 2];
            m[t] = f4_add(m[t], Tq[((x >> (8 * (j & 3))) & 255u) * 16 + k]);
        }
        if (qjl) u = f4_add(u, Tu[((ys[j >> 2] >> (8 * (j & 3))) & 255u) * 16 + k]);
    }
    float4 e = cq;   // c0 sum(q'), then the masked sums
#pragma unroll
    for (int t = 0; t < NT; ++t) e = f4_fma(kap[t], m[t], e);
    e = f4_scale(n, e);
    if (qjl) {   // + rho kq (2 M_u - sum u)
        e = f4_fma(rho, cu, e);
        e = f4_fma(rho * kq2, u, e);
    }
    return e;
}

__device__ __forceinline__ float4 f4_max(float4 a, float4 b) {
    return make_float4(fmaxf(a.x, b.x), fmaxf(a.y, b.y), fmaxf(a.z, b.z), fmaxf(a.w, b.w));
}
__device__ __forceinline__ float4 warp_max4(float4 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x = fmaxf(v.x, __shfl_xor_sync(0xffffffffu, v.x, o));
        v.y = fmaxf(v.y, __shfl_xor_sync(0xffffffffu, v.y, o));
        v.z = fmaxf(v.z, __shfl_xor_sync(0xffffffffu, v.z, o));
        v.w = fmaxf(v.w, __shfl_xor_sync(0xffffffffu, v.w, o));
    }
    return v;
}
__device__ __forceinline__ float4 warp_sum4(float4 v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
        v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
        v.z += __shfl_xor_sync(0xffffffffu, v.z, o);
        v.w += __shfl_xor_sync(0xffffffffu, v.w, o);
    }
    return v;
}
// Warp max of each component with the f32 warp reduction (one instruction per component).
__device__ __forceinline__ float4 warp_max4_redux(float4 v) {
    float4 r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r.x) : "f"(v.x));
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r.y) : "f"(v.y));
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r.z) : "f"(v.z));
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r.w) : "f"(v.w));
    return r;
}
// exp(l - m) with exp(-inf - anything) = 0 (no NaN when both are -inf).
__device__ __forceinline__ float safe_exp(float l, float m) { return l == -INFINITY ? 0.f : __expf(l - m); }
__device__ __forceinline__ float rescale(float m_old, float m_new) {
    return m_old == -INFINITY ? 0.f : expf(m_old - m_new);
}

}  // namespace
}  // namespace tq
