// Softmax-weighted value accumulation for one warp: acc[h][j] += w_h(t) * v_hat(t)_j.
//
// Lanes own coordinates, keys are taken one at a time per warp, and the weights of a key
// (4 query heads, float4) come from shared memory.  v_hat is either a bf16 value row or an
// MSE-only code row (planes [P][W]) dequantized in the value context's rotated basis:
// c_v[idx_j] (the norm is folded into the weight and the rotation back is applied once per
// head after the sequence reduction).
#pragma once

#include "tq_device.cuh"

namespace tq {

struct ValueSrc {
    const void* values;   // bf16 [rows][d] or uint32 planes [rows][P][W]
    const uint16_t* norm; // fp16 norms of coded rows
    int P, W, d;
};

// Coordinates of lane `lane`, slot c: the nibble layout (4*lane + c) when NIB, else lane + 32c.
template <bool NIB>
__device__ __forceinline__ int owned_coord(int lane, int c) { return NIB ? 4 * lane + c : lane + 32 * c; }

template <int C, bool CODED, bool NIB>
__device__ __forceinline__ void accumulate_key(float4 (&acc)[C], const ValueSrc& v, size_t row, float4 w,
                                               const float* __restrict__ cv, int lane) {
    if constexpr (CODED) {
        const uint32_t* r = static_cast<const uint32_t*>(v.values) + row * (size_t)(v.P * v.W);
        if constexpr (NIB) {
            // d <= 128, W == 4: lane owns 4*lane .. 4*lane+3, a nibble of word lane/8 of each plane
            uint32_t nib[TQ_MAX_MSE_BITS];
            const int sh = 4 * (lane & 7);
#pragma unroll
            for (int p = 0; p < TQ_MAX_MSE_BITS; ++p)
                nib[p] = p < v.P ? (__ldg(r + p * 4 + (lane >> 3)) >> sh) & 15u : 0u;
#pragma unroll
            for (int c = 0; c < C; ++c) {
                int idx = 0;
#pragma unroll
                for (int p = 0; p < TQ_MAX_MSE_BITS; ++p) idx |= ((nib[p] >> c) & 1u) << p;
                acc[c] = f4_fma(cv[idx], w, acc[c]);
            }
        } else {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                if (c < v.W) {
                    int idx = 0;
                    for (int p = 0; p < v.P; ++p) idx |= ((__ldg(r + p * v.W + c) >> lane) & 1u) << p;
                    acc[c] = f4_fma(cv[idx], w, acc[c]);
                }
            }
        }
    } else {
        const uint16_t* r = static_cast<const uint16_t*>(v.values) + row * (size_t)v.d;
        if constexpr (NIB) {
            const uint2 raw = __ldg(reinterpret_cast<const uint2*>(r) + lane);   // 4 bf16: 4*lane..+3
            const float x[4] = {bf16_bits_to_float(raw.x & 0xffffu), bf16_bits_to_float(raw.x >> 16),
                                bf16_bits_to_float(raw.y & 0xffffu), bf16_bits_to_float(raw.y >> 16)};
#pragma unroll
            for (int c = 0; c < C; ++c) acc[c] = f4_fma(x[c], w, acc[c]);
        } else {
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const int j = lane + 32 * c;
                if (j < v.d) acc[c] = f4_fma(bf16_bits_to_float(__ldg(r + j)), w, acc[c]);
            }
        }
    }
}

}  // namespace tq
