// Attention logits for split (fractional bit width) key contexts: the first d_hi rotated
// coordinates are coded with the (P+1)-bit table and the rest with the P-bit one (juejin.cn post
// section 四: quality at 3.5 and 2.5 bits per channel).  The estimator is the same as for a
// uniform table (csdn tutorial section QJL step 3): n16 <Pi q, c_g[idx]> + rnorm16 sqrt(pi/2)/m
// <S q, 2 sign - 1>, with c_g the table of the coordinate's group.
//
// Thread per key: its code row (P full planes, then the partial top plane of the first d_hi
// coordinates) is decoded coordinate by coordinate against the 4 query heads of a GQA quad,
// staged in shared memory as float4 (q'_h0[j] .. q'_h3[j]); every thread reads the same j at the
// same time, so the query reads are broadcasts.  A straightforward first kernel for this row.
#include "tq_device.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kSplitThreads = 256;
constexpr int kSplitChunk = 4096;   // keys per CTA

struct SplitArgs {
    Params prm;
    const float* qrot;
    const float* qproj;
    int B, Hq, Hkv, G;
    KeyCache k;
    float scale;
    float* logits;
    int* err;
};

__global__ void __launch_bounds__(kSplitThreads) logits_split_kernel(const SplitArgs a) {
    extern __shared__ float4 sq4[];   // [d] query heads, then [m] projected query heads
    __shared__ float s_clo[kMaxLevels], s_chi[kMaxLevels];
    __shared__ float4 s_usum;
    const Params& prm = a.prm;
    const int d = prm.d, m = prm.m;
    const bool qjl = prm.qjl != 0;
    float4* su4 = sq4 + d;
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.k.len, b, a.k.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * kSplitChunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    const size_t qrow0 = (size_t)b * a.Hq + hbase;
    auto head = [&](const float* src, int n, int h, int j) -> float {
        return h < nh ? src[(qrow0 + h) * n + j] : 0.f;
    };
    for (int j = threadIdx.x; j < d; j += blockDim.x)
        sq4[j] = make_float4(head(a.qrot, d, 0, j), head(a.qrot, d, 1, j), head(a.qrot, d, 2, j), head(a.qrot, d, 3, j));
    if (qjl)
        for (int j = threadIdx.x; j < m; j += blockDim.x)
            su4[j] = make_float4(head(a.qproj, m, 0, j), head(a.qproj, m, 1, j), head(a.qproj, m, 2, j),
                                 head(a.qproj, m, 3, j));
    if (threadIdx.x < kMaxLevels) {
        s_clo[threadIdx.x] = prm.centroids[threadIdx.x];
        s_chi[threadIdx.x] = prm.centroids_hi[threadIdx.x];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (qjl)
            for (int j = 0; j < m; ++j) s = f4_add(s, su4[j]);
        s_usum = s;
    }
    __syncthreads();
    const float4 usum = s_usum;
    const float kq = prm.qjl_scale;
    const size_t cap = (size_t)a.k.cap;
    const size_t rowbase = (size_t)bh * cap;
    float* out = a.logits + qrow0 * cap;
    const int64_t iend = min((int64_t)L, i0 + kSplitChunk);
    for (int64_t i = i0 + threadIdx.x; i < iend; i += blockDim.x) {
        const size_t row = rowbase + i;
        const uint32_t* cr = a.k.planes + row * prm.row_words;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < prm.W; ++w) {
            uint32_t pw[TQ_MAX_MSE_BITS];
#pragma unroll
            for (int p = 0; p < TQ_MAX_MSE_BITS; ++p) pw[p] = p < prm.P ? __ldg(cr + p * prm.W + w) : 0u;
            const bool hi = 32 * w < prm.d_hi;   // whole words: d_hi % 32 == 0
            const uint32_t top = hi ? __ldg(cr + prm.P * prm.W + w) : 0u;
            const int nj = min(32, d - 32 * w);
            for (int t = 0; t < nj; ++t) {
                int idx = 0;
#pragma unroll
                for (int p = 0; p < TQ_MAX_MSE_BITS; ++p) idx |= (int)((pw[p] >> t) & 1u) << p;
                idx |= (int)((top >> t) & 1u) << prm.P;
                const float c = hi ? s_chi[idx] : s_clo[idx];
                acc = f4_fma(c, sq4[32 * w + t], acc);
            }
        }
        const float n = half_bits_to_float(__ldg(a.k.norm + row));
        float4 est = f4_scale(n, acc);
        if (qjl) {
            float4 mu = make_float4(0.f, 0.f, 0.f, 0.f);   // sum of u over the set sign bits
            for (int w = 0; w < prm.Ws; ++w) {
                const uint32_t sw = __ldg(a.k.signs + row * prm.Ws + w);
                const int nj = min(32, m - 32 * w);
                for (int t = 0; t < nj; ++t)
                    if ((sw >> t) & 1u) mu = f4_add(mu, su4[32 * w + t]);
            }
            // <S q, 2 sign - 1> = 2 mu - sum u
            const float rk = half_bits_to_float(__ldg(a.k.rnorm + row)) * kq;
            est = f4_fma(rk, make_float4(2.f * mu.x - usum.x, 2.f * mu.y - usum.y, 2.f * mu.z - usum.z,
                                         2.f * mu.w - usum.w), est);
        }
        out[i] = a.scale * est.x;
        if (nh > 1) out[cap + i] = a.scale * est.y;
        if (nh > 2) out[2 * cap + i] = a.scale * est.z;
        if (nh > 3) out[3 * cap + i] = a.scale * est.w;
    }
}

}  // namespace

cudaError_t launch_logits_split(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                                const KeyCache& k, float scale, float* logits, cudaStream_t s) {
    SplitArgs a{};
    a.prm = kc->prm;
    a.qrot = qrot;
    a.qproj = qproj;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.k = k;
    a.scale = scale;
    a.logits = logits;
    a.err = kc->derr;
    const size_t smem = (size_t)(kc->d + kc->m) * sizeof(float4);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(logits_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    const int quads = (a.G + 3) / 4;
    dim3 grid((unsigned)((k.cap + kSplitChunk - 1) / kSplitChunk), (unsigned)(B * Hkv), (unsigned)quads);
    logits_split_kernel<<<grid, kSplitThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace tq
