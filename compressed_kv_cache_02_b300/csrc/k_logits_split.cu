// Attention logits for split (fractional bit width) key contexts: the first d_hi rotated
// coordinates are coded with the (P+1)-bit table and the rest with the P-bit one (juejin.cn post
// section 四: quality at 3.5 and 2.5 bits per channel).  The estimator is the same as for a
// uniform table (csdn tutorial section QJL step 3): n16 <Pi q, c_g[idx]> + rnorm16 sqrt(pi/2)/m
// <S q, 2 sign - 1>, with c_g the table of the coordinate's group.
//
// Thread per key: its code row (P full planes, then the partial top plane of the first d_hi
// coordinates) is decoded coordinate by coordinate against the 4 query heads of a GQA quad,
// staged in shared memory as float4 (q'_h0[j] .. q'_h3[j]); every thread reads the same j at the
// same time, so the query reads are broadcasts (logits_split_kernel: any d).
//
// For d in (96, 128] with symmetric tables, logits_split_q8_kernel instead uses byte tables of
// the query quad (T[v][k] = sum of q' over the set bits of byte value v at byte position k,
// float4 over the 4 heads): with the Walsh form of each table, <q', c_g[idx]> = c0_hi sum_hi q'
// + c0_lo sum_lo q' + sum_k sum_t kappa_{g(k),t} T[x_t byte k][k], x_t the XOR of the planes
// of the t-th odd subset of the P + 1 planes (the top plane reads 0 at coordinates >= d_hi);
// the low table's coefficients of subsets holding the top plane are 0.  Lanes walk the 16 byte
// positions in a lane-rotated order so that a warp's table reads hit distinct banks.
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
            uint32_t pw[kFastBits];
#pragma unroll
            for (int p = 0; p < kFastBits; ++p) pw[p] = p < prm.P ? __ldg(cr + p * prm.W + w) : 0u;
            const bool hi = 32 * w < prm.d_hi;   // whole words: d_hi % 32 == 0
            const uint32_t top = hi ? __ldg(cr + prm.P * prm.W + w) : 0u;
            const int nj = min(32, d - 32 * w);
            for (int t = 0; t < nj; ++t) {
                int idx = 0;
#pragma unroll
                for (int p = 0; p < kFastBits; ++p) idx |= (int)((pw[p] >> t) & 1u) << p;
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

constexpr int kQ8SThreads = 512;

// t-th positive integer with an odd number of set bits: the odd subsets in increasing order
__host__ __device__ constexpr int odd_subset(int t) { return (2 * t) | (((t ^ (t >> 1) ^ (t >> 2)) & 1) ^ 1); }

// T[v * 16 + k] = sum over the set bits i of v of a[h][8 k + i], float4 over the 4 heads.
__device__ void build_byte_tables(float4* T, const float* a, int stride) {
    if (threadIdx.x < 16) T[threadIdx.x] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    for (int i = 0; i < 8; ++i) {
        const int half = 1 << i;
        for (int e = threadIdx.x; e < (16 << i); e += blockDim.x) {
            const int k = e & 15, v = half + (e >> 4), j = 8 * k + i;
            T[v * 16 + k] = f4_add(T[(v - half) * 16 + k],
                                   make_float4(a[j], a[stride + j], a[2 * stride + j], a[3 * stride + j]));
        }
        __syncthreads();
    }
}

// x rotated right by r bytes (0 <= r < 8) as a 128-bit little-endian vector.
__device__ __forceinline__ void rotate_bytes(const uint32_t (&x)[4], int r, uint32_t (&y)[4]) {
    const bool w1 = r >= 4;
    const uint32_t a0 = w1 ? x[1] : x[0], a1 = w1 ? x[2] : x[1], a2 = w1 ? x[3] : x[2], a3 = w1 ? x[0] : x[3];
    const int sh = 8 * (r & 3);
    y[0] = __funnelshift_r(a0, a1, sh);
    y[1] = __funnelshift_r(a1, a2, sh);
    y[2] = __funnelshift_r(a2, a3, sh);
    y[3] = __funnelshift_r(a3, a0, sh);
}

// PT = planes of a split row counting the top plane (MSE bits of the low table + 1).
template <int PT>
__global__ void __launch_bounds__(kQ8SThreads, 1) logits_split_q8_kernel(const SplitArgs a) {
    constexpr int NT = 1 << (PT - 1);   // odd subsets of PT planes
    extern __shared__ float4 sm[];
    float4* Tq = sm;
    float4* Tu = sm + 4096;
    float* qs = reinterpret_cast<float*>(sm + 8192);
    float* us = qs + 4 * 128;
    __shared__ float4 s_sum[3];   // sum of q' over hi bytes, over lo bytes; sum of u
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int quads = (a.G + 3) / 4, ngroups = a.B * a.Hkv * quads;
    const int khi = prm.d_hi / 8;   // byte positions of the (P+1)-bit coordinates
    int64_t total = 0;
    for (int g = 0; g < ngroups; ++g) {
        int L = a.k.len[g / (a.Hkv * quads)];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        total += (L + 31) / 32;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int b = 0; b < a.B; ++b)
            if (a.k.len[b] < 0 || a.k.len[b] > a.k.cap) set_error(a.err, TQ_DEVERR_LEN_RANGE);
    const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
    float kh[NT], kl[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        kh[t] = prm.kappa_hi[t];
        kl[t] = prm.kappa_lo_x[t];
    }
    const int r = threadIdx.x & 7;
    const int P = PT - 1, W = 4;
    int64_t acc0 = 0;
    for (int g = 0; g < ngroups && acc0 < hi; ++g) {
        const int b = g / (a.Hkv * quads), kvh = (g / quads) % a.Hkv, quad = g % quads;
        int L = a.k.len[b];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        const int64_t nblk = (L + 31) / 32;
        const int64_t b0 = max(lo, acc0) - acc0, b1 = min(hi, acc0 + nblk) - acc0;
        acc0 += nblk;
        if (b0 >= b1) continue;
        const int hbase = kvh * a.G + 4 * quad;
        const int nh = min(4, kvh * a.G + a.G - hbase);
        const size_t qrow0 = (size_t)b * a.Hq + hbase;
        __syncthreads();   // the previous group's tables are no longer read
        for (int e = threadIdx.x; e < 4 * 128; e += blockDim.x) {
            const int h = e >> 7, j = e & 127;
            qs[e] = (h < nh && j < prm.d) ? a.qrot[(qrow0 + h) * prm.d + j] : 0.f;
            us[e] = (qjl && h < nh && j < prm.m) ? a.qproj[(qrow0 + h) * prm.m + j] : 0.f;
        }
        __syncthreads();
        build_byte_tables(Tq, qs, 128);
        if (qjl) build_byte_tables(Tu, us, 128);
        if (threadIdx.x == 0) {
            float4 sh = make_float4(0.f, 0.f, 0.f, 0.f), sl = sh, su = sh;
            for (int k = 0; k < 16; ++k) {
                if (k < khi) sh = f4_add(sh, Tq[255 * 16 + k]);
                else sl = f4_add(sl, Tq[255 * 16 + k]);
                if (qjl) su = f4_add(su, Tu[255 * 16 + k]);
            }
            s_sum[0] = sh;
            s_sum[1] = sl;
            s_sum[2] = su;
        }
        __syncthreads();
        const float kq = prm.qjl_scale;
        const float4 cq = f4_fma(prm.c0_hi, s_sum[0], f4_scale(prm.c0, s_sum[1]));
        const float4 cu = f4_scale(-kq, s_sum[2]);
        const size_t rowbase = ((size_t)b * a.Hkv + kvh) * a.k.cap, cap = a.k.cap;
        float* out = a.logits + qrow0 * cap;
        const int64_t kend = min((int64_t)L, b1 * 32);
        for (int64_t key = b0 * 32 + threadIdx.x; key < kend; key += kQ8SThreads) {
            const size_t row = rowbase + key;
            const uint32_t* cr = a.k.planes + row * prm.row_words;
            uint32_t pl[PT][4], y[PT][4], sg[4], ys[4];
#pragma unroll
            for (int p = 0; p < PT; ++p)
#pragma unroll
                for (int w = 0; w < 4; ++w)
                    pl[p][w] = p < P ? __ldg(cr + p * W + w) : (w < prm.W_hi ? __ldg(cr + P * W + w) : 0u);
#pragma unroll
            for (int w = 0; w < 4; ++w) sg[w] = qjl ? __ldg(a.k.signs + row * 4 + w) : 0u;
            const float n = half_bits_to_float(__ldg(a.k.norm + row));
            const float rho = qjl ? half_bits_to_float(__ldg(a.k.rnorm + row)) : 0.f;
#pragma unroll
            for (int p = 0; p < PT; ++p) rotate_bytes(pl[p], r, y[p]);
            rotate_bytes(sg, r, ys);
            float4 m = make_float4(0.f, 0.f, 0.f, 0.f), u = m;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int k = (j + r) & 15;
                const bool hk = k < khi;
#pragma unroll
                for (int t = 0; t < NT; ++t) {
                    uint32_t x = 0u;
#pragma unroll
                    for (int p = 0; p < PT; ++p)
                        if ((odd_subset(t) >> p) & 1) x ^= y[p][j >> 2];
                    m = f4_fma(hk ? kh[t] : kl[t], Tq[((x >> (8 * (j & 3))) & 255u) * 16 + k], m);
                }
                if (qjl) u = f4_add(u, Tu[((ys[j >> 2] >> (8 * (j & 3))) & 255u) * 16 + k]);
            }
            float4 e = f4_scale(n, f4_add(cq, m));
            if (qjl) e = f4_fma(rho, f4_fma(2.f * kq, u, cu), e);
            out[key] = a.scale * e.x;
            if (nh > 1) out[cap + key] = a.scale * e.y;
            if (nh > 2) out[2 * cap + key] = a.scale * e.z;
            if (nh > 3) out[3 * cap + key] = a.scale * e.w;
        }
    }
}

template <int PT>
cudaError_t run_split_q8(const SplitArgs& a, int device, cudaStream_t s) {
    const size_t smem = 8192 * sizeof(float4) + 2 * 4 * 128 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(logits_split_q8_kernel<PT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    logits_split_q8_kernel<PT><<<sms, kQ8SThreads, smem, s>>>(a);
    return cudaGetLastError();
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
    const Params& p = kc->prm;
    if (p.W == 4 && (!p.qjl || p.Ws == 4) && p.split_walsh) {
        switch (p.P + 1) {
            case 2: return run_split_q8<2>(a, kc->device, s);
            case 3: return run_split_q8<3>(a, kc->device, s);
            case 4: return run_split_q8<4>(a, kc->device, s);
        }
    }
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
