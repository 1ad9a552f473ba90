// Byte lookup tables for the asymmetric estimator on CUDA cores.
//
// The estimator (juejin.cn post, section 二; csdn tutorial, QJL step 3) needs, per coded
// vector and per query q,
//     <Pi q, c[idx]> = c(0) sum_j q'_j + sum_S kappa_S * M(x_S)     (Walsh form of the table)
//     <S q, 2 sign - 1> = 2 M_u(sign) - sum_j u_j
// where M(x) = sum_j q'_j [bit j of x] is a masked sum of the rotated query over a bit-plane
// word vector x (x_S the XOR of the planes in S).  A masked sum over d bits is the sum of
// ceil(d/8) byte lookups into tables T[k][v] = sum_{i < 8, bit i of v} q'_{8k+i}.  Every
// table entry holds 4 queries (a float4: the GQA group of one KV head, or 4 search
// queries), so one 16-byte shared-memory load serves four dot products.
#pragma once

#include "tq_device.cuh"

namespace tq {

// T[k*256 + v] (k < nbytes) from the 4 rows of a ([4][stride] floats in shared memory,
// zero beyond the data).  Doubling over the bits: T[k][v + 2^i] = T[k][v] + a[8k + i].
__device__ __forceinline__ void build_byte_tables(float4* T, const float* a, int stride, int nbytes) {
    for (int k = threadIdx.x; k < nbytes; k += blockDim.x) T[k * 256] = make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    for (int i = 0; i < 8; ++i) {
        const int half = 1 << i;
        const int total = nbytes << i;
        for (int e = threadIdx.x; e < total; e += blockDim.x) {
            const int k = e >> i;
            const int v = half + (e & (half - 1));
            const int j = 8 * k + i;
            const float4 add = make_float4(a[j], a[stride + j], a[2 * stride + j], a[3 * stride + j]);
            T[k * 256 + v] = f4_add(T[k * 256 + v - half], add);
        }
        __syncthreads();
    }
}

// sum_k T[k][byte k of x] over the first nbytes bytes of the word vector x.
template <int W>
__device__ __forceinline__ float4 masked_sum(const float4* __restrict__ T, const uint32_t (&x)[W], int nbytes) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < W; ++w) {
#pragma unroll
        for (int b = 0; b < 4; ++b) {
            const int k = 4 * w + b;
            if (k < nbytes) s = f4_add(s, T[k * 256 + ((x[w] >> (8 * b)) & 255u)]);
        }
    }
    return s;
}

// Loads n consecutive 32-bit words with the widest aligned vector access the count allows.
template <int N>
__device__ __forceinline__ void load_words(uint32_t (&dst)[N], const uint32_t* __restrict__ src) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4*>(src) + i);
            dst[4 * i] = v.x; dst[4 * i + 1] = v.y; dst[4 * i + 2] = v.z; dst[4 * i + 3] = v.w;
        }
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int i = 0; i < N / 2; ++i) {
            const uint2 v = __ldg(reinterpret_cast<const uint2*>(src) + i);
            dst[2 * i] = v.x; dst[2 * i + 1] = v.y;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = __ldg(src + i);
    }
}

// One coded vector: P bit planes of W words, W sign words, fp16 norms as floats.
template <int W, int P>
struct Coded {
    uint32_t pl[P * W];
    uint32_t sg[W];
    float n, rho;
};

template <int W, int P>
__device__ __forceinline__ void load_coded(Coded<W, P>& k, const uint32_t* __restrict__ planes,
                                           const uint32_t* __restrict__ signs,
                                           const uint16_t* __restrict__ norm,
                                           const uint16_t* __restrict__ rnorm, size_t row, bool qjl) {
    load_words<P * W>(k.pl, planes + row * (P * W));
    k.n = half_bits_to_float(__ldg(norm + row));
    if (qjl) {
        load_words<W>(k.sg, signs + row * W);
        k.rho = half_bits_to_float(__ldg(rnorm + row));
    }
}

// est for the 4 queries of the tables against one coded vector.
template <int W, int P>
__device__ __forceinline__ float4 estimate4(const Params& prm, const float4* __restrict__ Tq,
                                            const float4* __restrict__ Tu, float4 qsum, float4 usum,
                                            int nbq, int nbu, const Coded<W, P>& k) {
    float4 mse = f4_scale(prm.c0, qsum);
#pragma unroll
    for (int t = 0; t < kMaxTerms; ++t) {
        if (t < prm.nterms) {
            const int mask = prm.mask[t];
            uint32_t x[W];
#pragma unroll
            for (int w = 0; w < W; ++w) {
                uint32_t v = 0u;
#pragma unroll
                for (int p = 0; p < P; ++p)
                    if ((mask >> p) & 1) v ^= k.pl[p * W + w];
                x[w] = v;
            }
            mse = f4_fma(prm.kappa[t], masked_sum<W>(Tq, x, nbq), mse);
        }
    }
    float4 e = f4_scale(k.n, mse);
    if (prm.qjl) {
        const float4 ms = masked_sum<W>(Tu, k.sg, nbu);
        const float r = k.rho * prm.qjl_scale;
        e.x = fmaf(r, 2.f * ms.x - usum.x, e.x);
        e.y = fmaf(r, 2.f * ms.y - usum.y, e.y);
        e.z = fmaf(r, 2.f * ms.z - usum.z, e.z);
        e.w = fmaf(r, 2.f * ms.w - usum.w, e.w);
    }
    return e;
}

// Copies 4 query rows (rows r0..r0+3 of src with row stride ld; rows >= nrows or columns
// >= len read as 0) into dst[4][stride] in shared memory.
__device__ __forceinline__ void stage_quad(float* dst, int stride, const float* __restrict__ src,
                                           size_t ld, int r0, int nrows, int len) {
    for (int e = threadIdx.x; e < 4 * stride; e += blockDim.x) {
        const int r = e / stride, j = e - r * stride;
        dst[e] = (r0 + r < nrows && j < len) ? src[(size_t)(r0 + r) * ld + j] : 0.f;
    }
}

// Sum of a table row's full-byte entries = sum of the staged query row (for the c(0) and
// sign-offset terms).  Thread 0 computes it after the tables are built.
__device__ __forceinline__ float4 table_total(const float4* T, int nbytes) {
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int k = 0; k < nbytes; ++k) s = f4_add(s, T[k * 256 + 255]);
    return s;
}

}  // namespace tq

namespace tq {

// Scores 4 staged queries against coded vectors.  Scorer<W, P> (W >= 1) uses the byte
// tables above (W = sign words = plane words, P planes, both compile-time); Scorer<0, 0>
// is the generic path for any d <= TQ_MAX_D: it decodes every coordinate and multiplies
// by the staged queries (float4 per coordinate), with no tables.
template <int W, int P>
struct Scorer {
    float4* Tq;
    float4* Tu;
    float4 qsum, usum;
    int nbq, nbu;

    static __host__ __device__ size_t smem_bytes(const Params& prm) {
        const int nbq = (prm.d + 7) / 8, nbu = prm.qjl ? (prm.m + 7) / 8 : 0;
        return (size_t)(nbq + nbu) * 256 * sizeof(float4) + 4ull * 8 * (nbq + nbu) * sizeof(float) +
               2 * sizeof(float4);
    }

    // Stages query rows qrow0..qrow0+nh-1 (nh <= 4) of qrot [.][d] and qproj [.][m] and
    // builds the tables.  Every thread of the block must call it; it synchronises.
    __device__ void setup(float4* sm, const Params& prm, const float* qrot, const float* qproj,
                          size_t qrow0, int nh) {
        nbq = (prm.d + 7) / 8;
        nbu = prm.qjl ? (prm.m + 7) / 8 : 0;
        Tq = sm;
        Tu = Tq + nbq * 256;
        float* qs = reinterpret_cast<float*>(Tu + nbu * 256);
        float* us = qs + 4 * 8 * nbq;
        float4* sums = reinterpret_cast<float4*>(us + 4 * 8 * nbu);
        stage_quad(qs, 8 * nbq, qrot + qrow0 * prm.d, prm.d, 0, nh, prm.d);
        if (prm.qjl) stage_quad(us, 8 * nbu, qproj + qrow0 * prm.m, prm.m, 0, nh, prm.m);
        __syncthreads();
        build_byte_tables(Tq, qs, 8 * nbq, nbq);
        if (prm.qjl) build_byte_tables(Tu, us, 8 * nbu, nbu);
        if (threadIdx.x == 0) {
            sums[0] = table_total(Tq, nbq);
            sums[1] = prm.qjl ? table_total(Tu, nbu) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        __syncthreads();
        qsum = sums[0];
        usum = sums[1];
    }

    __device__ __forceinline__ float4 operator()(const Params& prm, const uint32_t* planes,
                                                 const uint32_t* signs, const uint16_t* norm,
                                                 const uint16_t* rnorm, size_t row) const {
        Coded<W, P> k;
        load_coded(k, planes, signs, norm, rnorm, row, prm.qjl != 0);
        return estimate4<W, P>(prm, Tq, Tu, qsum, usum, nbq, nbu, k);
    }
};

template <>
struct Scorer<0, 0> {
    const float4* qg;   // [d] : the 4 staged rotated queries per coordinate
    const float4* ug;   // [m]
    const float* cv;    // [L] : the centroid table (from the context's device table, any P)

    static __host__ __device__ size_t smem_bytes(const Params& prm) {
        return (size_t)(prm.d + (prm.qjl ? prm.m : 0)) * sizeof(float4) + (size_t)kMaxCodeLevels * sizeof(float);
    }

    __device__ void setup(float4* sm, const Params& prm, const float* qrot, const float* qproj,
                          size_t qrow0, int nh) {
        float4* q4 = sm;
        float4* u4 = sm + prm.d;
        float* c = reinterpret_cast<float*>(u4 + (prm.qjl ? prm.m : 0));
        for (int j = threadIdx.x; j < prm.d; j += blockDim.x) {
            float v[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) v[r] = r < nh ? qrot[(qrow0 + r) * prm.d + j] : 0.f;
            q4[j] = make_float4(v[0], v[1], v[2], v[3]);
        }
        if (prm.qjl) {
            for (int j = threadIdx.x; j < prm.m; j += blockDim.x) {
                float v[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) v[r] = r < nh ? qproj[(qrow0 + r) * prm.m + j] : 0.f;
                u4[j] = make_float4(v[0], v[1], v[2], v[3]);
            }
        }
        for (int k = threadIdx.x; k < prm.L; k += blockDim.x) c[k] = prm.tab[k];
        __syncthreads();
        qg = q4;
        ug = u4;
        cv = c;
    }

    __device__ float4 operator()(const Params& prm, const uint32_t* planes, const uint32_t* signs,
                                 const uint16_t* norm, const uint16_t* rnorm, size_t row) const {
        const uint32_t* pr = planes + row * (size_t)(prm.P * prm.W);
        float4 mse = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < prm.W; ++w) {
            uint32_t pw[TQ_MAX_MSE_BITS];
            for (int p = 0; p < prm.P; ++p) pw[p] = __ldg(pr + p * prm.W + w);
            const int jend = min(32, prm.d - 32 * w);
            for (int bit = 0; bit < jend; ++bit) {
                int idx = 0;
                for (int p = 0; p < prm.P; ++p) idx |= ((pw[p] >> bit) & 1u) << p;
                mse = f4_fma(cv[idx], qg[32 * w + bit], mse);
            }
        }
        float4 e = f4_scale(half_bits_to_float(__ldg(norm + row)), mse);
        if (prm.qjl) {
            const uint32_t* sr = signs + row * (size_t)prm.Ws;
            float4 qj = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int w = 0; w < prm.Ws; ++w) {
                const uint32_t sw = __ldg(sr + w);
                const int jend = min(32, prm.m - 32 * w);
                for (int bit = 0; bit < jend; ++bit)
                    qj = f4_fma(((sw >> bit) & 1u) ? 1.f : -1.f, ug[32 * w + bit], qj);
            }
            const float r = half_bits_to_float(__ldg(rnorm + row)) * prm.qjl_scale;
            e = f4_fma(r, qj, e);
        }
        return e;
    }
};

// Whether the table path applies to a context (and its shared memory fits one CTA).
__host__ __device__ inline bool lut_path_ok(const Params& prm, size_t extra_smem, size_t smem_limit) {
    const int W = prm.W;
    if (W < 1 || W > 7 || prm.P < 1 || prm.P > kFastBits) return false;
    if (prm.qjl && prm.Ws != W) return false;
    const int nbq = (prm.d + 7) / 8, nbu = prm.qjl ? (prm.m + 7) / 8 : 0;
    const size_t need = (size_t)(nbq + nbu) * 256 * 16 + 4ull * 8 * (nbq + nbu) * 4 + 32 + extra_smem;
    return need <= smem_limit;
}

}  // namespace tq
