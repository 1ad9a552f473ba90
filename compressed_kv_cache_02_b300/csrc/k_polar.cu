// Recursive polar-angle encoder: quantize (rotate, polar transform, per-level angle codes, fp16
// radius, QJL signs of the residual) and scoring (the same asymmetric estimator), with the C-ABI
// entry points tq_polar_* of include/tq.h.
//
// Pages: csdn tutorial, section "将笛卡尔积坐标转为极坐标" (a radius kept at FP16 plus d - 1 low-bit
// angles) and section "TurboQuant原理剖析" (2 or 3 bits per angle, then 1 QJL bit per dimension);
// freelamp article, section "技术突破：极坐标量化" (rotation first, then a recursive polar transform
// into one radius and a series of angles with an analytic law).
//
// The transform pairs neighbours: level 1 maps (y_2i, y_2i+1) to a radius and an angle in
// [0, 2 pi), level l pairs the level-(l-1) radii into an angle in [0, pi/2], down to one radius.
// Codes of the d - 1 angles are consecutive b-bit fields of one bit stream, level 1 first.
#include <cuda_runtime.h>

#include <cmath>
#include <new>
#include <string>
#include <vector>

#include "lut.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"
#include "tq_kernels.h"

constexpr int kPolarMaxLevels = 8;   // d <= 256
constexpr int kPolarMaxCodes = 16;   // bits <= 4

struct PolarParams {
    int d, L, bits, m, qjl, cw, ws;   // cw code words, ws sign words per vector
    float qjl_scale;                  // sqrt(pi/2) / m
    float thr[kPolarMaxLevels][kPolarMaxCodes - 1];
    float ccos[kPolarMaxLevels][kPolarMaxCodes], csin[kPolarMaxLevels][kPolarMaxCodes];
};

struct tq_polar {
    int device = 0;
    int d = 0, L = 0, bits = 0, m = 0, qjl = 0;
    std::vector<float> Pi, S;
    std::vector<std::vector<double>> centroids, thresholds;   // per level
    PolarParams prm{};
    float* dPiT = nullptr;   // [d][d] PiT[j*d+i] = Pi[i][j]
    float* dPi = nullptr;    // [d][d] row-major
    float* dST = nullptr;    // [d][m] ST[j*m+i] = S[i][j]
    int* derr = nullptr;
    uint16_t* dbops = nullptr;   // d = 128: tcgen05 operands (Pi, S Pi^T as bf16 pieces)
    float* dcs = nullptr;        // d = 128: [7][32] centroid cosines then sines per level
    int kernel_path = TQ_PATH_AUTO;
};

namespace tq {
namespace {

constexpr int kPolarVecs = 8;       // vectors per quantize pass (each matrix load serves 8 FMAs)
constexpr int kPolarQThreads = 128;

// offset of level l's first angle in the code stream: d/2 + d/4 + ... (l - 1 terms)
__device__ __forceinline__ int level_offset(int d, int l) { return d - (d >> (l - 1)); }

// Shared memory of the quantize kernel (floats): x, y, radii per level (d - 1 in all), codes.
// All four arrays are [coordinate or node][vector], so a thread's loop over the vectors of one
// coordinate is two 16-byte loads and consecutive threads of the tree steps hit consecutive words.
struct QuantSmem {
    float x[256 * kPolarVecs];
    float y[256 * kPolarVecs];     // rotated rows, then the rebuilt y_hat
    float rad[256 * kPolarVecs];   // radii of every tree node (level-1 nodes first)
    unsigned char code[256 * kPolarVecs];
    float red[kPolarVecs][kPolarQThreads / 32];
    float nrm[kPolarVecs];
};

__device__ __forceinline__ int angle_code(float psi, const float* thr, int nthr) {
    int c = 0;
    for (int t = 0; t < nthr; ++t) c += psi > thr[t];
    return c;
}

// Block sum of v for each of the kPolarVecs vectors; every thread gets the totals in s.nrm.
__device__ __forceinline__ void block_sums(QuantSmem& s, float (&v)[kPolarVecs]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int r = 0; r < kPolarVecs; ++r) {
        float a = v[r];
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (lane == 0) s.red[r][warp] = a;
    }
    __syncthreads();
    if (threadIdx.x < kPolarVecs) {
        float a = 0.f;
        for (int w = 0; w < kPolarQThreads / 32; ++w) a += s.red[threadIdx.x][w];
        s.nrm[threadIdx.x] = a;
    }
    __syncthreads();
}

struct PolarQuantArgs {
    PolarParams prm;
    const void* x;
    int dtype;
    int64_t n, ld;
    const float* PiT;
    const float* Pi;
    const float* ST;
    uint32_t* codes;
    uint16_t* r16;
    uint32_t* signs;
    uint16_t* rnorm;
    int* err;
};

__global__ void __launch_bounds__(kPolarQThreads) polar_quantize_kernel(const PolarQuantArgs a) {
    __shared__ __align__(16) QuantSmem s;
    const PolarParams& p = a.prm;
    const int d = p.d, nthr = (1 << p.bits) - 1;
    for (int64_t v0 = (int64_t)blockIdx.x * kPolarVecs; v0 < a.n; v0 += (int64_t)gridDim.x * kPolarVecs) {
        const int nv = (int)min((int64_t)kPolarVecs, a.n - v0);
        // 1. rows in, squared norms
        float sq[kPolarVecs];
#pragma unroll
        for (int r = 0; r < kPolarVecs; ++r) sq[r] = 0.f;
        for (int j = threadIdx.x; j < d; j += blockDim.x) {
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) {
                float xv = 0.f;
                if (r < nv) {
                    const int64_t row = v0 + r;
                    xv = a.dtype == TQ_BF16 ? bf16_bits_to_float(static_cast<const uint16_t*>(a.x)[row * a.ld + j])
                                            : static_cast<const float*>(a.x)[row * a.ld + j];
                }
                s.x[(j) * kPolarVecs + (r)] = xv;
                sq[r] = fmaf(xv, xv, sq[r]);
            }
        }
        block_sums(s, sq);   // s.nrm = squared norms until step 6
        // 2. y = Pi x (thread i: row i of Pi through column i of PiT)
        for (int i = threadIdx.x; i < d; i += blockDim.x) {
            float acc[kPolarVecs];
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) acc[r] = 0.f;
            for (int j = 0; j < d; ++j) {
                const float w = __ldg(a.PiT + (size_t)j * d + i);
#pragma unroll
                for (int q = 0; q < kPolarVecs / 4; ++q) {
                    const float4 v = reinterpret_cast<const float4*>(&s.x[j * kPolarVecs])[q];
                    acc[4 * q] = fmaf(w, v.x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
                }
            }
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) s.y[(i) * kPolarVecs + (r)] = acc[r];
        }
        __syncthreads();
        // 3. polar transform level by level: node radii into rad, angle codes into code
        for (int l = 1; l <= p.L; ++l) {
            const int nodes = d >> l, off = level_offset(d, l), poff = l > 1 ? level_offset(d, l - 1) : 0;
            for (int e = threadIdx.x; e < nodes * kPolarVecs; e += blockDim.x) {
                const int i = e / kPolarVecs, r = e - i * kPolarVecs;
                float lo, hi;
                if (l == 1) {
                    lo = s.y[(2 * i) * kPolarVecs + (r)];
                    hi = s.y[(2 * i + 1) * kPolarVecs + (r)];
                } else {
                    lo = s.rad[(poff + 2 * i) * kPolarVecs + (r)];
                    hi = s.rad[(poff + 2 * i + 1) * kPolarVecs + (r)];
                }
                float psi = atan2f(hi, lo);
                if (l == 1 && psi < 0.f) psi += 6.28318530717958647692f;
                s.rad[(off + i) * kPolarVecs + (r)] = sqrtf(fmaf(lo, lo, hi * hi));
                s.code[(off + i) * kPolarVecs + (r)] = (unsigned char)angle_code(psi, p.thr[l - 1], nthr);
            }
            __syncthreads();
        }
        // 4. pack the code stream and store the radius
        for (int e = threadIdx.x; e < nv * p.cw; e += blockDim.x) {
            const int r = e / p.cw, w = e - r * p.cw;
            uint32_t word = 0u;
            for (int b = 0; b < 32; ++b) {
                const int t = 32 * w + b, an = t / p.bits;
                if (an < d - 1) word |= (uint32_t)((s.code[(an) * kPolarVecs + (r)] >> (t - an * p.bits)) & 1) << b;
            }
            a.codes[(v0 + r) * p.cw + w] = word;
        }
        if (threadIdx.x < nv) {
            const uint16_t h = float_to_half_bits(sqrtf(s.nrm[threadIdx.x]));
            if ((h & 0x7fffu) == 0x7c00u) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
            a.r16[v0 + threadIdx.x] = h;
        }
        if (!p.qjl) {
            __syncthreads();
            continue;
        }
        // 5. rebuild y_hat top-down from the stored radius and the angle centroids
        if (threadIdx.x < kPolarVecs)   // the root radius: the stored fp16 norm
            s.rad[(d - 2) * kPolarVecs + (threadIdx.x)] = half_bits_to_float(float_to_half_bits(sqrtf(s.nrm[threadIdx.x])));
        __syncthreads();
        for (int l = p.L; l >= 1; --l) {
            const int nodes = d >> l, off = level_offset(d, l), coff = l > 1 ? level_offset(d, l - 1) : 0;
            for (int e = threadIdx.x; e < nodes * kPolarVecs; e += blockDim.x) {
                const int i = e / kPolarVecs, r = e - i * kPolarVecs;
                const float rho = s.rad[(off + i) * kPolarVecs + (r)];
                const int c = s.code[(off + i) * kPolarVecs + (r)];
                const float lo = rho * p.ccos[l - 1][c], hi = rho * p.csin[l - 1][c];
                if (l == 1) {
                    s.y[(2 * i) * kPolarVecs + (r)] = lo;
                    s.y[(2 * i + 1) * kPolarVecs + (r)] = hi;
                } else {
                    s.rad[(coff + 2 * i) * kPolarVecs + (r)] = lo;
                    s.rad[(coff + 2 * i + 1) * kPolarVecs + (r)] = hi;
                }
            }
            __syncthreads();
        }
        // 6. residual x - Pi^T y_hat (into x) and its squared norm
        float rq[kPolarVecs];
#pragma unroll
        for (int r = 0; r < kPolarVecs; ++r) rq[r] = 0.f;
        for (int j = threadIdx.x; j < d; j += blockDim.x) {
            float acc[kPolarVecs];
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) acc[r] = 0.f;
            for (int i = 0; i < d; ++i) {
                const float w = __ldg(a.Pi + (size_t)i * d + j);
#pragma unroll
                for (int q = 0; q < kPolarVecs / 4; ++q) {
                    const float4 v = reinterpret_cast<const float4*>(&s.y[i * kPolarVecs])[q];
                    acc[4 * q] = fmaf(w, v.x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
                }
            }
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) {
                const float res = s.x[(j) * kPolarVecs + (r)] - acc[r];
                rq[r] = fmaf(res, res, rq[r]);
                acc[r] = res;
            }
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) s.rad[(j) * kPolarVecs + (r)] = acc[r];   // the residual rows
        }
        block_sums(s, rq);
        // 7. signs of S r (thread i: row i of S), one ballot word per warp
        for (int i0 = 0; i0 < p.m; i0 += blockDim.x) {
            const int i = i0 + threadIdx.x;
            float acc[kPolarVecs];
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) acc[r] = 0.f;
            if (i < p.m) {
                for (int j = 0; j < d; ++j) {
                    const float w = __ldg(a.ST + (size_t)j * p.m + i);
#pragma unroll
                    for (int q = 0; q < kPolarVecs / 4; ++q) {
                        const float4 v = reinterpret_cast<const float4*>(&s.rad[j * kPolarVecs])[q];
                        acc[4 * q] = fmaf(w, v.x, acc[4 * q]);
                        acc[4 * q + 1] = fmaf(w, v.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = fmaf(w, v.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = fmaf(w, v.w, acc[4 * q + 3]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kPolarVecs; ++r) {
                const uint32_t bal = __ballot_sync(0xffffffffu, i < p.m && acc[r] > 0.f);
                if ((threadIdx.x & 31) == 0 && r < nv && i < p.m) a.signs[(v0 + r) * p.ws + (i >> 5)] = bal;
            }
        }
        if (threadIdx.x < nv) {
            const uint16_t h = float_to_half_bits(sqrtf(s.nrm[threadIdx.x]));
            if ((h & 0x7fffu) == 0x7c00u) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
            a.rnorm[v0 + threadIdx.x] = h;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- scoring
//
// est(q, x) = r16 <Pi q, y_hat> + rnorm16 sqrt(pi/2)/m (2 M_u(signs) - sum u),  u = S q.
// <Pi q, y_hat> is evaluated bottom-up over the tree: a level-1 node i contributes
// q'_2i cos(c) + q'_2i+1 sin(c) (a table over the 2^b codes of pair i, 4 queries per float4), and
// a node above combines its children as cos(c) left + sin(c) right, which is rebuilding y_hat
// and taking the dot product in one pass.  One thread per key walks the d/2 leaves left to right
// with a stack of pending left children (one per level).

constexpr int kPolarSThreads = 256;

struct PolarScoreArgs {
    PolarParams prm;
    const float* q;       // [nq][d] raw queries
    int64_t nq;
    const float* PiT;
    const float* ST;
    const uint32_t* codes;
    const uint16_t* r16;
    const uint32_t* signs;
    const uint16_t* rnorm;
    int64_t n;
    float scale;
    float* out;           // [nq][n]
};

template <int D, int B>
struct PolarShape {
    static constexpr int L = D == 16 ? 4 : D == 32 ? 5 : D == 64 ? 6 : D == 128 ? 7 : 8;
    static constexpr int NC = 1 << B;
    static constexpr int CW = ((D - 1) * B + 31) / 32;
    static constexpr int WS = (D + 31) / 32;
    static size_t smem_bytes() {
        return sizeof(float4) * ((size_t)(D / 2) * NC + (size_t)(D / 8) * 256) + sizeof(float2) * (size_t)L * NC +
               sizeof(float) * 3 * 4 * D;
    }
};

// Code of angle a (a compile-time constant after unrolling): bits a*B .. a*B+B-1 of the stream.
template <int B, int CW>
__device__ __forceinline__ int angle_field(const uint32_t (&w)[CW], int a) {
    const int t = a * B, k = t >> 5, sh = t & 31;
    uint32_t v = w[k] >> sh;
    if (sh + B > 32) v |= w[k + 1] << (32 - sh);
    return (int)(v & ((1u << B) - 1u));
}

template <int D, int B>
__global__ void __launch_bounds__(kPolarSThreads) polar_scores_kernel(const PolarScoreArgs a) {
    using S = PolarShape<D, B>;
    constexpr int L = S::L, NC = S::NC, CW = S::CW, WS = S::WS;
    extern __shared__ float4 psm[];
    float4* T1 = psm;                                  // [D/2][NC]
    float4* Tu = T1 + (D / 2) * NC;                    // [D/8][256]
    float2* CS = reinterpret_cast<float2*>(Tu + (D / 8) * 256);   // [L][NC] (level l at l - 1)
    float* qraw = reinterpret_cast<float*>(CS + L * NC);          // [4][D]
    float* qs = qraw + 4 * D;                          // [4][D] Pi q
    float* us = qs + 4 * D;                            // [4][D] S q
    __shared__ float4 s_usum;
    const PolarParams& p = a.prm;
    const bool qjl = p.qjl != 0;
    const int64_t h0 = (int64_t)blockIdx.y * 4;
    const int nh = (int)min((int64_t)4, a.nq - h0);
    // queries of this quad, rotated and projected (rows past nq are zero)
    stage_quad(qraw, D, a.q, D, (int)h0, (int)min(a.nq, (int64_t)INT32_MAX), D);
    __syncthreads();
    for (int e = threadIdx.x; e < 4 * D; e += blockDim.x) {
        const int r = e / D, i = e - r * D;
        float aq = 0.f, au = 0.f;
        for (int j = 0; j < D; ++j) {
            const float x = qraw[r * D + j];
            aq = fmaf(__ldg(a.PiT + (size_t)j * D + i), x, aq);
            if (qjl) au = fmaf(__ldg(a.ST + (size_t)j * D + i), x, au);
        }
        qs[e] = aq;
        us[e] = au;
    }
    for (int e = threadIdx.x; e < L * NC; e += blockDim.x) {
        const int l = e / NC, c = e - l * NC;
        CS[e] = make_float2(p.ccos[l][c], p.csin[l][c]);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < (D / 2) * NC; e += blockDim.x) {
        const int i = e / NC, c = e - i * NC;
        const float cc = p.ccos[0][c], sc = p.csin[0][c];
        T1[e] = make_float4(fmaf(qs[2 * i], cc, qs[2 * i + 1] * sc), fmaf(qs[D + 2 * i], cc, qs[D + 2 * i + 1] * sc),
                            fmaf(qs[2 * D + 2 * i], cc, qs[2 * D + 2 * i + 1] * sc),
                            fmaf(qs[3 * D + 2 * i], cc, qs[3 * D + 2 * i + 1] * sc));
    }
    if (qjl) build_byte_tables(Tu, us, D, D / 8);
    __syncthreads();
    if (threadIdx.x == 0) s_usum = qjl ? table_total(Tu, D / 8) : make_float4(0.f, 0.f, 0.f, 0.f);
    __syncthreads();
    const float4 usum = s_usum;
    const float kq = p.qjl_scale;
    for (int64_t key = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; key < a.n; key += (int64_t)gridDim.x * blockDim.x) {
        uint32_t w[CW];
#pragma unroll
        for (int k = 0; k < CW; ++k) w[k] = __ldg(a.codes + key * CW + k);
        float4 st[L];
        float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int i = 0; i < D / 2; ++i) {
            v = T1[i * NC + angle_field<B>(w, i)];
#pragma unroll
            for (int l = 1; l < L; ++l) {
                if (((i >> (l - 1)) & 1) == 0) {   // a left child at level l: park it
                    st[l] = v;
                    break;
                }
                // a right child: the parent at level l + 1, index i >> l
                const float2 cs = CS[l * NC + angle_field<B>(w, (D - (D >> l)) + (i >> l))];
                v = make_float4(fmaf(cs.x, st[l].x, cs.y * v.x), fmaf(cs.x, st[l].y, cs.y * v.y),
                                fmaf(cs.x, st[l].z, cs.y * v.z), fmaf(cs.x, st[l].w, cs.y * v.w));
            }
        }
        float4 e = f4_scale(half_bits_to_float(__ldg(a.r16 + key)), v);
        if (qjl) {
            uint32_t sg[WS];
#pragma unroll
            for (int k = 0; k < WS; ++k) sg[k] = __ldg(a.signs + key * WS + k);
            const float4 mu = masked_sum<WS>(Tu, sg, D / 8);
            const float rho = half_bits_to_float(__ldg(a.rnorm + key)) * kq;
            e = make_float4(fmaf(rho, 2.f * mu.x - usum.x, e.x), fmaf(rho, 2.f * mu.y - usum.y, e.y),
                            fmaf(rho, 2.f * mu.z - usum.z, e.z), fmaf(rho, 2.f * mu.w - usum.w, e.w));
        }
        float* o = a.out + h0 * a.n + key;
        o[0] = a.scale * e.x;
        if (nh > 1) o[a.n] = a.scale * e.y;
        if (nh > 2) o[2 * a.n] = a.scale * e.z;
        if (nh > 3) o[3 * a.n] = a.scale * e.w;
    }
}

template <int D, int B>
cudaError_t launch_polar_scores(const PolarScoreArgs& a, int sms, cudaStream_t s) {
    using S = PolarShape<D, B>;
    const size_t smem = S::smem_bytes();
    cudaError_t e = cudaFuncSetAttribute(polar_scores_kernel<D, B>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int64_t need = (a.n + kPolarSThreads - 1) / kPolarSThreads;
    const int64_t quads = (a.nq + 3) / 4;
    int64_t bx = (2 * (int64_t)sms + quads - 1) / quads;   // about two CTAs per SM in all
    if (bx > need) bx = need;
    if (bx < 1) bx = 1;
    polar_scores_kernel<D, B><<<dim3((unsigned)bx, (unsigned)quads), kPolarSThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_polar_scores_b(const PolarScoreArgs& a, int sms, cudaStream_t s) {
    switch (a.prm.bits) {
        case 1: return launch_polar_scores<D, 1>(a, sms, s);
        case 2: return launch_polar_scores<D, 2>(a, sms, s);
        case 3: return launch_polar_scores<D, 3>(a, sms, s);
        case 4: return launch_polar_scores<D, 4>(a, sms, s);
    }
    return cudaErrorInvalidValue;
}

cudaError_t launch_polar_scores_any(const PolarScoreArgs& a, int sms, cudaStream_t s) {
    switch (a.prm.d) {
        case 16: return launch_polar_scores_b<16>(a, sms, s);
        case 32: return launch_polar_scores_b<32>(a, sms, s);
        case 64: return launch_polar_scores_b<64>(a, sms, s);
        case 128: return launch_polar_scores_b<128>(a, sms, s);
        case 256: return launch_polar_scores_b<256>(a, sms, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace tq

// ---------------------------------------------------------------- C-ABI

namespace {

int polar_cuda_fail(cudaError_t e, const char* what) {
    return tq::fail(TQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

int check_polar(const tq_polar* c) {
    if (!c) return tq::fail(TQ_ERR_ARG, "polar context is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return polar_cuda_fail(e, "cudaGetDevice");
    if (dev != c->device) return tq::fail(TQ_ERR_ARG, "polar context was created on another device");
    return TQ_OK;
}

void free_polar(tq_polar* c) {
    if (!c) return;
    cudaFree(c->dPiT);
    cudaFree(c->dPi);
    cudaFree(c->dST);
    cudaFree(c->derr);
    cudaFree(c->dbops);
    cudaFree(c->dcs);
    delete c;
}

int polar_levels(int d) {
    int L = 0;
    while ((1 << L) < d) ++L;
    return (1 << L) == d ? L : -1;
}

template <typename T>
int upload_floats(T** dst, const std::vector<T>& src) {
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), src.size() * sizeof(T));
    if (e != cudaSuccess) {
        *dst = nullptr;
        cudaGetLastError();
        return tq::fail(TQ_ERR_OOM, std::string("cudaMalloc of polar tables failed: ") + cudaGetErrorString(e));
    }
    e = cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return polar_cuda_fail(e, "cudaMemcpy of polar tables");
    return TQ_OK;
}

// The tensor-core encoder's operands and centroid table (d = 128 only).
int upload_tc_tables(tq_polar* c) {
    std::vector<float> St;
    if (c->qjl) {   // (S Pi^T)[i][j] = sum_k S[i][k] Pi[j][k], in float64 from the float32 matrices
        St.resize((size_t)128 * 128);
        for (int i = 0; i < 128; ++i)
            for (int j = 0; j < 128; ++j) {
                double acc = 0.0;
                for (int k = 0; k < 128; ++k) acc += (double)c->S[(size_t)i * 128 + k] * (double)c->Pi[(size_t)j * 128 + k];
                St[(size_t)i * 128 + j] = static_cast<float>(acc);
            }
    }
    std::vector<uint16_t> ops;
    tq::build_tc_operands(c->Pi.data(), c->qjl ? St.data() : nullptr, ops);
    int rc = upload_floats(&c->dbops, ops);
    if (rc != TQ_OK) return rc;
    std::vector<float> cs((size_t)7 * 32, 0.f);
    for (int l = 0; l < 7; ++l)
        for (int j = 0; j < (1 << c->bits); ++j) {
            cs[(size_t)32 * l + j] = c->prm.ccos[l][j];
            cs[(size_t)32 * l + 16 + j] = c->prm.csin[l][j];
        }
    return upload_floats(&c->dcs, cs);
}

}  // namespace

extern "C" {

int tq_host_polar_codebook(int level, int bits, double* centroids, double* thresholds) {
    if (level < 1 || level > kPolarMaxLevels || bits < 1 || bits > TQ_POLAR_MAX_BITS || !centroids || !thresholds)
        return tq::fail(TQ_ERR_ARG, "tq_host_polar_codebook: level in 1..8, bits in 1..4, non-NULL outputs");
    std::vector<double> c, t;
    tq::polar_angle_codebook(level, bits, c, t);
    for (size_t i = 0; i < c.size(); ++i) centroids[i] = c[i];
    for (size_t i = 0; i < t.size(); ++i) thresholds[i] = t[i];
    return TQ_OK;
}

int tq_polar_init(tq_polar** out, uint64_t seed, int d, int bits, int qjl, const float* Pi_host, const float* S_host) {
    if (!out) return tq::fail(TQ_ERR_ARG, "tq_polar_init: out is NULL");
    *out = nullptr;
    const int L = polar_levels(d);
    if (L < 4 || L > kPolarMaxLevels) return tq::fail(TQ_ERR_ARG, "tq_polar_init: d must be 16, 32, 64, 128 or 256");
    if (bits < 1 || bits > TQ_POLAR_MAX_BITS) return tq::fail(TQ_ERR_ARG, "tq_polar_init: bits must be in 1..4");
    if (qjl != 0 && qjl != 1) return tq::fail(TQ_ERR_ARG, "tq_polar_init: qjl must be 0 or 1");
    tq_polar* c = new (std::nothrow) tq_polar();
    if (!c) return tq::fail(TQ_ERR_OOM, "tq_polar_init: host allocation failed");
    cudaError_t ce = cudaGetDevice(&c->device);
    if (ce != cudaSuccess) {
        delete c;
        return polar_cuda_fail(ce, "cudaGetDevice");
    }
    c->d = d;
    c->L = L;
    c->bits = bits;
    c->qjl = qjl;
    c->m = qjl ? d : 0;
    std::vector<double> Pd, Sd;
    if (!Pi_host || (qjl && !S_host)) tq::seeded_matrices(seed, d, d, Pd, Sd);
    c->Pi.resize((size_t)d * d);
    for (size_t i = 0; i < c->Pi.size(); ++i) c->Pi[i] = Pi_host ? Pi_host[i] : (float)Pd[i];
    if (qjl) {
        c->S.resize((size_t)d * d);
        for (size_t i = 0; i < c->S.size(); ++i) c->S[i] = S_host ? S_host[i] : (float)Sd[i];
    }
    for (float v : c->Pi)
        if (!std::isfinite(v)) {
            delete c;
            return tq::fail(TQ_ERR_ARG, "tq_polar_init: Pi has a non-finite entry");
        }
    PolarParams& p = c->prm;
    p.d = d;
    p.L = L;
    p.bits = bits;
    p.m = c->m;
    p.qjl = qjl;
    p.cw = ((d - 1) * bits + 31) / 32;
    p.ws = qjl ? (d + 31) / 32 : 0;
    p.qjl_scale = qjl ? (float)(std::sqrt(M_PI / 2.0) / d) : 0.f;
    c->centroids.resize(L);
    c->thresholds.resize(L);
    for (int l = 1; l <= L; ++l) {
        tq::polar_angle_codebook(l, bits, c->centroids[l - 1], c->thresholds[l - 1]);
        for (int j = 0; j < (1 << bits); ++j) {
            p.ccos[l - 1][j] = (float)std::cos(c->centroids[l - 1][j]);
            p.csin[l - 1][j] = (float)std::sin(c->centroids[l - 1][j]);
        }
        for (int j = 0; j + 1 < (1 << bits); ++j) p.thr[l - 1][j] = (float)c->thresholds[l - 1][j];
    }
    std::vector<float> PiT((size_t)d * d), ST;
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) PiT[(size_t)j * d + i] = c->Pi[(size_t)i * d + j];
    int rc = upload_floats(&c->dPiT, PiT);
    if (rc == TQ_OK) rc = upload_floats(&c->dPi, c->Pi);
    if (rc == TQ_OK && qjl) {
        ST.resize((size_t)d * d);
        for (int i = 0; i < d; ++i)
            for (int j = 0; j < d; ++j) ST[(size_t)j * d + i] = c->S[(size_t)i * d + j];
        rc = upload_floats(&c->dST, ST);
    }
    if (rc == TQ_OK && d == 128) rc = upload_tc_tables(c);
    if (rc == TQ_OK) {
        ce = cudaMalloc(reinterpret_cast<void**>(&c->derr), sizeof(int));
        if (ce == cudaSuccess) ce = cudaMemset(c->derr, 0, sizeof(int));
        if (ce != cudaSuccess) rc = polar_cuda_fail(ce, "cudaMalloc of the polar error word");
    }
    if (rc != TQ_OK) {
        free_polar(c);
        return rc;
    }
    *out = c;
    return TQ_OK;
}

void tq_polar_destroy(tq_polar* ctx) { free_polar(ctx); }

int tq_polar_layout(const tq_polar* ctx, int* code_words, int* sign_words) {
    if (!ctx) return tq::fail(TQ_ERR_ARG, "tq_polar_layout: context is NULL");
    if (code_words) *code_words = ctx->prm.cw;
    if (sign_words) *sign_words = ctx->prm.ws;
    return TQ_OK;
}

int tq_polar_quantize(tq_polar* ctx, const void* x, int dtype, int64_t n, int64_t ld_x, uint32_t* codes,
                      uint16_t* r16, uint32_t* signs, uint16_t* rnorm16, void* stream) {
    int rc = check_polar(ctx);
    if (rc != TQ_OK) return rc;
    if (n < 0 || (dtype != TQ_F32 && dtype != TQ_BF16) || ld_x < ctx->d)
        return tq::fail(TQ_ERR_ARG, "tq_polar_quantize: n >= 0, dtype TQ_F32 or TQ_BF16, ld_x >= d");
    if (n == 0) return TQ_OK;
    if (!x || !codes || !r16 || (ctx->qjl && (!signs || !rnorm16)))
        return tq::fail(TQ_ERR_ARG, "tq_polar_quantize: NULL buffer");
    const bool tc_fits = ctx->dbops && dtype == TQ_BF16 && (ld_x % 8) == 0 && (reinterpret_cast<uintptr_t>(x) % 16) == 0;
    if (tc_fits && (ctx->kernel_path == TQ_PATH_TENSOR || (ctx->kernel_path == TQ_PATH_AUTO && n >= 4096))) {
        tq::PolarTcLaunch L{};
        L.device = ctx->device;
        L.x = x;
        L.n = n;
        L.ld_x = ld_x;
        L.bops = ctx->dbops;
        L.cs = ctx->dcs;
        L.bits = ctx->bits;
        L.qjl = ctx->qjl;
        L.cw = ctx->prm.cw;
        for (int l = 2; l <= 7; ++l)
            for (int t = 0; t + 1 < (1 << ctx->bits); ++t) {
                const double tn = std::tan(ctx->thresholds[l - 1][t]);
                L.tau[l - 2][t] = (float)(tn * tn);
            }
        L.codes = codes;
        L.r16 = r16;
        L.signs = signs;
        L.rnorm = rnorm16;
        L.err = ctx->derr;
        cudaError_t e = tq::launch_polar_tc(L, static_cast<cudaStream_t>(stream));
        return e == cudaSuccess ? TQ_OK : polar_cuda_fail(e, "polar_tc2_kernel launch");
    }
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device);
    tq::PolarQuantArgs a{ctx->prm, x, dtype, n, ld_x, ctx->dPiT, ctx->dPi, ctx->dST, codes, r16, signs, rnorm16, ctx->derr};
    const int64_t passes = (n + tq::kPolarVecs - 1) / tq::kPolarVecs;
    const int grid = (int)std::min<int64_t>(passes, (int64_t)sms * 8);
    tq::polar_quantize_kernel<<<grid, tq::kPolarQThreads, 0, static_cast<cudaStream_t>(stream)>>>(a);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? TQ_OK : polar_cuda_fail(e, "polar_quantize_kernel launch");
}

int tq_polar_set_kernel_path(tq_polar* ctx, int path) {
    if (!ctx) return tq::fail(TQ_ERR_ARG, "tq_polar_set_kernel_path: context is NULL");
    if (path != TQ_PATH_AUTO && path != TQ_PATH_CUDA_CORE && path != TQ_PATH_TENSOR)
        return tq::fail(TQ_ERR_ARG, "tq_polar_set_kernel_path: path must be TQ_PATH_AUTO, TQ_PATH_CUDA_CORE or TQ_PATH_TENSOR");
    ctx->kernel_path = path;
    return TQ_OK;
}

int tq_polar_scores(tq_polar* ctx, const float* q, int64_t nq, const uint32_t* codes, const uint16_t* r16,
                    const uint32_t* signs, const uint16_t* rnorm16, int64_t n, float scale, float* out, void* stream) {
    int rc = check_polar(ctx);
    if (rc != TQ_OK) return rc;
    if (nq < 0 || n < 0 || nq > 4 * (int64_t)65535) return tq::fail(TQ_ERR_ARG, "tq_polar_scores: 0 <= nq <= 262140, n >= 0");
    if (nq == 0 || n == 0) return TQ_OK;
    if (!q || !codes || !r16 || !out || (ctx->qjl && (!signs || !rnorm16)))
        return tq::fail(TQ_ERR_ARG, "tq_polar_scores: NULL buffer");
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, ctx->device);
    tq::PolarScoreArgs a{ctx->prm, q, nq, ctx->dPiT, ctx->dST, codes, r16, signs, rnorm16, n, scale, out};
    cudaError_t e = tq::launch_polar_scores_any(a, sms, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : polar_cuda_fail(e, "polar_scores_kernel launch");
}

int tq_polar_sync_status(tq_polar* ctx, void* stream, int* flags) {
    int rc = check_polar(ctx);
    if (rc != TQ_OK) return rc;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return polar_cuda_fail(e, "cudaStreamSynchronize");
    int h = 0;
    e = cudaMemcpy(&h, ctx->derr, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(ctx->derr, 0, sizeof(int));
    if (e != cudaSuccess) return polar_cuda_fail(e, "reading the polar error word");
    if (flags) *flags = h;
    return h ? tq::fail(TQ_ERR_DEVICE, "a device-side check failed (flags " + std::to_string(h) + ")") : TQ_OK;
}

}  // extern "C"
