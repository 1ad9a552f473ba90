// Quantization kernels: rotate + norm + scalar code + bit-pack (PolarQuant stage) fused with
// the residual and its QJL sign sketch; decode-step append; query preparation.
//
// Pages: gitcode.csdn.net tutorial, sections PolarQuant (rotate first), 将笛卡尔积坐标转为
// 极坐标 (r = ||x|| kept as FP16) and QJL steps 1-2 (residual = original - reconstruction,
// Gaussian projection, keep signs > 0 -> 1); juejin.cn post section 二 (most bits on the
// rotated scalar codes, ~1 bit of QJL on the residual).
//
// The residual's projection is computed in the rotated basis: with r' = Pi x - n16 c[idx],
// S r = S Pi^T (Pi x - n16 c[idx]) = (S Pi^T) r'   (Pi orthogonal), and ||r|| = ||r'||.
// S Pi^T is formed once on the host in float64 (tq_api.cu).
#include "tq_device.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kApplyRows = 8;     // input rows per CTA in apply_rows_kernel
constexpr int kQuantThreads = 256;    // bulk inputs (16 vectors per CTA)
constexpr int kAppendThreads = 1024;  // decode appends (4 vectors per CTA, sums split 8 ways)
constexpr int kQuantBatch = 16;       // matrix loads issued before their FMAs

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// out[v][i] = sum_j MT[j][i] in[v][j] for kApplyRows rows per CTA: MT is read coalesced along i,
// each value reused for all rows staged in shared memory.  The sum over j of an output is split
// between S threads (quant_split below: 8 ways at dout <= 128 with 1024 threads), each issuing
// its loads kQuantBatch at a time, and the parts meet in shared memory.
__host__ __device__ constexpr int apply_split(int dout, int T) {
    return dout <= T / 8 ? 8 : (dout <= T / 4 ? 4 : (dout <= T / 2 ? 2 : 1));
}

constexpr int kApplyThreads = 1024;

__global__ void __launch_bounds__(kApplyThreads) apply_rows_kernel(const float* __restrict__ MT, int din, int dout,
                                                                   const float* __restrict__ in, size_t ldi, int64_t nv,
                                                                   float* __restrict__ out, size_t ldo) {
    extern __shared__ float4 xs4[];   // [din][kApplyRows] floats, then the partial sums
    float* xs = reinterpret_cast<float*>(xs4);
    const int S = apply_split(dout, kApplyThreads);
    const int span = kApplyThreads / S, part = threadIdx.x / span, ii = threadIdx.x - part * span;
    float* red = xs + (size_t)din * kApplyRows;   // [S - 1][span][kApplyRows]
    const int64_t v0 = (int64_t)blockIdx.x * kApplyRows;
    for (int e = threadIdx.x; e < din * kApplyRows; e += blockDim.x) {
        const int v = e / din, j = e - v * din;
        xs[j * kApplyRows + v] = (v0 + v < nv) ? in[(size_t)(v0 + v) * ldi + j] : 0.f;
    }
    __syncthreads();
    const int j0 = part * din / S, j1 = (part + 1) * din / S;
    for (int i0 = blockIdx.y * span; i0 < dout; i0 += gridDim.y * span) {
        const int i = i0 + ii;
        const bool valid = i < dout;
        float acc[kApplyRows];
#pragma unroll
        for (int v = 0; v < kApplyRows; ++v) acc[v] = 0.f;
        if (valid) {
            for (int jb = j0; jb < j1; jb += 16) {
                float mv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) mv[u] = jb + u < j1 ? __ldg(MT + (size_t)(jb + u) * dout + i) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    if (jb + u >= j1) break;
                    const float4 a = xs4[(jb + u) * 2], b = xs4[(jb + u) * 2 + 1];
                    acc[0] = fmaf(mv[u], a.x, acc[0]); acc[1] = fmaf(mv[u], a.y, acc[1]);
                    acc[2] = fmaf(mv[u], a.z, acc[2]); acc[3] = fmaf(mv[u], a.w, acc[3]);
                    acc[4] = fmaf(mv[u], b.x, acc[4]); acc[5] = fmaf(mv[u], b.y, acc[5]);
                    acc[6] = fmaf(mv[u], b.z, acc[6]); acc[7] = fmaf(mv[u], b.w, acc[7]);
                }
            }
        }
        if (S > 1) {   // uniform: the loop runs once (span >= dout)
            if (part > 0 && valid)
#pragma unroll
                for (int v = 0; v < kApplyRows; ++v) red[((part - 1) * span + ii) * kApplyRows + v] = acc[v];
            __syncthreads();
            if (part == 0 && valid)
                for (int q = 1; q < S; ++q)
#pragma unroll
                    for (int v = 0; v < kApplyRows; ++v) acc[v] += red[((q - 1) * span + ii) * kApplyRows + v];
        }
        if (part == 0 && valid) {
#pragma unroll
            for (int v = 0; v < kApplyRows; ++v)
                if (v0 + v < nv) out[(size_t)(v0 + v) * ldo + i] = acc[v];
        }
    }
}

struct QuantArgs {
    Params prm;
    const float* PiT;   // [d][d]
    const float* StT;   // [d][m]
    const void* x;
    int dtype;
    int64_t n, ld_x;
    int H;
    int64_t cap;
    const int32_t* len;
    uint32_t* planes;
    uint32_t* signs;
    uint16_t* norm;
    uint16_t* rnorm;
    int* err;
};

// Ways the sum over j of one output coordinate is split between threads (T threads per CTA):
// as many as leave one pass over the outputs, at most 8; 1 for d > T / 2.
__host__ __device__ constexpr int quant_split(int d, int T) {
    return d <= T / 8 ? 8 : (d <= T / 4 ? 4 : (d <= T / 2 ? 2 : 1));
}

// One CTA codes kQuantRows vectors with kT threads (16 vectors and 256 threads for bulk inputs,
// 4 vectors and 1024 threads for the few vectors of a decode append).  Shared memory: the input
// tile and the residual tile, both stored [coordinate][vector] so the matrix-vector loops read
// kQuantRows vectors per j with 16-byte broadcasts, then the split partial sums.
// WIDE (more than kFastBits MSE bits, MSE mode): the table is read from prm.tab into shared
// memory instead of the kernel parameters.
template <int kQuantRows, int kT, bool WIDE>
__global__ void __launch_bounds__(kT) quantize_kernel(const QuantArgs a) {
    static_assert(kQuantRows % 4 == 0, "rows are read four at a time");
    extern __shared__ float4 sm4[];
    const Params& prm = a.prm;
    const int d = prm.d, m = prm.m;
    float* xT = reinterpret_cast<float*>(sm4);   // [d][kQuantRows]
    float* rT = xT + (size_t)d * kQuantRows;      // [d][kQuantRows]
    __shared__ float s_n[kQuantRows], s_n16[kQuantRows], s_r[kQuantRows];
    __shared__ long long s_row[kQuantRows];
    // The tables in shared memory (the binary search indexes them per lane, which the kernel-
    // parameter space would serialise); WIDE: read from prm.tab, up to 256 levels.
    constexpr int kTab = WIDE ? kMaxCodeLevels : kMaxLevels;
    __shared__ float s_cen[kTab], s_thr[kTab], s_cen_hi[kMaxLevels], s_thr_hi[kMaxLevels];
    if constexpr (WIDE) {
        for (int k = threadIdx.x; k < kMaxCodeLevels; k += kT) {
            s_cen[k] = k < prm.L ? prm.tab[k] : 0.f;
            s_thr[k] = k < prm.L - 1 ? prm.tab[prm.L + k] : INFINITY;
        }
    } else if (threadIdx.x < kMaxLevels) {
        s_cen[threadIdx.x] = prm.centroids[threadIdx.x];
        s_thr[threadIdx.x] = prm.thresholds[threadIdx.x];
        s_cen_hi[threadIdx.x] = prm.centroids_hi[threadIdx.x];
        s_thr_hi[threadIdx.x] = prm.thresholds_hi[threadIdx.x];
    }

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t v0 = (int64_t)blockIdx.x * kQuantRows;

    if (tid < kQuantRows) {
        const int64_t v = v0 + tid;
        long long row = -1;
        if (v < a.n) {
            if (a.cap == 0) {
                row = v;
            } else {
                const int L = a.len[v / a.H];
                if (L < 0 || L >= a.cap) set_error(a.err, TQ_DEVERR_LEN_RANGE);
                else row = (long long)v * a.cap + L;
            }
        }
        s_row[tid] = row;
    }
    for (int e = tid; e < kQuantRows * d; e += kT) {
        const int v = e / d, j = e - v * d;
        float val = 0.f;
        if (v0 + v < a.n) {
            const size_t off = (size_t)(v0 + v) * a.ld_x + j;
            val = (a.dtype == TQ_BF16) ? bf16_bits_to_float(static_cast<const uint16_t*>(a.x)[off])
                                       : static_cast<const float*>(a.x)[off];
        }
        xT[j * kQuantRows + v] = val;
    }
    __syncthreads();

    // n = ||x||, n16 = fp16(n)
    for (int v = warp; v < kQuantRows; v += kT / 32) {
        float s = 0.f;
        for (int j = lane; j < d; j += 32) { const float t = xT[j * kQuantRows + v]; s = fmaf(t, t, s); }
        s = warp_sum(s);
        if (lane == 0) {
            const float n = sqrtf(s);
            s_n[v] = n;
            s_n16[v] = half_bits_to_float(float_to_half_bits(n));
        }
    }
    __syncthreads();

    // y = Pi x; idx_j = #(thresholds < y_j / n); planes by warp ballots; r' = y - n16 c[idx].
    // For d <= 128 every output coordinate's sum over j is split between S = 2 (d <= 64: 4)
    // threads, whose partial sums meet in shared memory: all threads load the matrix, and each
    // runs half (a quarter) of the dependent loads, which is what a decode append waits on.
    const int S = quant_split(d, kT);
    const int span = kT / S, part = tid / span, ii = tid - part * span;
    float* red = rT + (size_t)d * kQuantRows;   // [S - 1][span][kQuantRows] partial sums
    const float4* xT4 = reinterpret_cast<const float4*>(xT);
    for (int i0 = 0; i0 < d; i0 += span) {
        const int i = i0 + ii;
        const bool valid = i < d;
        const int j0 = part * d / S, j1 = (part + 1) * d / S;
        float acc[kQuantRows];
#pragma unroll
        for (int v = 0; v < kQuantRows; ++v) acc[v] = 0.f;
        if (valid) {
            // kQuantBatch loads of Pi^T issued before their FMAs (it is usually not in L2 for a decode
            // append, which waits on these rounds of latency)
            for (int jb = j0; jb < j1; jb += kQuantBatch) {
                float pv[kQuantBatch];
#pragma unroll
                for (int u = 0; u < kQuantBatch; ++u) pv[u] = jb + u < j1 ? __ldg(a.PiT + (size_t)(jb + u) * d + i) : 0.f;
#pragma unroll
                for (int u = 0; u < kQuantBatch; ++u) {
                    if (jb + u >= j1) break;
#pragma unroll
                    for (int q = 0; q < kQuantRows / 4; ++q) {
                        const float4 xv = xT4[(jb + u) * (kQuantRows / 4) + q];
                        acc[4 * q] = fmaf(pv[u], xv.x, acc[4 * q]);
                        acc[4 * q + 1] = fmaf(pv[u], xv.y, acc[4 * q + 1]);
                        acc[4 * q + 2] = fmaf(pv[u], xv.z, acc[4 * q + 2]);
                        acc[4 * q + 3] = fmaf(pv[u], xv.w, acc[4 * q + 3]);
                    }
                }
            }
        }
        if (S > 1) {   // one pass (span >= d): fold the parts into part 0
            if (part > 0 && valid)
                for (int v = 0; v < kQuantRows; ++v) red[((part - 1) * span + ii) * kQuantRows + v] = acc[v];
            __syncthreads();
            if (part == 0 && valid)
                for (int q = 1; q < S; ++q)
                    for (int v = 0; v < kQuantRows; ++v) acc[v] += red[((q - 1) * span + ii) * kQuantRows + v];
        }
        if (part > 0) continue;   // whole warps: span is a multiple of 32
        const int word = (i0 >> 5) + warp;
        // split contexts: coordinates below d_hi (whole words, as d_hi % 32 == 0) use the
        // (P+1)-bit table, whose top bit goes to the partial plane after the P full ones
        const bool hi = i < prm.d_hi;
        const int nb = prm.P + (hi ? 1 : 0);
#pragma unroll
        for (int v = 0; v < kQuantRows; ++v) {
            const float n = s_n[v];
            const float u = (n > 0.f) ? acc[v] / n : 0.f;
            // #{k : t_k < u} by binary search over the sorted thresholds
            int idx = 0;
            if constexpr (WIDE) {
#pragma unroll
                for (int b = TQ_MAX_MSE_BITS - 1; b >= 0; --b)
                    if (b < nb) {
                        const int k = idx + (1 << b) - 1;
                        if (u > s_thr[k]) idx += 1 << b;
                    }
            } else {
#pragma unroll
                for (int b = kFastBits - 1; b >= 0; --b)
                    if (b < nb) {
                        const int k = idx + (1 << b) - 1;
                        if (u > (hi ? s_thr_hi[k] : s_thr[k])) idx += 1 << b;
                    }
            }
            const float cval = WIDE ? s_cen[idx] : (hi ? s_cen_hi[idx] : s_cen[idx]);
            if (valid) rT[i * kQuantRows + v] = acc[v] - s_n16[v] * cval;
            const long long row = s_row[v];
            for (int p = 0; p < prm.P; ++p) {
                const unsigned bits = __ballot_sync(0xffffffffu, valid && ((idx >> p) & 1));
                if (lane == 0 && word < prm.W && row >= 0)
                    a.planes[(size_t)row * prm.row_words + (size_t)p * prm.W + word] = bits;
            }
            if (prm.d_hi) {
                const unsigned bits = __ballot_sync(0xffffffffu, valid && hi && ((idx >> prm.P) & 1));
                if (lane == 0 && word < prm.W_hi && row >= 0)
                    a.planes[(size_t)row * prm.row_words + (size_t)prm.P * prm.W + word] = bits;
            }
        }
    }

    if (prm.qjl) {
        __syncthreads();
        for (int v = warp; v < kQuantRows; v += kT / 32) {
            float s = 0.f;
            for (int j = lane; j < d; j += 32) { const float t = rT[j * kQuantRows + v]; s = fmaf(t, t, s); }
            s = warp_sum(s);
            if (lane == 0) s_r[v] = sqrtf(s);
        }
        // sign_j = [((S Pi^T) r')_j > 0], the sum over j split as for y
        const float4* rT4 = reinterpret_cast<const float4*>(rT);
        const int Sm = quant_split(m, kT);
        const int spm = kT / Sm, pm = tid / spm, im = tid - pm * spm;
        for (int i0 = 0; i0 < m; i0 += spm) {
            const int i = i0 + im;
            const bool valid = i < m;
            const int j0 = pm * d / Sm, j1 = (pm + 1) * d / Sm;
            float acc[kQuantRows];
#pragma unroll
            for (int v = 0; v < kQuantRows; ++v) acc[v] = 0.f;
            if (valid) {
                for (int jb = j0; jb < j1; jb += kQuantBatch) {
                    float sv[kQuantBatch];
#pragma unroll
                    for (int u = 0; u < kQuantBatch; ++u) sv[u] = jb + u < j1 ? __ldg(a.StT + (size_t)(jb + u) * m + i) : 0.f;
#pragma unroll
                    for (int u = 0; u < kQuantBatch; ++u) {
                        if (jb + u >= j1) break;
#pragma unroll
                        for (int q = 0; q < kQuantRows / 4; ++q) {
                            const float4 rv = rT4[(jb + u) * (kQuantRows / 4) + q];
                            acc[4 * q] = fmaf(sv[u], rv.x, acc[4 * q]);
                            acc[4 * q + 1] = fmaf(sv[u], rv.y, acc[4 * q + 1]);
                            acc[4 * q + 2] = fmaf(sv[u], rv.z, acc[4 * q + 2]);
                            acc[4 * q + 3] = fmaf(sv[u], rv.w, acc[4 * q + 3]);
                        }
                    }
                }
            }
            if (Sm > 1) {
                __syncthreads();   // the y pass's partial sums are no longer read
                if (pm > 0 && valid)
                    for (int v = 0; v < kQuantRows; ++v) red[((pm - 1) * spm + im) * kQuantRows + v] = acc[v];
                __syncthreads();
                if (pm == 0 && valid)
                    for (int q = 1; q < Sm; ++q)
                        for (int v = 0; v < kQuantRows; ++v) acc[v] += red[((q - 1) * spm + im) * kQuantRows + v];
            }
            if (pm > 0) continue;
            const int word = (i0 >> 5) + warp;
#pragma unroll
            for (int v = 0; v < kQuantRows; ++v) {
                const unsigned bits = __ballot_sync(0xffffffffu, valid && acc[v] > 0.f);
                const long long row = s_row[v];
                if (lane == 0 && word < prm.Ws && row >= 0) a.signs[(size_t)row * prm.Ws + word] = bits;
            }
        }
    }
    __syncthreads();
    if (tid < kQuantRows && s_row[tid] >= 0) {
        const long long row = s_row[tid];
        const uint16_t nh = float_to_half_bits(s_n[tid]);
        a.norm[row] = nh;
        bool overflow = __hisinf(__ushort_as_half(nh));
        if (prm.qjl) {
            const uint16_t rh = float_to_half_bits(s_r[tid]);
            a.rnorm[row] = rh;
            overflow = overflow || __hisinf(__ushort_as_half(rh));
        }
        if (overflow) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
    }
}

__global__ void advance_len_kernel(int32_t* len, int B, int64_t cap, int step, int* err) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    long long v = (long long)len[b] + step;
    if (v < 0 || v > cap) {
        set_error(err, TQ_DEVERR_LEN_RANGE);
        v = v < 0 ? 0 : cap;
    }
    len[b] = static_cast<int32_t>(v);
}

}  // namespace

cudaError_t launch_apply_rows(const float* MT, int din, int dout, const float* in, size_t ldi,
                              int64_t nv, float* out, size_t ldo, cudaStream_t s) {
    if (nv <= 0) return cudaSuccess;
    const int S = apply_split(dout, kApplyThreads), span = kApplyThreads / S;
    const size_t smem = ((size_t)din + (size_t)(S - 1) * span) * kApplyRows * sizeof(float);
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(apply_rows_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    dim3 grid((unsigned)((nv + kApplyRows - 1) / kApplyRows), (unsigned)((dout + span - 1) / span));
    apply_rows_kernel<<<grid, kApplyThreads, smem, s>>>(MT, din, dout, in, ldi, nv, out, ldo);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const tq_ctx* c, const void* x, int dtype, int64_t n, int64_t ld_x,
                            int H, int64_t cap, const int32_t* len, uint32_t* planes,
                            uint32_t* signs, uint16_t* norm, uint16_t* rnorm, cudaStream_t s) {
    if (n <= 0) return cudaSuccess;
    QuantArgs a;
    a.prm = c->prm;
    a.PiT = c->dPiT;
    a.StT = c->dStT;
    a.x = x;
    a.dtype = dtype;
    a.n = n;
    a.ld_x = ld_x;
    a.H = H;
    a.cap = cap;
    a.len = len;
    a.planes = planes;
    a.signs = signs;
    a.norm = norm;
    a.rnorm = rnorm;
    a.err = c->derr;
    // 16 rows per CTA once that fills the SMs twice over, else 4 (decode appends) with 1024
    // threads, which split every sum 8 ways: an append is a chain of dependent loads
    const bool bulk = n >= 2 * 148 * 16;
    const int rows = bulk ? 16 : 4;
    const int T = bulk ? kQuantThreads : kAppendThreads;
    const int S = quant_split(c->d, T), Sm = c->m ? quant_split(c->m, T) : 1;
    const int extra = std::max((S - 1) * (T / S), (Sm - 1) * (T / Sm));
    const size_t smem = (2ull * c->d + extra) * rows * sizeof(float);   // + the split partial sums
    const unsigned blocks = (unsigned)((n + rows - 1) / rows);
    auto run = [&](auto kernel, int threads) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        kernel<<<blocks, threads, smem, s>>>(a);
        return cudaGetLastError();
    };
    if (c->P > kFastBits)
        return bulk ? run(quantize_kernel<16, kQuantThreads, true>, kQuantThreads)
                    : run(quantize_kernel<4, kAppendThreads, true>, kAppendThreads);
    return bulk ? run(quantize_kernel<16, kQuantThreads, false>, kQuantThreads)
                : run(quantize_kernel<4, kAppendThreads, false>, kAppendThreads);
}

cudaError_t launch_advance_len(int32_t* len, int B, int64_t cap, int step, int* err, cudaStream_t s) {
    if (B <= 0) return cudaSuccess;
    advance_len_kernel<<<(B + 127) / 128, 128, 0, s>>>(len, B, cap, step, err);
    return cudaGetLastError();
}

}  // namespace tq
