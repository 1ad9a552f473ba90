// Attention logits on tensor cores for 96 < d <= 128 and m <= 128 (the head dimension of the
// decode workloads): mma.sync m16n8k32 with e4m3 operands and fp32 accumulation.
//
// Why tensor cores: scoring the 4 query heads of a GQA group needs 2 x 4 x 128 multiply-adds
// per key (MSE part and QJL part), about 15 flop per byte of packed key; on CUDA cores the
// table-lookup form of lut.cuh is bound by shared-memory lookups near 30 % of HBM bandwidth.
// The same masked sums are a small dense contraction: A = the key's bit planes (16 keys x K
// bits, each bit exactly 0 or 2^-6 in e4m3), B = the queries (K x 8 columns).
//
// Walsh form (host_setup.cpp): <Pi q, c[idx]> = c0 sum_j q'_j + sum_t kappa_t M_t, M_t the sum
// of q' over the bits of the XOR of the planes in term t; <S q, 2 sign - 1> = 2 M_u - sum_j u_j.
// The MSE columns stack the terms along K with kappa_t folded into B; the QJL columns use the
// sign bits against u.  B must be exact to ~16 bits while e4m3 keeps 4, so each query value is
// split into 4 e4m3 pieces x = b0 + b1/16 + b2/256 + b3/4096 (times a power-of-two column
// scale), one column per (head, piece): 16 MSE columns and 16 QJL columns.
//
// Fragment layout (m16n8k32, 8-bit types): thread (g = lane/4, t = lane%4) holds A rows g and
// g+8, k = 4t..4t+3 and 4t+16..4t+19; B column g, the same k; C rows g, g+8, columns 2t, 2t+1.
// Coordinates map to k so that thread t only needs word t of each bit plane: at k-step s,
// a0 byte i (k = 4t+i) is bit 2s+8i of the word and a2 byte i (k = 4t+16+i) is bit 2s+1+8i.
#include "mma_e4m3.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kThreads = 256;
// 16-key blocks per warp pass (the loads of all of them are in flight together)
template <int P> struct Unroll { static constexpr int n = P <= 2 ? 4 : 2; };

struct MmaArgs {
    Params prm;
    const float* qrot;
    const float* qproj;
    int B, Hq, Hkv, G;
    KeyCache k;
    float scale;
    float* logits;
    int* err;
};

template <int P>
struct Smem {
    static constexpr int T = 1 << (P - 1);   // Walsh terms
    float qv[4][128], uv[4][128];
    uint2 Bm[T * 4 * 2][32];                  // MSE fragments, index (t*4 + s)*2 + nb
    uint2 Bq[4 * 2][32];                      // QJL fragments, index s*2 + nb
    float fm[16], fq[16];                     // column factors 2^-e0 16^-pc, column = h*4 + pc
    float qsum[4], usum[4];
    float vmax[2][4];
};

// Stages the quad's queries and builds the fragments (every thread calls it; it synchronises).
template <int P>
__device__ void setup_group(Smem<P>& S, const MmaArgs& a, size_t qrow0, int nh) {
    constexpr int T = Smem<P>::T;
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    for (int e = threadIdx.x; e < 4 * 128; e += kThreads) {
        const int h = e >> 7, j = e & 127;
        S.qv[h][j] = (h < nh && j < prm.d) ? a.qrot[(qrow0 + h) * prm.d + j] : 0.f;
        S.uv[h][j] = (qjl && h < nh && j < prm.m) ? a.qproj[(qrow0 + h) * prm.m + j] : 0.f;
    }
    __syncthreads();
    // per head: sums and the largest scaled magnitude of each column family (warps 0-3 MSE, 4-7 QJL)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, h = warp & 3;
        float mx = 0.f, sum = 0.f;
        for (int j = lane; j < 128; j += 32) {
            if (warp < 4) {
                const float q = S.qv[h][j];
                sum += q;
#pragma unroll
                for (int t = 0; t < T; ++t) mx = fmaxf(mx, fabsf(prm.kappa[t] * q * 64.f));
            } else {
                const float u = S.uv[h][j];
                sum += u;
                mx = fmaxf(mx, fabsf(u * 64.f));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
            sum += __shfl_xor_sync(0xffffffffu, sum, o);
        }
        if (lane == 0) {
            S.vmax[warp >> 2][h] = mx;
            if (warp < 4) S.qsum[h] = sum; else S.usum[h] = sum;
        }
    }
    __syncthreads();
    // column exponents: e0 = 8 - E with max = f 2^E, f in [0.5, 1), so max 2^e0 in [128, 256)
    if (threadIdx.x < 32) {
        const int fam = threadIdx.x >> 4, col = threadIdx.x & 15, h = col >> 2, pc = col & 3;
        const float mx = S.vmax[fam][h];
        int E = 0;
        frexpf(mx, &E);
        const int e0 = mx > 0.f ? 8 - E : 0;
        const float f = ldexpf(1.f, -e0 - 4 * pc);
        if (fam == 0) S.fm[col] = f; else S.fq[col] = f;
    }
    __syncthreads();
    const int nm = T * 4 * 2, nq = qjl ? 4 * 2 : 0;
    for (int e = threadIdx.x; e < (nm + nq) * 32; e += kThreads) {
        const int mi = e >> 5, ln = e & 31, g = ln >> 2, tg = ln & 3;
        const bool isq = mi >= nm;
        const int li = isq ? mi - nm : mi;
        const int t = isq ? 0 : li >> 3, s = (li >> 1) & 3, nb = li & 1;
        const int col = nb * 8 + g, h = col >> 2, pc = col & 3;
        const float mx = S.vmax[isq ? 1 : 0][h];
        int E = 0;
        frexpf(mx, &E);
        const int e0 = mx > 0.f ? 8 - E : 0;
        uint32_t reg[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            uint32_t w = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 32 * tg + 2 * s + r + 8 * i;
                const float v = isq ? S.uv[h][j] * 64.f : prm.kappa[t] * S.qv[h][j] * 64.f;
                w |= piece(v, e0, pc) << (8 * i);
            }
            reg[r] = w;
        }
        if (isq) S.Bq[li][ln] = make_uint2(reg[0], reg[1]);
        else S.Bm[li][ln] = make_uint2(reg[0], reg[1]);
    }
    __syncthreads();
}

template <int P>
__global__ void __launch_bounds__(kThreads) logits_mma_kernel(const MmaArgs a) {
    constexpr int T = Smem<P>::T;
    constexpr int kUnroll = Unroll<P>::n;
    __shared__ Smem<P> S;
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int quads = (a.G + 3) / 4;
    const int ngroups = a.B * a.Hkv * quads;
    int64_t total = 0;
    for (int g = 0; g < ngroups; ++g) {
        int L = a.k.len[g / (a.Hkv * quads)];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        total += (L + 15) / 16;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0)
        for (int b = 0; b < a.B; ++b)
            if (a.k.len[b] < 0 || a.k.len[b] > a.k.cap) set_error(a.err, TQ_DEVERR_LEN_RANGE);
    const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = kThreads / 32;
    const int g8 = lane >> 2, tg = lane & 3;
    const int hsel = tg >> 1, pc0 = 2 * (tg & 1);
    const float c0 = prm.c0, kq = prm.qjl_scale;
    int64_t acc = 0;
    for (int g = 0; g < ngroups && acc < hi; ++g) {
        const int b = g / (a.Hkv * quads), kvh = (g / quads) % a.Hkv, quad = g % quads;
        int L = a.k.len[b];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        const int64_t nblk = (L + 15) / 16;
        const int64_t b0 = max(lo, acc) - acc, b1 = min(hi, acc + nblk) - acc;
        acc += nblk;
        if (b0 >= b1) continue;
        const int hbase = kvh * a.G + 4 * quad;
        const int nh = min(4, kvh * a.G + a.G - hbase);
        const size_t qrow0 = (size_t)b * a.Hq + hbase;
        __syncthreads();   // the previous group's fragments are no longer read
        setup_group<P>(S, a, qrow0, nh);
        // per-thread epilogue constants for its two heads (nb = 0, 1)
        float fm0[2], fm1[2], fq0[2], fq1[2], cq[2], cu[2];
#pragma unroll
        for (int nb = 0; nb < 2; ++nb) {
            const int h = nb * 2 + hsel;
            fm0[nb] = S.fm[h * 4 + pc0];
            fm1[nb] = S.fm[h * 4 + pc0 + 1];
            fq0[nb] = S.fq[h * 4 + pc0];
            fq1[nb] = S.fq[h * 4 + pc0 + 1];
            cq[nb] = c0 * S.qsum[h];
            cu[nb] = -kq * S.usum[h];
        }
        const size_t rowbase = ((size_t)b * a.Hkv + kvh) * a.k.cap;
        const size_t cap = a.k.cap;
        float* out = a.logits + qrow0 * cap;
        for (int64_t blk0 = b0 + (int64_t)warp * kUnroll; blk0 < b1; blk0 += (int64_t)nwarps * kUnroll) {
            uint32_t pw[kUnroll][2][P], sw[kUnroll][2];
            float nn[kUnroll][2], rr[kUnroll][2];
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
                for (int rsel = 0; rsel < 2; ++rsel) {
                    const int64_t key = (blk0 + u) * 16 + g8 + 8 * rsel;
                    const bool valid = (blk0 + u) < b1 && key < L;
                    const size_t row = rowbase + (valid ? key : 0);
#pragma unroll
                    for (int p = 0; p < P; ++p) pw[u][rsel][p] = valid ? __ldg(a.k.planes + row * (P * 4) + p * 4 + tg) : 0u;
                    nn[u][rsel] = valid ? half_bits_to_float(__ldg(a.k.norm + row)) : 0.f;
                    sw[u][rsel] = (qjl && valid) ? __ldg(a.k.signs + row * 4 + tg) : 0u;
                    rr[u][rsel] = (qjl && valid) ? half_bits_to_float(__ldg(a.k.rnorm + row)) : 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kUnroll; ++u) {
                if (blk0 + u >= b1) break;
                float am[2][4] = {}, aq[2][4] = {};
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    uint32_t xa = 0u, xb = 0u;
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        if ((odd_mask(t) >> p) & 1) {
                            xa ^= pw[u][0][p];
                            xb ^= pw[u][1][p];
                        }
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t a0 = ext(xa, 2 * s), a1 = ext(xb, 2 * s);
                        const uint32_t a2 = ext(xa, 2 * s + 1), a3 = ext(xb, 2 * s + 1);
                        mma_e4m3(am[0], a0, a1, a2, a3, S.Bm[(t * 4 + s) * 2 + 0][lane]);
                        mma_e4m3(am[1], a0, a1, a2, a3, S.Bm[(t * 4 + s) * 2 + 1][lane]);
                    }
                }
                if (qjl) {
#pragma unroll
                    for (int s = 0; s < 4; ++s) {
                        const uint32_t a0 = ext(sw[u][0], 2 * s), a1 = ext(sw[u][1], 2 * s);
                        const uint32_t a2 = ext(sw[u][0], 2 * s + 1), a3 = ext(sw[u][1], 2 * s + 1);
                        mma_e4m3(aq[0], a0, a1, a2, a3, S.Bq[s * 2 + 0][lane]);
                        mma_e4m3(aq[1], a0, a1, a2, a3, S.Bq[s * 2 + 1][lane]);
                    }
                }
#pragma unroll
                for (int nb = 0; nb < 2; ++nb) {
                    // rows g8 (key A) and g8 + 8 (key B); this thread holds 2 of the head's 4 pieces
                    float mA = fmaf(am[nb][0], fm0[nb], am[nb][1] * fm1[nb]);
                    float mB = fmaf(am[nb][2], fm0[nb], am[nb][3] * fm1[nb]);
                    float qA = fmaf(aq[nb][0], fq0[nb], aq[nb][1] * fq1[nb]);
                    float qB = fmaf(aq[nb][2], fq0[nb], aq[nb][3] * fq1[nb]);
                    mA += __shfl_xor_sync(0xffffffffu, mA, 1);
                    mB += __shfl_xor_sync(0xffffffffu, mB, 1);
                    qA += __shfl_xor_sync(0xffffffffu, qA, 1);
                    qB += __shfl_xor_sync(0xffffffffu, qB, 1);
                    const int h = nb * 2 + hsel;
                    const int rsel = tg & 1;   // even threads store key A, odd threads key B
                    const float m = rsel ? mB : mA, qv = rsel ? qB : qA;
                    const float n = rsel ? nn[u][1] : nn[u][0], rho = rsel ? rr[u][1] : rr[u][0];
                    float est = n * (cq[nb] + m);
                    if (qjl) est = fmaf(rho, fmaf(2.f * kq, qv, cu[nb]), est);
                    const int64_t key = (blk0 + u) * 16 + g8 + 8 * rsel;
                    if (key < L && h < nh) out[h * cap + key] = a.scale * est;
                }
            }
        }
    }
}

template <int P>
cudaError_t run(const MmaArgs& a, cudaStream_t s) {
    static int grid = 0;
    if (!grid) {
        int sms = 148, per = 1, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, logits_mma_kernel<P>, kThreads, 0);
        grid = sms * (per > 0 ? per : 1);
    }
    logits_mma_kernel<P><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool logits_mma_supported(const tq_ctx* kc) {
    const Params& p = kc->prm;
    return p.W == 4 && (!p.qjl || p.Ws == 4) && p.odd_walsh && p.P >= 1 && p.P <= 3;
}

cudaError_t launch_logits_mma(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                              const KeyCache& k, float scale, float* logits, cudaStream_t s) {
    MmaArgs a{};
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
    switch (kc->prm.P) {
        case 1: return run<1>(a, s);
        case 2: return run<2>(a, s);
        case 3: return run<3>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
