// Attention over a compressed KV cache: logits (the operation the juejin.cn post, section
// 三, reports the blog timing on H100) and the softmax-weighted sum of values (keys and
// values are both cached and compressed: nonndazone.ru essay, section 2).
//
// Work split: one CTA per (sequence chunk, batch x KV head, quad of query heads); the GQA
// group's 4 query heads share every key load and every table lookup (lut.cuh).  The
// output kernel runs flash-decoding style: per chunk a running max, a running sum and the
// weighted value sum (in the value context's rotated basis), then one log-sum-exp combine
// per query head which also rotates back (o = Pi_v^T a, one d x d product per head).
#include <cfloat>

#include "lut.cuh"
#include "attn_q8.cuh"
#include "tq_kernels.h"
#include "values.cuh"

namespace tq {
namespace {

constexpr int kThreads = 512;
constexpr size_t kSmemLimit = 227 * 1024;

struct AttnArgs {
    Params prm;
    const float* qrot;
    const float* qproj;
    int B, Hq, Hkv, G;
    KeyCache k;
    float scale;
    int chunk, nchunk;
    int* err;
    float* logits;        // logits kernel
    // output kernel
    int vmode;            // 0: bf16 values, 1: MSE codes
    Params vprm;
    const void* values;
    const uint16_t* vnorm;
    float* partials;      // [(b*Hq + h)*nchunk + c][2 + d]
};

template <int W, int P>
__global__ void __launch_bounds__(kThreads) logits_kernel(const AttnArgs a) {
    extern __shared__ float4 sm[];
    const Params& prm = a.prm;
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.k.len, b, a.k.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * a.chunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    Scorer<W, P> sc;
    sc.setup(sm, prm, a.qrot, a.qproj, (size_t)b * a.Hq + hbase, nh);
    const int64_t iend = min((int64_t)L, i0 + a.chunk);
    const size_t rowbase = (size_t)bh * a.k.cap;
    const size_t cap = a.k.cap;
    float* out = a.logits + ((size_t)b * a.Hq + hbase) * cap;
    for (int64_t i = i0 + threadIdx.x; i < iend; i += blockDim.x) {
        const float4 e = sc(prm, a.k.planes, a.k.signs, a.k.norm, a.k.rnorm, rowbase + i);
        out[i] = a.scale * e.x;
        if (nh > 1) out[cap + i] = a.scale * e.y;
        if (nh > 2) out[2 * cap + i] = a.scale * e.z;
        if (nh > 3) out[3 * cap + i] = a.scale * e.w;
    }
}

// ---------------------------------------------------------------------------------------
// Logits at W == 4 (96 < d <= 128, m <= 128), thread per key, without bank conflicts.
// The byte tables of lut.cuh are stored as T[v][k] (entry v of group k at v * 16 + k, 16 groups
// of 8 bits).  At step j a thread looks up group k = (j + r) mod 16, r = lane mod 8, so the 8
// lanes of each quarter-warp always hit 8 different bank slots (k mod 8) whatever their byte
// values.  To keep the byte positions static, each thread first rotates its 128-bit code
// vectors right by r bytes.  Arithmetic on the 4 query heads runs as packed fp32 pairs.
//
// Scheduling is persistent: one CTA per SM walks a contiguous share of all (batch, KV head,
// head quad) groups' keys, rebuilding the tables only when the group changes.
// 512 threads with two keys each per pass.  768 or 1024 threads with one key each (more warps
// to hide the lookup latency) run no faster: the shared-memory pipe is what bounds the kernel.
constexpr int kQ8Threads = 512;
constexpr int kQ8Keys = 2;

template <int P>
__global__ void __launch_bounds__(kQ8Threads, 1) logits_q8_kernel(const AttnArgs a) {
    extern __shared__ float4 sm[];
    const Params& prm = a.prm;
    float4* Tq = sm;
    float4* Tu = sm + 4096;
    float* qs = reinterpret_cast<float*>(sm + 8192);
    float* us = qs + 4 * 128;
    __shared__ float4 s_sum[2];
    const bool qjl = prm.qjl != 0;
    const int quads = (a.G + 3) / 4;
    const int ngroups = a.B * a.Hkv * quads;
    // keys of all groups in blocks of 32, split evenly across the CTAs
    int64_t total = 0;
    for (int g = 0; g < ngroups; ++g) {
        const int b = g / (a.Hkv * quads);
        int L = a.k.len[b];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        total += (L + 31) / 32;
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        for (int b = 0; b < a.B; ++b)
            if (a.k.len[b] < 0 || a.k.len[b] > a.k.cap) set_error(a.err, TQ_DEVERR_LEN_RANGE);
    }
    const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x;
    float kap[OddMasks<P>::n];
#pragma unroll
    for (int t = 0; t < OddMasks<P>::n; ++t) kap[t] = prm.kappa[t];
    const int r = threadIdx.x & 7;
    int64_t acc = 0;
    for (int g = 0; g < ngroups && acc < hi; ++g) {
        const int b = g / (a.Hkv * quads), kvh = (g / quads) % a.Hkv, quad = g % quads;
        int L = a.k.len[b];
        L = L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
        const int64_t nblk = (L + 31) / 32;
        const int64_t b0 = max(lo, acc) - acc, b1 = min(hi, acc + nblk) - acc;
        acc += nblk;
        if (b0 >= b1) continue;
        const int hbase = kvh * a.G + 4 * quad;
        const int nh = min(4, kvh * a.G + a.G - hbase);
        const size_t qrow0 = (size_t)b * a.Hq + hbase;
        __syncthreads();   // the previous group's tables are no longer read
        stage_quad(qs, 128, a.qrot + qrow0 * prm.d, prm.d, 0, nh, prm.d);
        if (qjl) stage_quad(us, 128, a.qproj + qrow0 * prm.m, prm.m, 0, nh, prm.m);
        __syncthreads();
        build_tables_vk(Tq, qs, 128);
        if (qjl) build_tables_vk(Tu, us, 128);
        if (threadIdx.x == 0) {
            float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), su = sq;
            for (int k = 0; k < 16; ++k) {
                sq = f4_add(sq, Tq[255 * 16 + k]);
                if (qjl) su = f4_add(su, Tu[255 * 16 + k]);
            }
            s_sum[0] = sq;
            s_sum[1] = su;
        }
        __syncthreads();
        const float4 qsum = s_sum[0], usum = s_sum[1];
        const float kq = prm.qjl_scale, c0 = prm.c0;
        const float4 cq = f4_scale(c0, qsum), cu = f4_scale(-kq, usum);
        const size_t rowbase = ((size_t)b * a.Hkv + kvh) * a.k.cap;
        const size_t cap = a.k.cap;
        float* out = a.logits + qrow0 * cap;
        const int64_t kend = min((int64_t)L, b1 * 32);
        for (int64_t k0 = b0 * 32 + threadIdx.x; k0 < kend; k0 += kQ8Keys * kQ8Threads) {
            // kQ8Keys keys per thread per pass: their loads are in flight before any is scored
            int64_t kk[kQ8Keys];
#pragma unroll
            for (int u = 0; u < kQ8Keys; ++u) kk[u] = k0 + (int64_t)u * kQ8Threads;
            uint32_t pl[kQ8Keys][P][4], sg[kQ8Keys][4];
            float n[kQ8Keys], rho[kQ8Keys];
#pragma unroll
            for (int u = 0; u < kQ8Keys; ++u) {
                const bool valid = kk[u] < kend;
                const size_t row = rowbase + (valid ? kk[u] : 0);
                const uint4* pr = reinterpret_cast<const uint4*>(a.k.planes + row * (P * 4));
#pragma unroll
                for (int p = 0; p < P; ++p) {
                    const uint4 v = valid ? __ldg(pr + p) : make_uint4(0u, 0u, 0u, 0u);
                    pl[u][p][0] = v.x; pl[u][p][1] = v.y; pl[u][p][2] = v.z; pl[u][p][3] = v.w;
                }
                n[u] = valid ? half_bits_to_float(__ldg(a.k.norm + row)) : 0.f;
                if (qjl && valid) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(a.k.signs + row * 4));
                    sg[u][0] = v.x; sg[u][1] = v.y; sg[u][2] = v.z; sg[u][3] = v.w;
                    rho[u] = half_bits_to_float(__ldg(a.k.rnorm + row));
                } else {
                    sg[u][0] = sg[u][1] = sg[u][2] = sg[u][3] = 0u;
                    rho[u] = 0.f;
                }
            }
#pragma unroll
            for (int u = 0; u < kQ8Keys; ++u) {
                if (kk[u] < kend) {
                    const float4 e = score_key<P>(Tq, Tu, pl[u], sg[u], n[u], rho[u], r, kap, cq, cu, 2.f * kq, qjl);
                    const int64_t key = kk[u];
                    out[key] = a.scale * e.x;
                    if (nh > 1) out[cap + key] = a.scale * e.y;
                    if (nh > 2) out[2 * cap + key] = a.scale * e.z;
                    if (nh > 3) out[3 * cap + key] = a.scale * e.w;
                }
            }
        }
    }
}

// Online softmax over one tile of keys and the weighted value sum, shared by the fused
// output kernel (logits from the scorer) and the values kernel (logits read from HBM).
// Every thread of the block calls it with its own key's logits l4 (-inf when it has none)
// and value norm vn; the warps then sweep the tile's keys with lanes owning coordinates.
template <int C, bool CODED, bool NIB, int NT>
__device__ __forceinline__ void softmax_tile(float4 l4, float vn, int ntile, size_t row0, const ValueSrc& v,
                                             float4* sW, float4* sRed, float4& s_m, float4& s_l, float4& s_alpha,
                                             const float* cv, float4 (&acc)[C]) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int NW = NT / 32;
    const float4 wm = warp_max4(l4);
    if (lane == 0) sRed[warp] = wm;
    __syncthreads();
    if (threadIdx.x == 0) {
        float4 mx = sRed[0];
        for (int w = 1; w < NW; ++w) mx = f4_max(mx, sRed[w]);
        const float4 mo = s_m;
        const float4 mn = f4_max(mo, mx);
        s_alpha = make_float4(rescale(mo.x, mn.x), rescale(mo.y, mn.y), rescale(mo.z, mn.z), rescale(mo.w, mn.w));
        s_m = mn;
    }
    __syncthreads();
    const float4 mn = s_m, alpha = s_alpha;
    const float4 p = make_float4(safe_exp(l4.x, mn.x), safe_exp(l4.y, mn.y), safe_exp(l4.z, mn.z),
                                 safe_exp(l4.w, mn.w));
    sW[threadIdx.x] = f4_scale(vn, p);
    const float4 ps = warp_sum4(p);
    __syncthreads();   // everyone has read sRed (the max) and written sW
    if (lane == 0) sRed[warp] = ps;
    __syncthreads();
    if (threadIdx.x == 0) {
        float4 sum = sRed[0];
        for (int w = 1; w < NW; ++w) sum = f4_add(sum, sRed[w]);
        const float4 lo = s_l;
        s_l = make_float4(fmaf(lo.x, alpha.x, sum.x), fmaf(lo.y, alpha.y, sum.y), fmaf(lo.z, alpha.z, sum.z),
                          fmaf(lo.w, alpha.w, sum.w));
    }
#pragma unroll
    for (int c = 0; c < C; ++c)
        acc[c] = make_float4(acc[c].x * alpha.x, acc[c].y * alpha.y, acc[c].z * alpha.z, acc[c].w * alpha.w);
    for (int t = warp; t < ntile; t += NW) accumulate_key<C, CODED, NIB>(acc, v, row0 + t, sW[t], cv, lane);
    __syncthreads();   // sW and sRed are rewritten by the next tile
}

// Sums the warps' accumulators (through shared memory at red, NW * 32 * C float4) and writes
// this chunk's partial state (max, sum, acc[d]) for the nh heads of the quad.
template <int C, bool NIB, int NT>
__device__ __forceinline__ void write_partial(const float4 (&acc)[C], float4* red, const float4& s_m,
                                              const float4& s_l, float* pbase, size_t hstride, int nh, int d) {
    constexpr int NW = NT / 32;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int c = 0; c < C; ++c) red[(warp * C + c) * 32 + lane] = acc[c];
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * C; e += NT) {
        const int c = e / 32, l = e % 32;
        float4 s = red[c * 32 + l];
        for (int w = 1; w < NW; ++w) s = f4_add(s, red[(w * C + c) * 32 + l]);
        const int j = owned_coord<NIB>(l, c);
        if (j < d) {
            const float vv[4] = {s.x, s.y, s.z, s.w};
            for (int h = 0; h < nh; ++h) pbase[h * hstride + 2 + j] = vv[h];
        }
    }
    if (threadIdx.x == 0) {
        const float mv[4] = {s_m.x, s_m.y, s_m.z, s_m.w}, lv[4] = {s_l.x, s_l.y, s_l.z, s_l.w};
        for (int h = 0; h < nh; ++h) {
            pbase[h * hstride] = mv[h];
            pbase[h * hstride + 1] = lv[h];
        }
    }
}

// Fused output: logits from the key codes (scorer), then softmax_tile.  C = ceil(d/32)
// coordinates per lane (nibble layout when NIB); d <= 32 * C.
template <int W, int P, int C, bool CODED, bool NIB>
__global__ void __launch_bounds__(kThreads) attn_partial_kernel(const AttnArgs a) {
    extern __shared__ float4 sm[];
    const Params& prm = a.prm;
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.k.len, b, a.k.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * a.chunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);

    Scorer<W, P> sc;
    sc.setup(sm, prm, a.qrot, a.qproj, (size_t)b * a.Hq + hbase, nh);
    float4* sW = sm + Scorer<W, P>::smem_bytes(prm) / sizeof(float4);   // [kThreads]
    float4* sRed = sW + kThreads;                                        // [kThreads / 32]
    __shared__ float4 s_m, s_l, s_alpha;
    __shared__ float s_cv[kMaxCodeLevels];   // the value table (coded values; any MSE width)
    if (threadIdx.x == 0) {
        s_m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        s_l = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k = threadIdx.x; k < a.vprm.L; k += blockDim.x) s_cv[k] = a.vprm.tab[k];
    const ValueSrc v{a.values, a.vnorm, a.vprm.P, a.vprm.W, prm.d};
    float4 acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t iend = min((int64_t)L, i0 + a.chunk);
    const size_t rowbase = (size_t)bh * a.k.cap;
    __syncthreads();
    for (int64_t t0 = i0; t0 < iend; t0 += kThreads) {
        const int ntile = (int)min((int64_t)kThreads, iend - t0);
        float4 l4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        float vn = 0.f;
        if ((int)threadIdx.x < ntile) {
            const float4 e = sc(prm, a.k.planes, a.k.signs, a.k.norm, a.k.rnorm, rowbase + t0 + threadIdx.x);
            l4.x = a.scale * e.x;
            if (nh > 1) l4.y = a.scale * e.y;
            if (nh > 2) l4.z = a.scale * e.z;
            if (nh > 3) l4.w = a.scale * e.w;
            vn = CODED ? half_bits_to_float(__ldg(a.vnorm + rowbase + t0 + threadIdx.x)) : 1.f;
        }
        softmax_tile<C, CODED, NIB, kThreads>(l4, vn, ntile, rowbase + t0, v, sW, sRed, s_m, s_l, s_alpha, s_cv, acc);
    }
    const size_t stride = (size_t)prm.d + 2;
    float* pbase = a.partials + (((size_t)b * a.Hq + hbase) * a.nchunk + blockIdx.x) * stride;
    write_partial<C, NIB, kThreads>(acc, sm, s_m, s_l, pbase, (size_t)a.nchunk * stride, nh, prm.d);
}

// Softmax + value sum from logits already in HBM ([B][Hq][cap], scaled).
constexpr int kValThreads = 256;

struct ValuesArgs {
    const float* logits;
    int B, Hq, Hkv, G, d;
    int64_t cap;
    const int32_t* len;
    int chunk, nchunk;
    int* err;
    Params vprm;          // centroids of the value context (coded values)
    ValueSrc v;
    float* partials;
};

template <int C, bool CODED, bool NIB>
__global__ void __launch_bounds__(kValThreads) values_kernel(const ValuesArgs a) {
    __shared__ float4 sW[kValThreads];
    __shared__ float4 sRed[kValThreads / 32];
    extern __shared__ float4 red[];   // [kValThreads / 32][C][32]
    __shared__ float4 s_m, s_l, s_alpha;
    __shared__ float s_cv[kMaxCodeLevels];   // the value table (coded values; any MSE width)
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.len, b, a.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * a.chunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    if (threadIdx.x == 0) {
        s_m = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        s_l = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int k = threadIdx.x; k < a.vprm.L; k += blockDim.x) s_cv[k] = a.vprm.tab[k];
    float4 acc[C];
#pragma unroll
    for (int c = 0; c < C; ++c) acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
    const int64_t iend = min((int64_t)L, i0 + a.chunk);
    const size_t rowbase = (size_t)bh * a.cap;
    const float* lg = a.logits + ((size_t)b * a.Hq + hbase) * a.cap;
    __syncthreads();
    for (int64_t t0 = i0; t0 < iend; t0 += kValThreads) {
        const int ntile = (int)min((int64_t)kValThreads, iend - t0);
        float4 l4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        float vn = 0.f;
        const int64_t i = t0 + threadIdx.x;
        if ((int)threadIdx.x < ntile) {
            l4.x = __ldg(lg + i);
            if (nh > 1) l4.y = __ldg(lg + a.cap + i);
            if (nh > 2) l4.z = __ldg(lg + 2 * a.cap + i);
            if (nh > 3) l4.w = __ldg(lg + 3 * a.cap + i);
            vn = CODED ? half_bits_to_float(__ldg(a.v.norm + rowbase + i)) : 1.f;
        }
        softmax_tile<C, CODED, NIB, kValThreads>(l4, vn, ntile, rowbase + t0, a.v, sW, sRed, s_m, s_l, s_alpha, s_cv,
                                                 acc);
    }
    const size_t stride = (size_t)a.d + 2;
    float* pbase = a.partials + (((size_t)b * a.Hq + hbase) * a.nchunk + blockIdx.x) * stride;
    write_partial<C, NIB, kValThreads>(acc, red, s_m, s_l, pbase, (size_t)a.nchunk * stride, nh, a.d);
}

// o = Pi_v^T orot (orot in shared memory, d values followed by room for the split sums), or a copy
// when Pi_v is NULL (bf16 values: no rotation).  Each output's sum over j is split between
// S = blockDim / span threads, loads issued 16 at a time (the values pass has usually evicted Pi_v
// from L2).  Every thread of the block calls it after orot is written and visible.
__device__ void back_rotate_store(float* orot, int d, const float* __restrict__ PiV, float* __restrict__ o) {
    if (!PiV) {
        for (int i = threadIdx.x; i < d; i += blockDim.x) o[i] = orot[i];
        return;
    }
    const int span = d < (int)blockDim.x ? ((d + 31) / 32) * 32 : (int)blockDim.x;
    const int S = blockDim.x / span, part = threadIdx.x / span, ii = threadIdx.x - part * span;
    const bool active = part < S;   // blockDim need not be a multiple of span
    float* red = orot + d;   // [S - 1][span]
    const int j0 = part * d / S, j1 = (part + 1) * d / S;
    for (int i0 = 0; i0 < d; i0 += span) {   // one pass when S > 1
        const int i = i0 + ii;
        float acc = 0.f;
        if (active && i < d) {
            for (int jb = j0; jb < j1; jb += 16) {
                float pv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) pv[u] = jb + u < j1 ? __ldg(PiV + (size_t)(jb + u) * d + i) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    if (jb + u < j1) acc = fmaf(pv[u], orot[jb + u], acc);
            }
        }
        if (S > 1) {
            if (active && part > 0 && i < d) red[(part - 1) * span + ii] = acc;
            __syncthreads();
            if (part == 0 && i < d)
                for (int q = 1; q < S; ++q) acc += red[(q - 1) * span + ii];
        }
        if (part == 0 && i < d) o[i] = acc;
    }
}

// out[b][h] = Pi_v^T (sum_c e^{m_c - M} a_c) / (sum_c e^{m_c - M} l_c) over the chunks that
// hold keys; Pi_v NULL for bf16 values (no rotation).
__global__ void attn_combine_kernel(const float* __restrict__ partials, int nchunk, int chunk, int d,
                                    int Hq, const int32_t* len, int64_t cap, const float* PiV,
                                    float* __restrict__ out) {
    extern __shared__ float orot[];
    const int bh = blockIdx.x, b = bh / Hq;
    int L = len[b];
    L = L < 0 ? 0 : (L > cap ? (int)cap : L);
    const int nc = (L + chunk - 1) / chunk;
    float* o = out + (size_t)bh * d;
    if (nc == 0) {
        for (int i = threadIdx.x; i < d; i += blockDim.x) o[i] = 0.f;
        return;
    }
    const size_t stride = (size_t)d + 2;
    const float* p = partials + (size_t)bh * nchunk * stride;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, p[c * stride]);
    float tot = 0.f;
    for (int c = 0; c < nc; ++c) tot += p[c * stride + 1] * rescale(p[c * stride], M);
    const float inv = 1.f / tot;
    for (int j = threadIdx.x; j < d; j += blockDim.x) {
        float s = 0.f;
        for (int c = 0; c < nc; ++c) s = fmaf(p[c * stride + 2 + j], rescale(p[c * stride], M), s);
        orot[j] = s * inv;
    }
    __syncthreads();
    back_rotate_store(orot, d, PiV, o);
}

// The state of a whole (batch, query head) over this call's keys, for a merge with other shards
// of the sequence: part[bh] = (M, sum_c e^{m_c - M} l_c, sum_c e^{m_c - M} a_c[0..d)) over the chunks
// that hold keys, unnormalised and in the value context's rotated basis; (-inf, 0, 0...) when the
// sequence holds no keys here.
__global__ void chunks_to_partial_kernel(const float* __restrict__ partials, int nchunk, int chunk, int d, int Hq,
                                         const int32_t* len, int64_t cap, float* __restrict__ part) {
    const int bh = blockIdx.x, b = bh / Hq;
    int L = len[b];
    L = L < 0 ? 0 : (L > cap ? (int)cap : L);
    const int nc = (L + chunk - 1) / chunk;
    const size_t stride = (size_t)d + 2;
    float* o = part + (size_t)bh * stride;
    const float* p = partials + (size_t)bh * nchunk * stride;
    float M = -INFINITY;
    for (int c = 0; c < nc; ++c) M = fmaxf(M, p[c * stride]);
    float tot = 0.f;
    for (int c = 0; c < nc; ++c) tot += p[c * stride + 1] * rescale(p[c * stride], M);
    if (threadIdx.x == 0) {
        o[0] = M;
        o[1] = tot;
    }
    for (int j = threadIdx.x; j < d; j += blockDim.x) {
        float s = 0.f;
        for (int c = 0; c < nc; ++c) s = fmaf(p[c * stride + 2 + j], rescale(p[c * stride], M), s);
        o[2 + j] = s;
    }
}

// out[bh] = Pi_v^T (sum_r e^{m_r - M} a_r) / (sum_r e^{m_r - M} l_r) over R shards' partial states
// parts[r][bh] = (m_r, l_r, a_r[0..d)); zeros when every shard is empty (all l_r = 0).
__global__ void merge_partials_kernel(const float* __restrict__ parts, int R, int64_t BH, int d, const float* PiV,
                                      float* __restrict__ out) {
    extern __shared__ float orot[];
    const int64_t bh = blockIdx.x;
    const size_t stride = (size_t)d + 2;
    float* o = out + (size_t)bh * d;
    float M = -INFINITY;
    for (int r = 0; r < R; ++r) M = fmaxf(M, parts[((size_t)r * BH + bh) * stride]);
    float tot = 0.f;
    for (int r = 0; r < R; ++r) {
        const float* p = parts + ((size_t)r * BH + bh) * stride;
        tot += p[1] * rescale(p[0], M);
    }
    if (!(tot > 0.f)) {
        for (int i = threadIdx.x; i < d; i += blockDim.x) o[i] = 0.f;
        return;
    }
    const float inv = 1.f / tot;
    for (int j = threadIdx.x; j < d; j += blockDim.x) {
        float acc = 0.f;
        for (int r = 0; r < R; ++r) {
            const float* p = parts + ((size_t)r * BH + bh) * stride;
            acc = fmaf(p[2 + j], rescale(p[0], M), acc);
        }
        orot[j] = acc * inv;
    }
    __syncthreads();
    back_rotate_store(orot, d, PiV, o);
}

template <typename K>
cudaError_t launch_with_smem(K kernel, dim3 grid, size_t smem, const AttnArgs& a, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kernel<<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

struct LogitsLaunch {
    template <int W, int P>
    static cudaError_t run(const AttnArgs& a, dim3 grid, cudaStream_t s) {
        const size_t smem = Scorer<W, P>::smem_bytes(a.prm);
        return launch_with_smem(logits_kernel<W, P>, grid, smem, a, s);
    }
};

// Coordinates per lane for the value sum: C = W on the table path (d <= 224); 16 on the
// generic path (d <= 512).  The nibble layout serves W == 4.
template <int W, int P, bool CODED>
cudaError_t run_output(const AttnArgs& a, dim3 grid, cudaStream_t s) {
    constexpr int C = W > 0 ? W : 16;
    const size_t scorer = Scorer<W, P>::smem_bytes(a.prm) + (kThreads + kThreads / 32) * sizeof(float4);
    const size_t red = (size_t)(kThreads / 32) * 32 * C * sizeof(float4);
    const size_t smem = scorer > red ? scorer : red;
    const bool nib = (W == 4) && (CODED || a.prm.d == 128);
    if (nib) return launch_with_smem(attn_partial_kernel<W, P, C, CODED, (W == 4)>, grid, smem, a, s);
    return launch_with_smem(attn_partial_kernel<W, P, C, CODED, false>, grid, smem, a, s);
}

struct OutputLaunch {
    template <int W, int P>
    static cudaError_t run(const AttnArgs& a, dim3 grid, cudaStream_t s) {
        if (a.vmode) return run_output<W, P, true>(a, grid, s);
        return run_output<W, P, false>(a, grid, s);
    }
};

template <class Op>
cudaError_t dispatch(const AttnArgs& a, bool lut, dim3 grid, cudaStream_t s) {
    if (!lut) return Op::template run<0, 0>(a, grid, s);
#define TQ_CASE_P(WV)                                                  \
    switch (a.prm.P) {                                                 \
        case 1: return Op::template run<WV, 1>(a, grid, s);            \
        case 2: return Op::template run<WV, 2>(a, grid, s);            \
        case 3: return Op::template run<WV, 3>(a, grid, s);            \
        case 4: return Op::template run<WV, 4>(a, grid, s);            \
    }                                                                  \
    break;
    switch (a.prm.W) {
        case 1: TQ_CASE_P(1)
        case 2: TQ_CASE_P(2)
        case 3: TQ_CASE_P(3)
        case 4: TQ_CASE_P(4)
        case 5: TQ_CASE_P(5)
        case 6: TQ_CASE_P(6)
        case 7: TQ_CASE_P(7)
    }
#undef TQ_CASE_P
    return cudaErrorInvalidValue;
}

AttnArgs make_args(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                   const KeyCache& k, float scale) {
    AttnArgs a{};
    a.prm = kc->prm;
    a.qrot = qrot;
    a.qproj = qproj;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.k = k;
    a.scale = scale;
    a.err = kc->derr;
    attn_chunking(kc, B, Hq, Hkv, k.cap, &a.chunk, &a.nchunk);
    return a;
}

// ---------------------------------------------------------------------------------------
// Tuned paths for W == 4 (96 < d <= 128), the head dimension of the decode workloads.

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
    const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }
__device__ __forceinline__ void cp_async_wait0() { asm volatile("cp.async.wait_group 0;\n" ::); }

// Threads per CTA of the coded-value kernel below (8 warps).
constexpr int kV2Threads = 256;

// Coded values at d <= 128 as independent per-warp streams: warp w takes the 32-key blocks w,
// w + 8, ... of the CTA's chunk, double-buffers their value rows with cp.async, keeps its own
// online softmax (running max per head, per-lane partial sums, accumulators rescaled when the
// max grows) and meets the other warps only once, at the end of the chunk (log-sum-exp merge of
// the 8 warp partials).  Lane l owns the coordinates 32 (l / 8) + l % 8 + 8 c, c = 0..3: bits
// l % 8 + 8 c of word l / 8 of each plane, so one rotate and one and-or per plane leave byte c of
// z = 4 * index of coordinate c, and a byte-permute plus one 4-byte shared load fetch its
// centroid.  The packed FFMA2 runs over the head pairs (0, 1) and (2, 3) against the centroid
// doubled in registers, so a key's four weights are one 16-byte broadcast load.  What bounds this
// loop is the shared-memory data return (lanes x bytes per load): per key 12 B of plane words,
// 16 B of centroids and 16 B of weights per lane.
template <int P, bool SPLIT>
__global__ void __launch_bounds__(kV2Threads, 4) values_coded128_kernel(const ValuesArgs a) {
    constexpr int NW = kV2Threads / 32;
    constexpr int ROW = P * 4;                  // words per value row (split rows: row_words)
    constexpr int BUFW = 32 * (SPLIT ? ROW + 4 : ROW);   // words per 32-key buffer
    constexpr int SVW = NW * 2 * BUFW > 4 * NW * 32 * 4 ? NW * 2 * BUFW : 4 * NW * 32 * 4;   // + room for the merge
    __shared__ __align__(16) uint32_t sV[SVW];
    __shared__ ulonglong2 sW[NW][32];           // per key: (w0, w1), (w2, w3)
    __shared__ float4 s_wm[NW], s_wl[NW];
    __shared__ float s_cv[kMaxLevels], s_cv_hi[kMaxLevels];
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.len, b, a.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * a.chunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < kMaxLevels) s_cv[threadIdx.x] = a.vprm.centroids[threadIdx.x];
    if (SPLIT && threadIdx.x < kMaxLevels) s_cv_hi[threadIdx.x] = a.vprm.centroids_hi[threadIdx.x];
    __syncthreads();
    // split rows: P full planes, then the top plane of the first d_hi coordinates (W_hi words)
    const int rw = SPLIT ? a.vprm.row_words : ROW;
    const int64_t iend = min((int64_t)L, i0 + a.chunk);
    const int nblk = (int)((iend - i0 + 31) / 32);
    const size_t rowbase = (size_t)bh * a.cap;
    const float* lg = a.logits + ((size_t)b * a.Hq + hbase) * a.cap;
    const uint32_t* vrows = static_cast<const uint32_t*>(a.v.values);
    uint32_t* buf0 = sV + warp * 2 * BUFW;

    auto issue_block = [&](int j, int buf) {   // the value rows of block j into buffer buf
        const int64_t k0 = i0 + (int64_t)j * 32;
        const int n = (int)min((int64_t)32, iend - k0);
        if constexpr (SPLIT) {   // rows of row_words words need not start on 16 bytes
            const uint32_t* src = vrows + (rowbase + k0) * rw;
            uint32_t* dst = buf0 + buf * BUFW;
            for (int e = lane; e < n * rw; e += 32) cp_async4(dst + e, src + e);
        } else {
            const uint4* src = reinterpret_cast<const uint4*>(vrows + (rowbase + k0) * ROW);
            uint4* dst = reinterpret_cast<uint4*>(buf0 + buf * BUFW);
            for (int e = lane; e < n * P; e += 32) cp_async16(dst + e, src + e);
        }
    };
    auto load_logits = [&](int j, float4& l4, float& vn) {   // key k0 + lane of block j
        const int64_t i = i0 + (int64_t)j * 32 + lane;
        l4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        vn = 0.f;
        if (j < nblk && i < iend) {
            l4.x = __ldg(lg + i);
            if (nh > 1) l4.y = __ldg(lg + a.cap + i);
            if (nh > 2) l4.z = __ldg(lg + 2 * a.cap + i);
            if (nh > 3) l4.w = __ldg(lg + 3 * a.cap + i);
            vn = half_bits_to_float(__ldg(a.v.norm + rowbase + i));
        }
    };

    u64 acc[4][2];   // owned coordinate c: heads (0, 1) in acc[c][0], (2, 3) in acc[c][1]
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0ull;
    float4 m4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 ls = make_float4(0.f, 0.f, 0.f, 0.f);   // this lane's share of the softmax sums
    float4 l4, nl4;
    float vn, nvn;
    load_logits(warp, l4, vn);
    if (warp < nblk) issue_block(warp, 0);
    cp_async_commit();
    const int wsel = lane >> 3;
    int rot[P];   // right-rotation moving bit lane % 8 + 8 c of plane pp to bit 8 c + pp + 2
#pragma unroll
    for (int pp = 0; pp < P; ++pp) rot[pp] = ((lane & 7) - pp - 2) & 31;
    // split contexts: a lane's coordinates share word wsel, so the (P+1)-bit table is per lane
    const bool hi = SPLIT && 32 * wsel < a.vprm.d_hi;
    const int rot_top = ((lane & 7) - P - 2) & 31;
    const unsigned char* cvl = reinterpret_cast<const unsigned char*>(hi ? s_cv_hi : s_cv);
    const ulonglong2* sWw = sW[warp];
    int buf = 0;
    for (int j = warp; j < nblk; j += NW, buf ^= 1) {
        const int jn = j + NW;
        if (jn < nblk) issue_block(jn, buf ^ 1);
        cp_async_commit();
        load_logits(jn, nl4, nvn);
        // online softmax over this block (one key per lane)
        const float4 mn = f4_max(m4, warp_max4_redux(l4));
        if (mn.x != m4.x || mn.y != m4.y || mn.z != m4.z || mn.w != m4.w) {   // warp-uniform
            // the running max grew: rescale the sums and accumulators by exp(old - new)
            const float4 alpha = make_float4(rescale(m4.x, mn.x), rescale(m4.y, mn.y), rescale(m4.z, mn.z), rescale(m4.w, mn.w));
            m4 = mn;
            ls = make_float4(ls.x * alpha.x, ls.y * alpha.y, ls.z * alpha.z, ls.w * alpha.w);
            const u64 a01 = pk2(alpha.x, alpha.y), a23 = pk2(alpha.z, alpha.w);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[c][0] = mul2(acc[c][0], a01);
                acc[c][1] = mul2(acc[c][1], a23);
            }
        }
        const float4 p = make_float4(safe_exp(l4.x, m4.x), safe_exp(l4.y, m4.y), safe_exp(l4.z, m4.z), safe_exp(l4.w, m4.w));
        ls = f4_add(ls, p);
        {
            const float4 w = f4_scale(vn, p);
            sW[warp][lane] = make_ulonglong2(pk2(w.x, w.y), pk2(w.z, w.w));
        }
        cp_async_wait1();   // this block's value rows have landed
        __syncwarp();
        const uint32_t* tile = buf0 + buf * BUFW;
        // All 32 rows, also in a partial block: a key past the end has weight exactly 0 (vn = 0,
        // p = 0) and its stale row still selects finite centroids, so it adds nothing.
#pragma unroll 8
        for (int t = 0; t < 32; ++t) {
            const uint32_t* row = tile + t * (SPLIT ? rw : ROW);
            // byte c of z = 4 * index of owned coordinate c: the offset of its centroid
            uint32_t z = 0u;
#pragma unroll
            for (int pp = 0; pp < P; ++pp) {
                const uint32_t wd = row[pp * 4 + wsel];
                z |= __funnelshift_r(wd, wd, rot[pp]) & (0x04040404u << pp);
            }
            if (SPLIT && hi) {
                const uint32_t wd = row[P * 4 + wsel];
                z |= __funnelshift_r(wd, wd, rot_top) & (0x04040404u << P);
            }
            const ulonglong2 w = sWw[t];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                const float cv = *reinterpret_cast<const float*>(cvl + __byte_perm(z, 0u, 0x4440 + c));
                const u64 cc = pk2(cv, cv);
                acc[c][0] = fma2(cc, w.x, acc[c][0]);
                acc[c][1] = fma2(cc, w.y, acc[c][1]);
            }
        }
        __syncwarp();   // sW and this buffer are reused
        l4 = nl4;
        vn = nvn;
    }
    cp_async_wait0();
    // merge the warps: M = max of their maxima, each warp's share scaled by exp(m_w - M)
    ls = warp_sum4(ls);
    if (lane == 0) {
        s_wm[warp] = m4;
        s_wl[warp] = ls;
    }
    __syncthreads();   // every warp's cp.async and reads of sV are done; sV becomes the merge buffer
    float4 M = s_wm[0];
    for (int w = 1; w < NW; ++w) M = f4_max(M, s_wm[w]);
    const float4 sc = make_float4(rescale(m4.x, M.x), rescale(m4.y, M.y), rescale(m4.z, M.z), rescale(m4.w, M.w));
    float4* red = reinterpret_cast<float4*>(sV);   // [NW][4][32]
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 h01 = upk2(acc[c][0]), h23 = upk2(acc[c][1]);
        red[(warp * 4 + c) * 32 + lane] = make_float4(h01.x * sc.x, h01.y * sc.y, h23.x * sc.z, h23.y * sc.w);
    }
    __syncthreads();
    const size_t stride = (size_t)a.d + 2;
    const size_t hstride = (size_t)a.nchunk * stride;
    float* pbase = a.partials + (((size_t)b * a.Hq + hbase) * a.nchunk + blockIdx.x) * stride;
    if (threadIdx.x < 128) {
        const int c = threadIdx.x >> 5, l = threadIdx.x & 31, jc = 32 * (l >> 3) + (l & 7) + 8 * c;
        float4 sum = red[c * 32 + l];
        for (int w = 1; w < NW; ++w) sum = f4_add(sum, red[(w * 4 + c) * 32 + l]);
        if (jc < a.d) {
            const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
            for (int h = 0; h < nh; ++h) pbase[h * hstride + 2 + jc] = vv[h];
        }
    }
    if (threadIdx.x == 0) {
        float4 lt = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < NW; ++w) {
            const float4 mw = s_wm[w], lw = s_wl[w];
            lt.x = fmaf(lw.x, rescale(mw.x, M.x), lt.x);
            lt.y = fmaf(lw.y, rescale(mw.y, M.y), lt.y);
            lt.z = fmaf(lw.z, rescale(mw.z, M.z), lt.z);
            lt.w = fmaf(lw.w, rescale(mw.w, M.w), lt.w);
        }
        const float mv[4] = {M.x, M.y, M.z, M.w}, lv[4] = {lt.x, lt.y, lt.z, lt.w};
        for (int h = 0; h < nh; ++h) {
            pbase[h * hstride] = mv[h];
            pbase[h * hstride + 1] = lv[h];
        }
    }
}

template <int P>
cudaError_t run_values_coded128(const ValuesArgs& a, dim3 grid, cudaStream_t s) {
    if constexpr (P < kFastBits) {
        if (a.vprm.d_hi) {
            values_coded128_kernel<P, true><<<grid, kV2Threads, 0, s>>>(a);
            return cudaGetLastError();
        }
    }
    values_coded128_kernel<P, false><<<grid, kV2Threads, 0, s>>>(a);
    return cudaGetLastError();
}

template <int C, bool CODED, bool NIB>
cudaError_t run_values(const ValuesArgs& a, dim3 grid, cudaStream_t s) {
    const size_t smem = (size_t)(kValThreads / 32) * 32 * C * sizeof(float4);
    cudaError_t e = cudaFuncSetAttribute(values_kernel<C, CODED, NIB>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    values_kernel<C, CODED, NIB><<<grid, kValThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

void attn_chunking(const tq_ctx* kc, int B, int Hq, int Hkv, int64_t cap, int* chunk, int* nchunk) {
    // Aim for ~4 waves of one CTA per SM over all (batch, KV head, head quad) groups; at
    // least 4 tiles of keys per CTA so the table build is amortised.
    const int quads = (Hq / Hkv + 3) / 4;
    const int64_t groups = (int64_t)B * Hkv * quads;
    int64_t c = (groups * cap + 148 * 4 - 1) / (148 * 4);
    c = ((c + kThreads - 1) / kThreads) * kThreads;
    if (c < 4 * kThreads) c = 4 * kThreads;
    if (c > (1 << 20)) c = 1 << 20;
    *chunk = (int)c;
    *nchunk = (int)((cap + c - 1) / c);
    (void)kc;
}

template <int P>
cudaError_t run_logits_q8(const AttnArgs& a, dim3 grid, cudaStream_t s) {
    const size_t smem = 8192 * sizeof(float4) + 2 * 4 * 128 * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(logits_q8_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    logits_q8_kernel<P><<<grid, kQ8Threads, smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_logits(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq,
                          int Hkv, const KeyCache& k, float scale, float* logits, void* image, cudaStream_t s) {
    // AUTO takes the tensor-core kernel where it measured faster than the byte tables: keys of
    // 2 MSE bits + QJL (at 1 or 3 MSE bits, and below ~2^18 keys x head quads, the byte tables win)
    const int64_t quad_keys = (int64_t)B * Hkv * ((Hq / Hkv + 3) / 4) * k.cap;
    const bool tc_auto = kc->kernel_path == TQ_PATH_AUTO && kc->prm.qjl && kc->prm.P == 2 && quad_keys >= (1 << 18);
    if ((kc->kernel_path == TQ_PATH_TENSOR || tc_auto) && logits_tc_ok(kc, k))
        return launch_logits_tc(kc, qrot, qproj, B, Hq, Hkv, k, scale, logits, image, s);
    AttnArgs a = make_args(kc, qrot, qproj, B, Hq, Hkv, k, scale);
    a.logits = logits;
    if (a.prm.W == 4 && (!a.prm.qjl || a.prm.Ws == 4) && a.prm.odd_walsh) {
        static int sms = 0;
        if (!sms && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, kc->device) != cudaSuccess) sms = 148;
        dim3 grid(sms);
        switch (a.prm.P) {
            case 1: return run_logits_q8<1>(a, grid, s);
            case 2: return run_logits_q8<2>(a, grid, s);
            case 3: return run_logits_q8<3>(a, grid, s);
            case 4: return run_logits_q8<4>(a, grid, s);
        }
    }
    const bool lut = lut_path_ok(a.prm, 0, kSmemLimit);
    dim3 grid(a.nchunk, B * Hkv, (a.G + 3) / 4);
    return dispatch<LogitsLaunch>(a, lut, grid, s);
}

cudaError_t launch_attn_values(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                               const int32_t* len, const void* values, const uint16_t* vnorm, int* err,
                               float* partials, float* out, cudaStream_t s, float* part_out, bool allow_tc) {
    ValuesArgs a{};
    a.logits = logits;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.d = d;
    a.cap = cap;
    a.len = len;
    a.err = err;
    if (vc) a.vprm = vc->prm;
    a.v = ValueSrc{values, vnorm, vc ? vc->P : 0, vc ? vc->W : 0, d};
    a.partials = partials;
    attn_chunking(nullptr, B, Hq, Hkv, cap, &a.chunk, &a.nchunk);
    // the tensor-core kernel copies the norms as 4-byte pairs: an even capacity and a 4-byte
    // aligned norm array keep every pair aligned and inside its sequence's rows
    const bool tc = allow_tc && vc && vc->kernel_path == TQ_PATH_TENSOR && values_tc_supported(vc, d) &&
                    cap % 2 == 0 && (reinterpret_cast<uintptr_t>(vnorm) & 3u) == 0;
    if (tc) {
        a.chunk = values_tc_chunk(B, Hq, Hkv, cap);
        a.nchunk = (int)((cap + a.chunk - 1) / a.chunk);
    }
    dim3 grid(a.nchunk, B * Hkv, (a.G + 3) / 4);
    const int W = (d + 31) / 32;
    cudaError_t e;
    if (tc) {
        e = launch_values_tc(vc, d, logits, B, Hq, Hkv, cap, len, values, vnorm, err, partials, a.chunk, a.nchunk, s);
    } else if (vc && W == 4 && vc->P <= kFastBits) {
        switch (vc->P) {
            case 1: e = run_values_coded128<1>(a, grid, s); break;
            case 2: e = run_values_coded128<2>(a, grid, s); break;
            case 3: e = run_values_coded128<3>(a, grid, s); break;
            default: e = run_values_coded128<4>(a, grid, s); break;
        }
    }
    else if (!vc && d == 128) e = run_values<4, false, true>(a, grid, s);
    else if (W <= 8) e = vc ? run_values<8, true, false>(a, grid, s) : run_values<8, false, false>(a, grid, s);
    else e = vc ? run_values<16, true, false>(a, grid, s) : run_values<16, false, false>(a, grid, s);
    if (e != cudaSuccess) return e;
    if (part_out) {   // this call's shard of the sequence: per (batch, head) state, no normalisation
        const int pt = d >= 256 ? 256 : ((d + 31) / 32) * 32;
        chunks_to_partial_kernel<<<B * Hq, pt, 0, s>>>(partials, a.nchunk, a.chunk, d, Hq, len, cap, part_out);
        return cudaGetLastError();
    }
    // 512 threads: the back-rotation's sums split 4 ways at d <= 128 (2 at d <= 256)
    const int threads = vc ? 512 : (d >= 256 ? 256 : ((d + 31) / 32) * 32);
    const int span = d < threads ? ((d + 31) / 32) * 32 : threads;
    const size_t csmem = ((size_t)d + (size_t)(threads / span - 1) * span) * sizeof(float);
    attn_combine_kernel<<<B * Hq, threads, csmem, s>>>(partials, a.nchunk, a.chunk, d, Hq, len, cap,
                                                       vc ? vc->dPi : nullptr, out);
    return cudaGetLastError();
}

cudaError_t launch_merge_partials(const tq_ctx* vc, int d, const float* parts, int R, int64_t BH, float* out,
                                  cudaStream_t s) {
    if (BH <= 0) return cudaSuccess;
    const int threads = vc ? 512 : (d >= 256 ? 256 : ((d + 31) / 32) * 32);
    const int span = d < threads ? ((d + 31) / 32) * 32 : threads;
    const size_t smem = ((size_t)d + (size_t)(threads / span - 1) * span) * sizeof(float);
    merge_partials_kernel<<<(unsigned)BH, threads, smem, s>>>(parts, R, BH, d, vc ? vc->dPi : nullptr, out);
    return cudaGetLastError();
}

cudaError_t launch_attn_output(const tq_ctx* kc, const tq_ctx* vc, const float* qrot,
                               const float* qproj, int B, int Hq, int Hkv, const KeyCache& k,
                               float scale, const void* values, const uint16_t* vnorm,
                               float* partials, float* out, cudaStream_t s) {
    AttnArgs a = make_args(kc, qrot, qproj, B, Hq, Hkv, k, scale);
    a.vmode = vc ? 1 : 0;
    if (vc) a.vprm = vc->prm;
    a.values = values;
    a.vnorm = vnorm;
    a.partials = partials;
    const size_t extra = (kThreads + kThreads / 32) * sizeof(float4);
    const bool lut = lut_path_ok(a.prm, extra, kSmemLimit);
    dim3 grid(a.nchunk, B * Hkv, (a.G + 3) / 4);
    cudaError_t e = dispatch<OutputLaunch>(a, lut, grid, s);
    if (e != cudaSuccess) return e;
    const int d = kc->d;
    const int threads = d >= 256 ? 256 : ((d + 31) / 32) * 32;
    attn_combine_kernel<<<B * Hq, threads, d * sizeof(float), s>>>(partials, a.nchunk, a.chunk, d, Hq, k.len,
                                                                  k.cap, vc ? vc->dPi : nullptr, out);
    return cudaGetLastError();
}

}  // namespace tq
