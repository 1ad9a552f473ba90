// Top-k vector search over compressed vectors (juejin.cn post, section 三: GloVe d=200
// Recall@1@k; section 四: near-zero indexing time, i.e. coding is the only index build).
//
// Pass 1: one CTA per (database chunk, quad of queries).  Each thread scores one vector for
// the 4 queries with the shared byte tables (lut.cuh); a score that beats the query's
// current k-th best (score descending, equal scores by lower index) is appended to a
// shared candidate buffer, which is merged into the sorted top-k list whenever another
// tile could overflow it.  Scores never go to HBM.  Pass 2: one CTA per query sorts the
// per-chunk lists and keeps the first k.
#include "lut.cuh"
#include "mma_e4m3.cuh"
#include "search_topk.cuh"

namespace tq {
namespace {

constexpr int kThreads = 256;      // one tile = kThreads vectors
constexpr size_t kSmemLimit = 227 * 1024;
using SearchState = SearchStateT<4>;

template <int W, int P>
__global__ void __launch_bounds__(kThreads) search_chunk_kernel(const SearchArgs a) {
    extern __shared__ float4 sm[];
    const Params& prm = a.prm;
    const int64_t q0 = 4 * (int64_t)blockIdx.y;
    const int nh = (int)min((int64_t)4, a.nq - q0);
    const int64_t c0 = (int64_t)blockIdx.x * a.chunk;
    const int64_t cend = min(a.n, c0 + a.chunk);
    SearchState& st = *reinterpret_cast<SearchState*>(sm + Scorer<W, P>::smem_bytes(prm) / sizeof(float4));
    if (threadIdx.x < 4) {
        st.nb[threadIdx.x] = 0;
        st.cnt[threadIdx.x] = 0;
        st.ts[threadIdx.x] = -INFINITY;
        st.ti[threadIdx.x] = INT_MAX;
    }
    Scorer<W, P> sc;
    sc.setup(sm, prm, a.qrot, a.qproj, (size_t)q0, nh);   // synchronises
    const int lane = threadIdx.x & 31;
    for (int64_t t0 = c0; t0 < cend; t0 += kThreads) {
        const int64_t i = t0 + threadIdx.x;
        const bool valid = i < cend;
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid) {
            const float4 e = sc(prm, a.planes, a.signs, a.norm, a.rnorm, (size_t)i);
            sv[0] = e.x; sv[1] = e.y; sv[2] = e.z; sv[3] = e.w;
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const bool pass = valid && h < nh && better(sv[h], (int)i, st.ts[h], st.ti[h]);
            const unsigned bal = __ballot_sync(0xffffffffu, pass);
            if (bal) {
                int base = 0;
                if (lane == 0) base = atomicAdd(&st.cnt[h], __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                if (pass) {
                    const int pos = base + __popc(bal & ((1u << lane) - 1u));
                    st.cs[h][pos] = sv[h];
                    st.ci[h][pos] = (int)i;
                }
            }
        }
        __syncthreads();
        for (int h = 0; h < nh; ++h)
            if (st.cnt[h] > kCand - kThreads) merge_candidates<4, kThreads, 0>(st, h, a.k, threadIdx.x);
    }
    for (int h = 0; h < nh; ++h)
        if (st.cnt[h] > 0) merge_candidates<4, kThreads, 0>(st, h, a.k, threadIdx.x);
    for (int h = 0; h < nh; ++h) {
        const size_t base = ((size_t)(q0 + h) * a.nchunk + blockIdx.x) * a.k;
        for (int t = threadIdx.x; t < a.k; t += blockDim.x) {
            const bool ok = t < st.nb[h];
            a.cand_s[base + t] = ok ? st.bs[h][t] : -INFINITY;
            a.cand_i[base + t] = ok ? st.bi[h][t] : INT_MAX;
        }
    }
}

__global__ void __launch_bounds__(kThreads) search_merge_kernel(const float* __restrict__ cand_s,
                                                                const int* __restrict__ cand_i, int per_query,
                                                                int npow, int k, float* top_s, int32_t* top_i) {
    extern __shared__ float msm[];
    float* s = msm;
    int* id = reinterpret_cast<int*>(msm + npow);
    const size_t q = blockIdx.x;
    for (int t = threadIdx.x; t < npow; t += blockDim.x) {
        const bool ok = t < per_query;
        s[t] = ok ? cand_s[q * per_query + t] : -INFINITY;
        id[t] = ok ? cand_i[q * per_query + t] : INT_MAX;
    }
    __syncthreads();
    bitonic_sort<kThreads, 0>(s, id, npow, threadIdx.x);
    for (int t = threadIdx.x; t < k; t += blockDim.x) {
        top_s[q * k + t] = s[t];
        top_i[q * k + t] = id[t];
    }
}

// Per query: the R shards' k candidates each (rows shifted to global numbers by the shard's
// offset; INT_MAX marks padding and keeps a score of -inf), sorted best first, the first k kept.
__global__ void __launch_bounds__(kThreads) shard_topk_merge_kernel(const float* __restrict__ cand_s,
                                                                   const int32_t* __restrict__ cand_i, int R,
                                                                   int64_t nq, int k, int npow, const ShardOffsets offs,
                                                                   float* top_s, int32_t* top_i) {
    extern __shared__ float msm[];
    float* s = msm;
    int* id = reinterpret_cast<int*>(msm + npow);
    const size_t q = blockIdx.x;
    for (int t = threadIdx.x; t < npow; t += blockDim.x) {
        float sc = -INFINITY;
        int ix = INT_MAX;
        if (t < R * k) {
            const int r = t / k, j = t - r * k;
            const size_t at = ((size_t)r * nq + q) * k + j;
            const int32_t li = cand_i[at];
            if (li != INT_MAX) {
                sc = cand_s[at];
                ix = (int)(li + offs.off[r]);
            }
        }
        s[t] = sc;
        id[t] = ix;
    }
    __syncthreads();
    bitonic_sort<kThreads, 0>(s, id, npow, threadIdx.x);
    for (int t = threadIdx.x; t < k; t += blockDim.x) {
        top_s[q * k + t] = s[t];
        top_i[q * k + t] = id[t];
    }
}

// ---------------------------------------------------------------------------------------
// Tensor-core scoring (mma.sync m16n8k32, e4m3, fp32 accumulate) for d <= 256: a CTA takes 8
// queries and a database chunk, streamed in tiles of 128 vectors staged in shared memory.
// Each warp scores 16 vectors against the 8 queries: A = the vectors' bit planes (a k-step is
// one 32-bit word; thread t's bytes are bits 4t..4t+3 and 16+4t..16+4t+3, each 0 or 2^-6), B =
// the queries split into 4 e4m3 pieces (columns = query x piece).  The
// fp32 scores go straight into the per-query top-k of the CTA.
constexpr int kSQ = 8;         // queries per CTA
constexpr int kSTile = 128;    // vectors per tile (8 warps x 16)

template <int P, int W>
struct SMmaSmem {
    static constexpr int T = 1 << (P - 1);
    static constexpr int RW = (P * W) | 1;   // odd row strides: conflict-free row reads
    static constexpr int SW = W | 1;
    SearchStateT<kSQ> st;
    float qv[kSQ][W * 32], uv[kSQ][W * 32];
    uint2 Bm[T * W][4][32];
    uint2 Bq[W][4][32];
    float fm[32], fq[32], qsum[kSQ], usum[kSQ], vmax[2][kSQ];
    uint32_t tp[kSTile][RW];
    uint32_t tsg[kSTile][SW];
    float tn[kSTile], tr[kSTile];
};

template <int P, int W>
__global__ void __launch_bounds__(kThreads) search_mma_kernel(const SearchArgs a) {
    using Sm = SMmaSmem<P, W>;
    constexpr int T = Sm::T;
    extern __shared__ __align__(16) unsigned char smraw[];
    Sm& S = *reinterpret_cast<Sm*>(smraw);
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int64_t q0 = (int64_t)kSQ * blockIdx.y;
    const int nqt = (int)min((int64_t)kSQ, a.nq - q0);
    const int64_t c0 = (int64_t)blockIdx.x * a.chunk, cend = min(a.n, c0 + a.chunk);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (threadIdx.x < kSQ) {
        S.st.nb[threadIdx.x] = 0;
        S.st.cnt[threadIdx.x] = 0;
        S.st.ts[threadIdx.x] = -INFINITY;
        S.st.ti[threadIdx.x] = INT_MAX;
    }
    for (int e = threadIdx.x; e < kSQ * W * 32; e += kThreads) {
        const int ql = e / (W * 32), j = e - ql * (W * 32);
        S.qv[ql][j] = (ql < nqt && j < prm.d) ? a.qrot[(size_t)(q0 + ql) * prm.d + j] : 0.f;
        S.uv[ql][j] = (qjl && ql < nqt && j < prm.m) ? a.qproj[(size_t)(q0 + ql) * prm.m + j] : 0.f;
    }
    __syncthreads();
    {   // warp w: sums and largest scaled magnitudes of query w
        float mq = 0.f, mu = 0.f, sq = 0.f, su = 0.f;
        for (int j = lane; j < W * 32; j += 32) {
            const float q = S.qv[warp][j], u = S.uv[warp][j];
            sq += q;
            su += u;
#pragma unroll
            for (int t = 0; t < T; ++t) mq = fmaxf(mq, fabsf(prm.kappa[t] * q * 64.f));
            mu = fmaxf(mu, fabsf(u * 64.f));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
            mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
            sq += __shfl_xor_sync(0xffffffffu, sq, o);
            su += __shfl_xor_sync(0xffffffffu, su, o);
        }
        if (lane == 0) {
            S.vmax[0][warp] = mq;
            S.vmax[1][warp] = mu;
            S.qsum[warp] = sq;
            S.usum[warp] = su;
        }
    }
    __syncthreads();
    if (threadIdx.x < 64) {
        const int fam = threadIdx.x >> 5, col = threadIdx.x & 31, ql = col >> 2, pc = col & 3;
        const float f = ldexpf(1.f, -column_exponent(S.vmax[fam][ql]) - 4 * pc);
        if (fam == 0) S.fm[col] = f; else S.fq[col] = f;
    }
    const int nm = T * W * 4, nqf = qjl ? W * 4 : 0;
    for (int e = threadIdx.x; e < (nm + nqf) * 32; e += kThreads) {
        const int ln = e & 31, rest = e >> 5;
        const bool isq = rest >= nm;
        const int r2 = isq ? rest - nm : rest;
        const int nb = r2 & 3, ks = r2 >> 2;
        const int t = isq ? 0 : ks / W, sidx = isq ? ks : ks - (ks / W) * W;
        const int g = ln >> 2, tg = ln & 3, col = nb * 8 + g, ql = col >> 2, pc = col & 3;
        const int e0 = column_exponent(S.vmax[isq ? 1 : 0][ql]);
        uint32_t reg[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            uint32_t w = 0u;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 32 * sidx + 16 * r + 4 * tg + i;
                const float v = isq ? S.uv[ql][j] * 64.f : prm.kappa[t] * S.qv[ql][j] * 64.f;
                w |= piece(v, e0, pc) << (8 * i);
            }
            reg[r] = w;
        }
        if (isq) S.Bq[sidx][nb][ln] = make_uint2(reg[0], reg[1]);
        else S.Bm[ks][nb][ln] = make_uint2(reg[0], reg[1]);
    }
    __syncthreads();
    const int g8 = lane >> 2, tg = lane & 3, rsel = tg & 1, pc0 = 2 * (tg & 1);
    float fm0[4], fm1[4], fq0[4], fq1[4], cq[4], cu[4];
    const float c0v = prm.c0, kq = prm.qjl_scale;
#pragma unroll
    for (int nb = 0; nb < 4; ++nb) {
        const int ql = 2 * nb + (tg >> 1);
        fm0[nb] = S.fm[ql * 4 + pc0];
        fm1[nb] = S.fm[ql * 4 + pc0 + 1];
        fq0[nb] = S.fq[ql * 4 + pc0];
        fq1[nb] = S.fq[ql * 4 + pc0 + 1];
        cq[nb] = c0v * S.qsum[ql];
        cu[nb] = -kq * S.usum[ql];
    }
    for (int64_t tile0 = c0; tile0 < cend; tile0 += kSTile) {
        const int nt = (int)min((int64_t)kSTile, cend - tile0);
        for (int e = threadIdx.x; e < nt * P * W; e += kThreads) {
            const int r = e / (P * W), w = e - r * (P * W);
            S.tp[r][w] = __ldg(a.planes + (size_t)(tile0 + r) * (P * W) + w);
        }
        if (qjl)
            for (int e = threadIdx.x; e < nt * W; e += kThreads) {
                const int r = e / W, w = e - r * W;
                S.tsg[r][w] = __ldg(a.signs + (size_t)(tile0 + r) * W + w);
            }
        for (int r = threadIdx.x; r < nt; r += kThreads) {
            S.tn[r] = half_bits_to_float(__ldg(a.norm + tile0 + r));
            S.tr[r] = qjl ? half_bits_to_float(__ldg(a.rnorm + tile0 + r)) : 0.f;
        }
        __syncthreads();
        if (16 * warp < nt) {
            const int rowA = 16 * warp + g8, rowB = rowA + 8;
            const int ra = rowA < nt ? rowA : 0, rb = rowB < nt ? rowB : 0;   // stale rows are never reported
            float acc[8][4] = {};
#pragma unroll
            for (int t = 0; t < T; ++t) {
#pragma unroll
                for (int sI = 0; sI < W; ++sI) {
                    uint32_t xa = 0u, xb = 0u;
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        if ((odd_mask(t) >> p) & 1) {
                            xa ^= S.tp[ra][p * W + sI];
                            xb ^= S.tp[rb][p * W + sI];
                        }
                    const uint32_t a0 = ext_nibble(xa, tg), a1 = ext_nibble(xb, tg);
                    const uint32_t a2 = ext_nibble(xa >> 16, tg), a3 = ext_nibble(xb >> 16, tg);
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb) mma_e4m3(acc[nb], a0, a1, a2, a3, S.Bm[t * W + sI][nb][lane]);
                }
            }
            if (qjl) {
#pragma unroll
                for (int sI = 0; sI < W; ++sI) {
                    const uint32_t xa = S.tsg[ra][sI], xb = S.tsg[rb][sI];
                    const uint32_t a0 = ext_nibble(xa, tg), a1 = ext_nibble(xb, tg);
                    const uint32_t a2 = ext_nibble(xa >> 16, tg), a3 = ext_nibble(xb >> 16, tg);
#pragma unroll
                    for (int nb = 0; nb < 4; ++nb) mma_e4m3(acc[4 + nb], a0, a1, a2, a3, S.Bq[sI][nb][lane]);
                }
            }
            const int row = rsel ? rowB : rowA;
            const float n = S.tn[rsel ? rb : ra], rho = S.tr[rsel ? rb : ra];
#pragma unroll
            for (int nb = 0; nb < 4; ++nb) {
                float mA = fmaf(acc[nb][0], fm0[nb], acc[nb][1] * fm1[nb]);
                float mB = fmaf(acc[nb][2], fm0[nb], acc[nb][3] * fm1[nb]);
                float uA = fmaf(acc[4 + nb][0], fq0[nb], acc[4 + nb][1] * fq1[nb]);
                float uB = fmaf(acc[4 + nb][2], fq0[nb], acc[4 + nb][3] * fq1[nb]);
                mA += __shfl_xor_sync(0xffffffffu, mA, 1);
                mB += __shfl_xor_sync(0xffffffffu, mB, 1);
                uA += __shfl_xor_sync(0xffffffffu, uA, 1);
                uB += __shfl_xor_sync(0xffffffffu, uB, 1);
                const int ql = 2 * nb + (tg >> 1);
                const float m = rsel ? mB : mA, u = rsel ? uB : uA;
                float est = n * (cq[nb] + m);
                if (qjl) est = fmaf(rho, fmaf(2.f * kq, u, cu[nb]), est);
                const int idx = (int)(tile0 + row);
                if (row < nt && ql < nqt && better(est, idx, S.st.ts[ql], S.st.ti[ql])) {
                    const int pos = atomicAdd(&S.st.cnt[ql], 1);
                    S.st.cs[ql][pos] = est;
                    S.st.ci[ql][pos] = idx;
                }
            }
        }
        __syncthreads();
        for (int ql = 0; ql < nqt; ++ql)
            if (S.st.cnt[ql] > kCand - kSTile) merge_candidates<kSQ, kThreads, 0>(S.st, ql, a.k, threadIdx.x);
    }
    for (int ql = 0; ql < nqt; ++ql)
        if (S.st.cnt[ql] > 0) merge_candidates<kSQ, kThreads, 0>(S.st, ql, a.k, threadIdx.x);
    for (int ql = 0; ql < nqt; ++ql) {
        const size_t base = ((size_t)(q0 + ql) * a.nchunk + blockIdx.x) * a.k;
        for (int t = threadIdx.x; t < a.k; t += blockDim.x) {
            const bool ok = t < S.st.nb[ql];
            a.cand_s[base + t] = ok ? S.st.bs[ql][t] : -INFINITY;
            a.cand_i[base + t] = ok ? S.st.bi[ql][t] : INT_MAX;
        }
    }
}

template <int P, int W>
cudaError_t run_mma(const SearchArgs& a, cudaStream_t st) {
    const size_t smem = sizeof(SMmaSmem<P, W>);
    cudaError_t e = cudaFuncSetAttribute(search_mma_kernel<P, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nchunk, (unsigned)((a.nq + kSQ - 1) / kSQ));
    search_mma_kernel<P, W><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t dispatch_mma(const SearchArgs& a, cudaStream_t st) {
#define TQ_MMA_P(WV)                                   \
    switch (a.prm.P) {                                 \
        case 1: return run_mma<1, WV>(a, st);          \
        case 2: return run_mma<2, WV>(a, st);          \
        case 3: return run_mma<3, WV>(a, st);          \
    }                                                  \
    break;
    switch (a.prm.W) {
        case 4: TQ_MMA_P(4)
        case 7: TQ_MMA_P(7)
        case 8: TQ_MMA_P(8)
    }
#undef TQ_MMA_P
    return cudaErrorInvalidValue;
}

bool search_mma_ok(const tq_ctx* c) {
    const Params& p = c->prm;
    return c->kernel_path != TQ_PATH_CUDA_CORE && (p.W == 4 || p.W == 7 || p.W == 8) && (!p.qjl || p.Ws == p.W) &&
           p.odd_walsh && p.P >= 1 && p.P <= 3;
}

template <int W, int P>
cudaError_t run_chunk(const SearchArgs& a, cudaStream_t st) {
    const size_t smem = Scorer<W, P>::smem_bytes(a.prm) + sizeof(SearchState);
    cudaError_t e = cudaFuncSetAttribute(search_chunk_kernel<W, P>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.nchunk, (unsigned)((a.nq + 3) / 4));
    search_chunk_kernel<W, P><<<grid, kThreads, smem, st>>>(a);
    return cudaGetLastError();
}

cudaError_t dispatch_chunk(const SearchArgs& a, bool lut, cudaStream_t st) {
    if (!lut) return run_chunk<0, 0>(a, st);
#define TQ_CASE_P(WV)                                          \
    switch (a.prm.P) {                                         \
        case 1: return run_chunk<WV, 1>(a, st);                \
        case 2: return run_chunk<WV, 2>(a, st);                \
        case 3: return run_chunk<WV, 3>(a, st);                \
        case 4: return run_chunk<WV, 4>(a, st);                \
    }                                                          \
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

}  // namespace

void search_chunking(int64_t n, int k, int* chunk, int* nchunk) {
    // At most kMergeMax / k chunks (pass 2 sorts nchunk * k candidates per query in shared
    // memory); whole tiles per chunk.
    int64_t maxc = kMergeMax / k;
    if (maxc < 1) maxc = 1;
    int64_t tiles = (n + kThreads - 1) / kThreads;
    int64_t nc = tiles < maxc ? tiles : maxc;
    if (nc < 1) nc = 1;
    int64_t c = ((tiles + nc - 1) / nc) * kThreads;
    *chunk = (int)c;
    *nchunk = (int)((n + c - 1) / c);
}

cudaError_t launch_topk_merge(const float* cand_s, const int32_t* cand_i, int R, int64_t nq, int k,
                              const ShardOffsets& offs, float* top_s, int32_t* top_i, cudaStream_t s) {
    if (nq <= 0) return cudaSuccess;
    int npow = 1;
    while (npow < R * k) npow <<= 1;
    const size_t smem = (size_t)npow * (sizeof(float) + sizeof(int));
    cudaError_t e = cudaFuncSetAttribute(shard_topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    shard_topk_merge_kernel<<<(unsigned)nq, kThreads, smem, s>>>(cand_s, cand_i, R, nq, k, npow, offs, top_s, top_i);
    return cudaGetLastError();
}

cudaError_t launch_search(const tq_ctx* c, const float* qrot, const float* qproj, int64_t nq,
                          const uint32_t* planes, const uint32_t* signs, const uint16_t* norm,
                          const uint16_t* rnorm, int64_t n, int k, float* cand_s, int* cand_i,
                          float* top_s, int32_t* top_i, cudaStream_t s) {
    if (nq <= 0) return cudaSuccess;
    SearchArgs a{};
    a.prm = c->prm;
    a.qrot = qrot;
    a.qproj = qproj;
    a.nq = nq;
    a.planes = planes;
    a.signs = signs;
    a.norm = norm;
    a.rnorm = rnorm;
    a.n = n;
    a.k = k;
    a.cand_s = cand_s;
    a.cand_i = cand_i;
    search_chunking(n, k, &a.chunk, &a.nchunk);
    a.err = c->derr;
    static int sms = 0;
    if (!sms && cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess) sms = 148;
    cudaError_t e;
    if (search_tc_ok(c)) {
        e = launch_search_tc(a, sms, s);
    } else if (search_mma_ok(c)) {
        // Few chunks when there are many query tiles: the per-CTA set-up and top-k merging
        // then amortise over long scans; at least ~4 CTAs per SM overall.
        const int64_t qtiles = (nq + kSQ - 1) / kSQ;
        int64_t want = (4 * (int64_t)sms + qtiles - 1) / qtiles;
        if (want > a.nchunk) want = a.nchunk;
        if (want < 1) want = 1;
        const int64_t tiles = (n + kSTile - 1) / kSTile;
        a.chunk = (int)(((tiles + want - 1) / want) * kSTile);
        a.nchunk = (int)((n + a.chunk - 1) / a.chunk);
        e = dispatch_mma(a, s);
    } else {
        const bool lut = lut_path_ok(a.prm, sizeof(SearchState), kSmemLimit);
        e = dispatch_chunk(a, lut, s);
    }
    if (e != cudaSuccess) return e;
    const int per_query = a.nchunk * k;
    int npow = 1;
    while (npow < per_query) npow <<= 1;
    const size_t smem = (size_t)npow * (sizeof(float) + sizeof(int));
    e = cudaFuncSetAttribute(search_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    search_merge_kernel<<<(unsigned)nq, kThreads, smem, s>>>(cand_s, cand_i, per_query, npow, k, top_s, top_i);
    return cudaGetLastError();
}

}  // namespace tq
