// Top-k vector search over compressed vectors (juejin.cn post, section 三: GloVe d=200
// Recall@1@k; section 四: near-zero indexing time, i.e. coding is the only index build).
//
// Pass 1 on the tensor cores is search_tc_kernel (k_search_tc.cu); for the other shapes and
// TQ_PATH_CUDA_CORE: one CTA per (database chunk, quad of queries), each thread scoring one
// vector for the 4 queries with the shared byte tables (lut.cuh); a score that beats the
// query's current k-th best (score descending, equal scores by lower index) is appended to a
// shared candidate buffer, which is merged into the sorted top-k list whenever another tile
// could overflow it.  Scores never go to HBM.  Pass 2: one CTA per query sorts the per-chunk
// lists and keeps the first k.  Also here: the merge of several blocks' lists (sharded search).
#include "lut.cuh"
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
