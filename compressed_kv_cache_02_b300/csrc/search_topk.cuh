// Per-CTA top-k machinery of the search kernels (juejin.cn post, section 三: the k database rows
// with the largest estimate per query): the order (score descending, equal scores by lower row),
// a bitonic sort over shared memory, and per-query candidate buffers merged into a sorted best
// list.  The helpers take the number of participating threads (threads 0 .. NT-1) and the barrier
// they meet at (0: the whole CTA, __syncthreads; -1: one warp, __syncwarp; otherwise named barrier
// BAR of NT threads); r is
// the calling thread's rank 0 .. NT-1 among them.
#pragma once

#include <climits>

#include "tq_kernels.h"

namespace tq {

constexpr int kCand = 512;         // candidate buffer per query (>= rows per tile + TQ_MAX_TOPK)
constexpr int kMergeMax = 4096;    // per-query candidates entering the final merge

struct SearchArgs {
    Params prm;
    const float* qrot;
    const float* qproj;
    int64_t nq;
    const uint32_t* planes;
    const uint32_t* signs;
    const uint16_t* norm;
    const uint16_t* rnorm;
    int64_t n;
    int k, chunk, nchunk;
    float* cand_s;   // [nq][nchunk][k]
    int* cand_i;
    int* err;        // device error flags of the context
};

// tcgen05 search (k_search_tc.cu): shapes it takes, and its launch (chunking chosen there, within
// the nchunk the workspace was sized for, which it overwrites with the count used; sms = the
// device's multiprocessor count).
bool search_tc_ok(const tq_ctx* c);
cudaError_t launch_search_tc(SearchArgs& a, int sms, cudaStream_t s);

namespace {

template <int NT, int BAR>
__device__ __forceinline__ void group_sync() {
    if (BAR < 0) __syncwarp();
    else if (BAR == 0) __syncthreads();
    else asm volatile("bar.sync %0, %1;" ::"n"(BAR), "n"(NT) : "memory");
}

__device__ __forceinline__ bool better(float s1, int i1, float s2, int i2) {
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

// Sorts n (a power of two) pairs best-first.
template <int NT, int BAR>
__device__ void bitonic_sort(float* s, int* id, int n, int r) {
    for (int size = 2; size <= n; size <<= 1) {
        for (int stride = size >> 1; stride > 0; stride >>= 1) {
            for (int t = r; t < n / 2; t += NT) {
                const int lo = 2 * stride * (t / stride) + (t % stride), hi = lo + stride;
                const bool up = (lo & size) == 0;
                const bool hi_better = better(s[hi], id[hi], s[lo], id[lo]);
                if (up ? hi_better : !hi_better) {
                    const float ts = s[lo]; s[lo] = s[hi]; s[hi] = ts;
                    const int ti = id[lo]; id[lo] = id[hi]; id[hi] = ti;
                }
            }
            group_sync<NT, BAR>();
        }
    }
}

// Number of entries of the best-first array a[0..n) that are better than (s, i).
__device__ __forceinline__ int count_better(const float* as, const int* ai, int n, float s, int i) {
    int lo = 0, hi = n;
    while (lo < hi) {
        const int mid = (lo + hi) >> 1;
        if (better(as[mid], ai[mid], s, i)) lo = mid + 1; else hi = mid;
    }
    return lo;
}

template <int NQ>
struct SearchStateT {
    float bs[NQ][TQ_MAX_TOPK];
    int bi[NQ][TQ_MAX_TOPK];
    float cs[NQ][kCand];
    int ci[NQ][kCand];
    int nb[NQ], cnt[NQ];
    float ts[NQ];
    int ti[NQ];
};

// Merges query h's candidates into its best list (both in shared memory).
template <int NQ, int NT, int BAR>
__device__ void merge_candidates(SearchStateT<NQ>& st, int h, int k, int r) {
    const int n = st.cnt[h];
    for (int t = r; t < kCand; t += NT)
        if (t >= n) { st.cs[h][t] = -INFINITY; st.ci[h][t] = INT_MAX; }
    group_sync<NT, BAR>();
    bitonic_sort<NT, BAR>(st.cs[h], st.ci[h], kCand, r);
    const int nc = min(n, k), nbb = st.nb[h];
    float* os = st.cs[h] + k;   // scratch: entries k..2k of the sorted buffer are never read
    int* oi = st.ci[h] + k;
    for (int t = r; t < nbb + nc; t += NT) {
        float s; int i, r;
        if (t < nbb) { s = st.bs[h][t]; i = st.bi[h][t]; r = t + count_better(st.cs[h], st.ci[h], nc, s, i); }
        else { const int u = t - nbb; s = st.cs[h][u]; i = st.ci[h][u]; r = u + count_better(st.bs[h], st.bi[h], nbb, s, i); }
        if (r < k) { os[r] = s; oi[r] = i; }
    }
    group_sync<NT, BAR>();
    const int nn = min(k, nbb + nc);
    for (int t = r; t < nn; t += NT) { st.bs[h][t] = os[t]; st.bi[h][t] = oi[t]; }
    group_sync<NT, BAR>();
    if (r == 0) {
        st.nb[h] = nn;
        st.cnt[h] = 0;
        if (nn == k) { st.ts[h] = st.bs[h][k - 1]; st.ti[h] = st.bi[h][k - 1]; }
    }
    group_sync<NT, BAR>();
}

}  // namespace
}  // namespace tq
