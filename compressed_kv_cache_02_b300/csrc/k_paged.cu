// One decode step over a paged (block-table) compressed KV cache in a single persistent kernel:
// append the new token's key (PROD codes) and value (MSE codes) into their page slots, score every
// cached key against the step's queries, run the softmax and the value sum, merge the sequence
// chunks and rotate the result back, then advance the lengths.
//
// Pages: juejin.cn post, section 三 (attention logits over the compressed KV cache); csdn
// tutorial, section 背景 (every generated token joins the cache).  Readings: a page holds
// `page_size` consecutive token slots of one sequence for every KV head (pools
// [num_pages][Hkv][page_size][...]); block_table[b][i] is the page of tokens i*page_size ..
// (i+1)*page_size - 1 of sequence b; the step appends at position len[b] and attends over
// positions 0 .. len[b].
//
// Phases, separated by grid barriers (the launch is cooperative, so every CTA is resident; each
// wait is bounded and sets TQ_DEVERR_TIMEOUT when it gives up):
//   1. quantize the B x Hkv new keys and values, one vector per CTA pass, into their slots;
//   2. per (batch, KV head, head quad, chunk of 32-key blocks): rotate and project the 4 queries,
//      build their byte tables, and let each warp stream its blocks: score 32 keys (one per lane),
//      online softmax, value sum over the block's rows (lanes own coordinates); merge the warps
//      and write the chunk's (max, sum, rotated value sum) per head;
//   3. per (batch, query head): log-sum-exp merge of the chunks, back-rotation by Pi_v^T.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <string>

#include "attn_q8.cuh"
#include "tq_device.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kPThreads = 512;
constexpr int kPWarps = kPThreads / 32;
constexpr int kBarrierSpins = 1 << 22;   // x ~200 ns: a barrier gives up after about a second

__device__ __forceinline__ void cpa16(void* smem, const void* gmem) {
    const unsigned sa = static_cast<unsigned>(__cvta_generic_to_shared(smem));
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(sa), "l"(gmem));
}
__device__ __forceinline__ void cpa_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cpa_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }
__device__ __forceinline__ void cpa_wait0() { asm volatile("cp.async.wait_group 0;\n" ::); }

template <int PK>
struct KeyRow {
    uint32_t pl[PK][4], sg[4];
    float n, rho, vn;
    bool valid;
};

struct PagedArgs {
    Params kp, vp;
    const float* kPiT;    // [d][d]
    const float* kStT;    // [d][m] (S Pi^T)^T
    const float* kST;     // [d][m] S^T
    const float* vPiT;    // [d][d]
    const float* vPi;     // [d][d] row-major
    const float* q;       // [B][Hq][d]
    const void* k_new;    // [B][Hkv][d]
    const void* v_new;
    int dtype;
    int B, Hq, Hkv, G, quads, page_size, max_pages, num_pages, chunk, nchunk;
    const int32_t* table;  // [B][max_pages]
    int32_t* len;          // [B]
    uint32_t* kplanes;     // [num_pages][Hkv][page_size][PK][4]
    uint32_t* ksigns;      // [...][4]
    uint16_t* knorm;
    uint16_t* krnorm;
    uint32_t* vplanes;     // [...][PV][4]
    uint16_t* vnorm;
    float scale;
    float* out;            // [B][Hq][d]
    int* bar;              // 2 barrier counters, zero at launch
    int32_t* lenw;         // [B] the step's lengths (len + 1)
    float* partials;       // [B][Hq][nchunk][d + 2]
    int* err;
};

struct PagedShared {
    float4 Tq[4096];
    float4 Tu[4096];
    float qs[4 * 128];
    float us[4 * 128];
    float x[128], y[128], r[128];
    ulonglong2 sW[kPWarps][32];   // per key: (w0, w1), (w2, w3)
    uint4 vbuf[kPWarps][2][32 * 4];   // per warp, double-buffered value rows (up to 4 planes)
    float4 s_wm[kPWarps], s_wl[kPWarps];
    float red[kPWarps];
    float cv[kMaxLevels];
    float4 s_sum[2];
    int flag;
};

// Waits until *counter >= target, at most kBarrierSpins polls; on giving up it sets
// TQ_DEVERR_TIMEOUT and returns false.
__device__ bool bounded_wait(const int* counter, int target, int* err) {
    int spins = 0;
    while (*((const volatile int*)counter) < target) {
        if (++spins > kBarrierSpins) {
            set_error(err, TQ_DEVERR_TIMEOUT);
            return false;
        }
        __nanosleep(200);
    }
    return true;
}

__device__ bool grid_barrier(int* counter, int* err, int& abort_flag) {
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(counter, 1);
        if (!bounded_wait(counter, (int)gridDim.x, err)) abort_flag = 1;
        __threadfence();
    }
    __syncthreads();
    return abort_flag == 0;
}

// Self-test of the bounded wait: one thread arrives at a two-party barrier nobody else joins.
__global__ void wait_selftest_kernel(int* counter, int* err) {
    atomicAdd(counter, 1);
    bounded_wait(counter, 2, err);
}

__device__ __forceinline__ float block_sum(float v, PagedShared& s) {
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((threadIdx.x & 31) == 0) s.red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kPWarps; ++w) t += s.red[w];
    __syncthreads();
    return t;
}

// Phase 1 for one vector x (already in s.x): codes into the row at `row` of the pools.  With
// QJL (keys) the residual is taken in the rotated basis, y - n16 c[idx], and projected by S Pi^T.
template <int P>
__device__ void quantize_row(PagedShared& s, const Params& p, const float* PiT, const float* StT, size_t row,
                             uint32_t* planes, uint32_t* signs, uint16_t* norm, uint16_t* rnorm, int* err) {
    const int t = threadIdx.x;
    const float xv = t < 128 ? s.x[t] : 0.f;
    const float n = sqrtf(block_sum(xv * xv, s));
    const uint16_t n16b = float_to_half_bits(n);
    if ((n16b & 0x7fffu) == 0x7c00u && t == 0) set_error(err, TQ_DEVERR_NORM_OVERFLOW);
    const float n16 = half_bits_to_float(n16b);
    int idx = 0;
    float yv = 0.f;
    if (t < 128) {
        for (int j = 0; j < 128; ++j) yv = fmaf(__ldg(PiT + (size_t)j * 128 + t), s.x[j], yv);
        const float u = n > 0.f ? yv / n : 0.f;
        for (int k = 0; k + 1 < (1 << P); ++k) idx += u > p.thresholds[k];
        s.r[t] = yv - n16 * p.centroids[idx];
    }
    // bit planes: warp w < 4 holds coordinates 32 w .. 32 w + 31
#pragma unroll
    for (int b = 0; b < P; ++b) {
        const uint32_t word = __ballot_sync(0xffffffffu, (idx >> b) & 1);
        if (t < 128 && (t & 31) == 0) planes[row * (P * 4) + b * 4 + (t >> 5)] = word;
    }
    if (t == 0) norm[row] = n16b;
    if (!p.qjl) {
        __syncthreads();
        return;
    }
    const float rv = t < 128 ? s.r[t] : 0.f;
    const float rn = sqrtf(block_sum(rv * rv, s));   // its barrier also publishes s.r
    float zv = 0.f;
    if (t < 128) {
        for (int j = 0; j < 128; ++j) zv = fmaf(__ldg(StT + (size_t)j * 128 + t), s.r[j], zv);
    }
    const uint32_t sw = __ballot_sync(0xffffffffu, t < 128 && zv > 0.f);
    if (t < 128 && (t & 31) == 0) signs[row * 4 + (t >> 5)] = sw;
    if (t == 0) {
        const uint16_t rb = float_to_half_bits(rn);
        if ((rb & 0x7fffu) == 0x7c00u) set_error(err, TQ_DEVERR_NORM_OVERFLOW);
        rnorm[row] = rb;
    }
    __syncthreads();
}

__device__ __forceinline__ bool slot_of(const PagedArgs& a, int b, int pos, size_t h, size_t& row) {
    const int pi = pos / a.page_size;
    if (pos < 0 || pi >= a.max_pages) return false;
    const int page = a.table[(size_t)b * a.max_pages + pi];
    if (page < 0 || page >= a.num_pages) return false;
    row = ((size_t)page * a.Hkv + h) * a.page_size + (pos - pi * a.page_size);
    return true;
}

// Phase 2 for one (b, kvh, quad, chunk) item.
template <int PK, int PV>
__device__ void attend_chunk(const PagedArgs& a, PagedShared& s, int b, int kvh, int quad, int chunk) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int L = __ldcg(a.lenw + b);
    const int hbase = kvh * a.G + 4 * quad;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    const int k_lo = chunk * a.chunk, k_hi = min(L, k_lo + a.chunk);
    const size_t stride = 128 + 2;
    float* pbase = a.partials + (((size_t)b * a.Hq + hbase) * a.nchunk + chunk) * stride;
    const size_t hstride = (size_t)a.nchunk * stride;
    if (k_lo >= k_hi) {   // nothing cached here: an empty partial
        if (threadIdx.x < nh) {
            pbase[threadIdx.x * hstride] = -INFINITY;
            pbase[threadIdx.x * hstride + 1] = 0.f;
        }
        return;
    }
    // rotated and projected queries of the quad (rows past the group read as 0)
    const float* qrow = a.q + ((size_t)b * a.Hq + hbase) * 128;
    for (int e = threadIdx.x; e < 4 * 128; e += blockDim.x) {
        const int r = e >> 7, i = e & 127;
        float aq = 0.f, au = 0.f;
        if (r < nh) {
            const float* qr = qrow + (size_t)r * 128;
            for (int j = 0; j < 128; ++j) {
                const float qv = __ldg(qr + j);
                aq = fmaf(__ldg(a.kPiT + (size_t)j * 128 + i), qv, aq);
                au = fmaf(__ldg(a.kST + (size_t)j * 128 + i), qv, au);
            }
        }
        s.qs[e] = aq;
        s.us[e] = au;
    }
    __syncthreads();
    build_tables_vk(s.Tq, s.qs, 128);
    build_tables_vk(s.Tu, s.us, 128);
    if (threadIdx.x == 0) {
        float4 sq = make_float4(0.f, 0.f, 0.f, 0.f), su = sq;
        for (int k = 0; k < 16; ++k) {
            sq = f4_add(sq, s.Tq[255 * 16 + k]);
            su = f4_add(su, s.Tu[255 * 16 + k]);
        }
        s.s_sum[0] = sq;
        s.s_sum[1] = su;
    }
    __syncthreads();
    const float kq = a.kp.qjl_scale;
    const float4 cq = f4_scale(a.kp.c0, s.s_sum[0]), cu = f4_scale(-kq, s.s_sum[1]);
    float kap[OddMasks<PK>::n];
#pragma unroll
    for (int t = 0; t < OddMasks<PK>::n; ++t) kap[t] = a.kp.kappa[t];
    const int r8 = lane & 7, wsel = lane >> 3;
    int rot[PV];
#pragma unroll
    for (int pp = 0; pp < PV; ++pp) rot[pp] = ((lane & 7) - pp - 2) & 31;
    const unsigned char* cvb = reinterpret_cast<const unsigned char*>(s.cv);
    u64 acc[4][2];   // owned coordinate c: heads (0, 1) in acc[c][0], (2, 3) in acc[c][1]
#pragma unroll
    for (int c = 0; c < 4; ++c) acc[c][0] = acc[c][1] = 0ull;
    float4 m4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    float4 ls = make_float4(0.f, 0.f, 0.f, 0.f);
    const int nblk = (k_hi - k_lo + 31) / 32;
    // block jj's value rows (one page: page_size is a multiple of 32) into buffer buf, by cp.async
    auto issue_vals = [&](int jj, int buf) {
        size_t r0 = 0;
        if (jj >= nblk || !slot_of(a, b, k_lo + jj * 32, kvh, r0)) return;
        const int nk = min(32, k_hi - (k_lo + jj * 32));
        const uint4* src = reinterpret_cast<const uint4*>(a.vplanes + r0 * (PV * 4));
        for (int e = lane; e < nk * PV; e += 32) cpa16(&s.vbuf[warp][buf][e], src + e);
    };
    // this lane's key of block jj into registers
    auto load_key = [&](int jj, KeyRow<PK>& kr) {
        const int key = k_lo + jj * 32 + lane;
        size_t row = 0;
        kr.valid = jj < nblk && key < k_hi && slot_of(a, b, key, kvh, row);
        if (!kr.valid) return;
#pragma unroll
        for (int p = 0; p < PK; ++p) {
            const uint4 v = __ldcg(reinterpret_cast<const uint4*>(a.kplanes + row * (PK * 4)) + p);
            kr.pl[p][0] = v.x; kr.pl[p][1] = v.y; kr.pl[p][2] = v.z; kr.pl[p][3] = v.w;
        }
        const uint4 sv = __ldcg(reinterpret_cast<const uint4*>(a.ksigns + row * 4));
        kr.sg[0] = sv.x; kr.sg[1] = sv.y; kr.sg[2] = sv.z; kr.sg[3] = sv.w;
        kr.n = half_bits_to_float(__ldcg(a.knorm + row));
        kr.rho = half_bits_to_float(__ldcg(a.krnorm + row));
        kr.vn = half_bits_to_float(__ldcg(a.vnorm + row));
    };
    KeyRow<PK> cur, nxt;
    load_key(warp, cur);
    issue_vals(warp, 0);
    cpa_commit();
    int buf = 0;
    for (int j = warp; j < nblk; j += kPWarps, buf ^= 1) {
        const int jn = j + kPWarps;
        issue_vals(jn, buf ^ 1);   // the next block's rows and key are in flight while this one runs
        cpa_commit();
        load_key(jn, nxt);
        float4 l4 = make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
        float vn = 0.f;
        if (cur.valid) {
            const float4 e = score_key<PK>(s.Tq, s.Tu, cur.pl, cur.sg, cur.n, cur.rho, r8, kap, cq, cu, 2.f * kq, true);
            l4.x = a.scale * e.x;
            l4.y = nh > 1 ? a.scale * e.y : -INFINITY;
            l4.z = nh > 2 ? a.scale * e.z : -INFINITY;
            l4.w = nh > 3 ? a.scale * e.w : -INFINITY;
            vn = cur.vn;
        }
        // online softmax over the block (one key per lane)
        const float4 mn = f4_max(m4, warp_max4_redux(l4));
        if (mn.x != m4.x || mn.y != m4.y || mn.z != m4.z || mn.w != m4.w) {   // warp-uniform
            const float4 al = make_float4(rescale(m4.x, mn.x), rescale(m4.y, mn.y), rescale(m4.z, mn.z), rescale(m4.w, mn.w));
            m4 = mn;
            ls = make_float4(ls.x * al.x, ls.y * al.y, ls.z * al.z, ls.w * al.w);
            const u64 a01 = pk2(al.x, al.y), a23 = pk2(al.z, al.w);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                acc[c][0] = mul2(acc[c][0], a01);
                acc[c][1] = mul2(acc[c][1], a23);
            }
        }
        const float4 pr = make_float4(safe_exp(l4.x, m4.x), safe_exp(l4.y, m4.y), safe_exp(l4.z, m4.z), safe_exp(l4.w, m4.w));
        ls = f4_add(ls, pr);
        const float4 w = f4_scale(vn, pr);
        s.sW[warp][lane] = make_ulonglong2(pk2(w.x, w.y), pk2(w.z, w.w));
        size_t row0 = 0;
        const bool have = slot_of(a, b, k_lo + j * 32, kvh, row0);
        const int nk = min(32, k_hi - (k_lo + j * 32));
        cpa_wait1();   // this block's value rows have landed
        __syncwarp();
        if (have) {
            const uint32_t* vb = reinterpret_cast<const uint32_t*>(&s.vbuf[warp][buf][0]);
            for (int t = 0; t < nk; ++t) {
                const uint32_t* vr = vb + t * (PV * 4);
                uint32_t z = 0u;
#pragma unroll
                for (int pp = 0; pp < PV; ++pp) {
                    const uint32_t wd = vr[pp * 4 + wsel];
                    z |= __funnelshift_r(wd, wd, rot[pp]) & (0x04040404u << pp);
                }
                // the centroid of owned coordinate c doubled, against the head pairs' weights
                const ulonglong2 wv = s.sW[warp][t];
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const float cv = *reinterpret_cast<const float*>(cvb + __byte_perm(z, 0u, 0x4440 + c));
                    const u64 cc = pk2(cv, cv);
                    acc[c][0] = fma2(cc, wv.x, acc[c][0]);
                    acc[c][1] = fma2(cc, wv.y, acc[c][1]);
                }
            }
        }
        __syncwarp();   // sW and this buffer are reused
        cur = nxt;
    }
    cpa_wait0();
    // merge the warps of the CTA
    ls = warp_sum4(ls);
    if (lane == 0) {
        s.s_wm[warp] = m4;
        s.s_wl[warp] = ls;
    }
    __syncthreads();   // the tables are no longer read: Tq becomes the merge buffer
    float4 M = s.s_wm[0];
    for (int w = 1; w < kPWarps; ++w) M = f4_max(M, s.s_wm[w]);
    const float4 sc = make_float4(rescale(m4.x, M.x), rescale(m4.y, M.y), rescale(m4.z, M.z), rescale(m4.w, M.w));
    float4* red = s.Tq;   // [warps][4 coordinates][32 lanes]
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float2 h01 = upk2(acc[c][0]), h23 = upk2(acc[c][1]);
        red[(warp * 4 + c) * 32 + lane] = make_float4(h01.x * sc.x, h01.y * sc.y, h23.x * sc.z, h23.y * sc.w);
    }
    __syncthreads();
    if (threadIdx.x < 128) {
        const int c = threadIdx.x >> 5, l = threadIdx.x & 31, jc = 32 * (l >> 3) + (l & 7) + 8 * c;
        float4 sum = red[c * 32 + l];
        for (int w = 1; w < kPWarps; ++w) sum = f4_add(sum, red[(w * 4 + c) * 32 + l]);
        const float vv[4] = {sum.x, sum.y, sum.z, sum.w};
        for (int h = 0; h < nh; ++h) pbase[h * hstride + 2 + jc] = vv[h];
    }
    if (threadIdx.x == 0) {
        float4 lt = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int w = 0; w < kPWarps; ++w) {
            const float4 mw = s.s_wm[w], lw = s.s_wl[w];
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
    __syncthreads();
}

template <int PK, int PV>
__global__ void __launch_bounds__(kPThreads, 1) paged_decode_kernel(const PagedArgs a) {
    extern __shared__ __align__(16) unsigned char psm_raw[];
    PagedShared& s = *reinterpret_cast<PagedShared*>(psm_raw);
    if (threadIdx.x == 0) s.flag = 0;
    if (threadIdx.x < kMaxLevels) s.cv[threadIdx.x] = a.vp.centroids[threadIdx.x];
    __syncthreads();
    // ---- phase 1: append the new keys and values
    if (blockIdx.x == 0) {
        for (int b = threadIdx.x; b < a.B; b += blockDim.x) {   // no page for position len[b]: no append
            const int L = a.len[b], cap = a.max_pages * a.page_size;
            size_t row = 0;
            const bool ok = slot_of(a, b, L, 0, row);
            if (!ok) set_error(a.err, TQ_DEVERR_LEN_RANGE);
            a.lenw[b] = ok ? L + 1 : (L < 0 ? 0 : (L > cap ? cap : L));
        }
    }
    const int n1 = a.B * a.Hkv * 2;
    for (int it = blockIdx.x; it < n1; it += gridDim.x) {
        const int kind = it & 1, bh = it >> 1, b = bh / a.Hkv, h = bh - b * a.Hkv;
        const int pos = a.len[b];
        size_t row = 0;
        const bool ok = slot_of(a, b, pos, h, row);   // CTA-uniform
        if (!ok) continue;   // flagged above
        const void* src = kind == 0 ? a.k_new : a.v_new;
        const size_t off = ((size_t)b * a.Hkv + h) * 128;
        if (threadIdx.x < 128)
            s.x[threadIdx.x] = a.dtype == TQ_BF16 ? bf16_bits_to_float(static_cast<const uint16_t*>(src)[off + threadIdx.x])
                                                  : static_cast<const float*>(src)[off + threadIdx.x];
        __syncthreads();
        if (kind == 0)
            quantize_row<PK>(s, a.kp, a.kPiT, a.kStT, row, a.kplanes, a.ksigns, a.knorm, a.krnorm, a.err);
        else
            quantize_row<PV>(s, a.vp, a.vPiT, nullptr, row, a.vplanes, nullptr, a.vnorm, nullptr, a.err);
    }
    if (!grid_barrier(a.bar, a.err, s.flag)) return;
    // ---- phase 2: chunks of the attention
    const int n2 = a.B * a.Hkv * a.quads * a.nchunk;
    for (int it = blockIdx.x; it < n2; it += gridDim.x) {
        const int chunk = it % a.nchunk, r0 = it / a.nchunk;
        const int quad = r0 % a.quads, bh = r0 / a.quads;
        attend_chunk<PK, PV>(a, s, bh / a.Hkv, bh % a.Hkv, quad, chunk);
    }
    if (!grid_barrier(a.bar + 1, a.err, s.flag)) return;
    // ---- phase 3: merge the chunks per (batch, query head), rotate back, advance the length
    const size_t stride = 128 + 2;
    for (int it = blockIdx.x; it < a.B * a.Hq; it += gridDim.x) {
        const int b = it / a.Hq, h = it - b * a.Hq;
        const int L = __ldcg(a.lenw + b);
        const int nch = (L + a.chunk - 1) / a.chunk;
        const float* pb = a.partials + ((size_t)b * a.Hq + h) * a.nchunk * stride;
        float M = -INFINITY;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, __ldcg(pb + c * stride));
        float lsum = 0.f, acc = 0.f;
        for (int c = 0; c < nch; ++c) {
            const float mc = __ldcg(pb + c * stride);
            const float wgt = mc == -INFINITY ? 0.f : expf(mc - M);
            lsum = fmaf(wgt, __ldcg(pb + c * stride + 1), lsum);
            if (threadIdx.x < 128) acc = fmaf(wgt, __ldcg(pb + c * stride + 2 + threadIdx.x), acc);
        }
        if (threadIdx.x < 128) s.y[threadIdx.x] = lsum > 0.f ? acc / lsum : 0.f;
        __syncthreads();
        if (threadIdx.x < 128) {
            float o = 0.f;
            for (int i = 0; i < 128; ++i) o = fmaf(__ldg(a.vPi + (size_t)i * 128 + threadIdx.x), s.y[i], o);
            a.out[((size_t)b * a.Hq + h) * 128 + threadIdx.x] = o;
        }
        if (h == 0 && threadIdx.x == 0) a.len[b] = L;
        __syncthreads();
    }
}

template <int PK, int PV>
cudaError_t launch_paged(const PagedArgs& a, int device, cudaStream_t st) {
    const size_t smem = sizeof(PagedShared);
    cudaError_t e = cudaFuncSetAttribute(paged_decode_kernel<PK, PV>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, paged_decode_kernel<PK, PV>, kPThreads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int grid = sms * per_sm;
    void* args[] = {const_cast<PagedArgs*>(&a)};
    return cudaLaunchCooperativeKernel(reinterpret_cast<void*>(paged_decode_kernel<PK, PV>), dim3(grid), dim3(kPThreads),
                                       args, smem, st);
}

template <int PK>
cudaError_t launch_paged_v(const PagedArgs& a, int device, cudaStream_t st) {
    switch (a.vp.P) {
        case 1: return launch_paged<PK, 1>(a, device, st);
        case 2: return launch_paged<PK, 2>(a, device, st);
        case 3: return launch_paged<PK, 3>(a, device, st);
        case 4: return launch_paged<PK, 4>(a, device, st);
    }
    return cudaErrorInvalidValue;
}

// Tokens per chunk (a multiple of 32).  Phase 2 runs ceil(items / CTAs) rounds of items, items =
// groups x chunks, and each item pays for its table set-up (~2048 keys' worth of time), so the
// chunk count minimises rounds x (keys per chunk + 2048) for one CTA per SM of a B300 (148).
int paged_chunk(int B, int Hkv, int quads, int64_t cap) {
    const int64_t groups = (int64_t)B * Hkv * quads, ctas = 148;
    int64_t best_cost = -1, best = 32;
    for (int64_t nc = 1; nc <= 64; ++nc) {
        const int64_t chunk = ((cap + nc - 1) / nc + 31) / 32 * 32;
        const int64_t rounds = (groups * nc + ctas - 1) / ctas;
        const int64_t cost = rounds * (chunk + 2048);
        if (best_cost < 0 || cost < best_cost) {
            best_cost = cost;
            best = chunk;
        }
    }
    return (int)std::max<int64_t>(best, 32);
}

}  // namespace
}  // namespace tq

// ---------------------------------------------------------------- C-ABI

namespace {

size_t paged_ws_layout(int B, int Hq, int Hkv, int max_pages, int page_size, int* chunk, int* nchunk) {
    const int quads = (Hq / Hkv + 3) / 4;
    const int64_t cap = (int64_t)max_pages * page_size;
    const int c = tq::paged_chunk(B, Hkv, quads, cap);
    const int n = (int)((cap + c - 1) / c);
    if (chunk) *chunk = c;
    if (nchunk) *nchunk = n;
    const size_t head = 16 + (((size_t)B * 4 + 15) / 16) * 16;
    return head + (size_t)B * Hq * n * (128 + 2) * sizeof(float);
}

}  // namespace

extern "C" {

int tq_paged_workspace_size(int B, int Hq, int Hkv, int max_pages, int page_size, size_t* bytes) {
    if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv || max_pages < 1 || page_size < 32 || page_size % 32 || !bytes)
        return tq::fail(TQ_ERR_ARG, "tq_paged_workspace_size: B, Hkv >= 1, Hq a multiple of Hkv, max_pages >= 1, "
                                    "page_size a positive multiple of 32");
    *bytes = paged_ws_layout(B, Hq, Hkv, max_pages, page_size, nullptr, nullptr);
    return TQ_OK;
}

int tq_paged_decode_step(tq_ctx* kctx, const tq_ctx* vctx, const float* q, const void* k_new, const void* v_new,
                         int dtype, int B, int Hq, int Hkv, const int32_t* block_table, int max_pages, int page_size,
                         int num_pages, int32_t* len, uint32_t* kplanes, uint32_t* ksigns, uint16_t* knorm,
                         uint16_t* krnorm, uint32_t* vplanes, uint16_t* vnorm, float scale, float* out,
                         void* workspace, size_t workspace_bytes, void* stream) {
    if (!kctx || !vctx) return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: NULL context");
    int dev = -1;
    cudaError_t ce = cudaGetDevice(&dev);
    if (ce != cudaSuccess || dev != kctx->device || dev != vctx->device)
        return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: the contexts belong to another device");
    if (kctx->mode != TQ_MODE_PROD || kctx->d != 128 || kctx->m != 128 || kctx->d_hi || !kctx->prm.odd_walsh)
        return tq::fail(TQ_ERR_UNSUPPORTED, "tq_paged_decode_step: keys need a PROD context with d = m = 128 "
                                            "(not split)");
    if (vctx->mode != TQ_MODE_MSE || vctx->d != 128 || vctx->d_hi || vctx->P > tq::kFastBits)
        return tq::fail(TQ_ERR_UNSUPPORTED, "tq_paged_decode_step: values need an MSE context with d = 128 "
                                            "and 1..4 bits (not split)");
    if (dtype != TQ_F32 && dtype != TQ_BF16) return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: dtype");
    size_t need = 0;
    int rc = tq_paged_workspace_size(B, Hq, Hkv, max_pages, page_size, &need);
    if (rc != TQ_OK) return rc;
    if (num_pages < 1 || (int64_t)max_pages * page_size > (1 << 30))
        return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: num_pages >= 1, max_pages * page_size <= 2^30");
    if (!q || !k_new || !v_new || !block_table || !len || !kplanes || !ksigns || !knorm || !krnorm || !vplanes ||
        !vnorm || !out || !workspace)
        return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: NULL buffer");
    if (workspace_bytes < need) return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: workspace too small");
    if ((reinterpret_cast<uintptr_t>(kplanes) | reinterpret_cast<uintptr_t>(ksigns) |
         reinterpret_cast<uintptr_t>(vplanes) | reinterpret_cast<uintptr_t>(workspace)) % 16)
        return tq::fail(TQ_ERR_ARG, "tq_paged_decode_step: planes, signs and workspace must be 16-byte aligned");
    tq::PagedArgs a{};
    a.kp = kctx->prm;
    a.vp = vctx->prm;
    a.kPiT = kctx->dPiT;
    a.kStT = kctx->dStT;
    a.kST = kctx->dST;
    a.vPiT = vctx->dPiT;
    a.vPi = vctx->dPi;
    a.q = q;
    a.k_new = k_new;
    a.v_new = v_new;
    a.dtype = dtype;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.quads = (a.G + 3) / 4;
    a.page_size = page_size;
    a.max_pages = max_pages;
    a.num_pages = num_pages;
    paged_ws_layout(B, Hq, Hkv, max_pages, page_size, &a.chunk, &a.nchunk);
    a.table = block_table;
    a.len = len;
    a.kplanes = kplanes;
    a.ksigns = ksigns;
    a.knorm = knorm;
    a.krnorm = krnorm;
    a.vplanes = vplanes;
    a.vnorm = vnorm;
    a.scale = scale;
    a.out = out;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    a.bar = reinterpret_cast<int*>(ws);
    a.lenw = reinterpret_cast<int32_t*>(ws + 16);
    a.partials = reinterpret_cast<float*>(ws + 16 + (((size_t)B * 4 + 15) / 16) * 16);
    a.err = kctx->derr;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    ce = cudaMemsetAsync(a.bar, 0, 16, st);
    if (ce != cudaSuccess) return tq::fail(TQ_ERR_CUDA, std::string("cudaMemsetAsync: ") + cudaGetErrorString(ce));
    switch (kctx->P) {
        case 1: ce = tq::launch_paged_v<1>(a, dev, st); break;
        case 2: ce = tq::launch_paged_v<2>(a, dev, st); break;
        case 3: ce = tq::launch_paged_v<3>(a, dev, st); break;
        default: return tq::fail(TQ_ERR_UNSUPPORTED, "tq_paged_decode_step: keys need 1..3 MSE bits");
    }
    if (ce != cudaSuccess)
        return tq::fail(TQ_ERR_CUDA, std::string("paged_decode_kernel launch: ") + cudaGetErrorString(ce));
    return TQ_OK;
}

}  // extern "C"

extern "C" int tq_selftest_wait_timeout(tq_ctx* ctx, void* stream) {
    if (!ctx) return tq::fail(TQ_ERR_ARG, "tq_selftest_wait_timeout: context is NULL");
    int* counter = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&counter), sizeof(int));
    if (e != cudaSuccess) return tq::fail(TQ_ERR_CUDA, std::string("cudaMalloc: ") + cudaGetErrorString(e));
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(counter, 0, sizeof(int), st);
    if (e == cudaSuccess) {
        tq::wait_selftest_kernel<<<1, 1, 0, st>>>(counter, ctx->derr);
        e = cudaGetLastError();
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(counter);
    return e == cudaSuccess ? TQ_OK : tq::fail(TQ_ERR_CUDA, std::string("wait self-test: ") + cudaGetErrorString(e));
}
