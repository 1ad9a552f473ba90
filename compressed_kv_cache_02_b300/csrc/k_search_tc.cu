// Top-k vector search on the 5th-generation tensor cores (tcgen05.mma kind::f8f6f4, A in tensor
// memory) for database rows of W = 4, 7 or 8 words per bit plane (d in (96, 128] or (192, 256])
// and 1..3 MSE bits, with or without the QJL stage.
//
// Pages: juejin.cn post, section 三 (GloVe d=200 Recall@1@k) and section 四 (coding is the whole
// index); csdn tutorial, section QJL (the asymmetric estimator).  Per (query, row) pair the score is
// the estimator of the CUDA-core search (k_search.cu), in the Walsh form of host_setup.cpp:
//   est = n (c0 sum_j q'_j + sum_t kappa_t M_t) + rho kq (2 M_u - sum_j u_j)
// with M_t the sum of q' = Pi q over the set bits of x_t (the XOR of the planes in the t-th odd
// subset) and M_u the sum of u = S q over the set sign bits.  For a tile of 128 rows and 16 queries
// the masked sums are one dense contraction, D[row][4 h + pc] = sum_k A[row][k] B[k][4 h + pc]:
// A (TMEM): each row's bit vectors (T terms, then the signs), one e4m3 byte per bit
//   (tc::expand_word: bits 2 and 3 of a byte are exactly 2^-7 and 2^-6 in e4m3);
// B (shared memory, K-major no-swizzle; built by each CTA in its prologue): piece pc of
//   kappa_t q'_j (or u_j) x 2^e0_h x (2^7 or 2^6, undoing A's scale), four e4m3 pieces
//   b0 + b1/16 + b2/256 + b3/4096 (~16 bits; e0_h puts the query's largest value in [128, 256));
// D (TMEM, fp32): 64 MSE columns (the T terms accumulate) and 64 QJL columns per buffer.
//
// A CTA owns 16 queries and a chunk of rows, with three roles that meet only at mbarriers:
//  * expander warps (one group of 4 at 1 MSE bit, one per MMA warp from 2 bits: warp 8 + 4 e + q,
//    TMEM lanes 32 q ..) turn each row's codes into its bit vectors and store them into the A
//    slots as the slots free up;
//  * two MMA warps whose lane 0 issues the MMAs of the even and of the odd tiles (one thread issues
//    about one MMA per 75-90 cycles, measured, so two keep up with the tensor pipe at N = 64);
//  * 8 scorer warps (warps w and w + 4 share TMEM lanes 32 (w % 4) ..; one takes queries 0-7, the
//    other 8-15) copy a tile's D into registers, free the buffer, and score and select.
// Each MMA warp has two one-vector A slots (64 columns each) and a D buffer (128 columns): the 512
// TMEM columns, so one CTA runs per SM.  A row that beats a query's current k-th best (score
// descending, equal scores by lower row) goes to the query's candidate buffer: the thresholds are
// read once per row and one warp vote skips the (rare, once the lists are full) appends; a buffer
// that could overflow with the next tile is merged into the query's sorted best list
// (search_topk.cuh) by the scorers of its half, which meet once per tile.  The CTA's k best per
// query go to HBM and search_merge_kernel keeps the first k over the chunks.  Every wait is
// bounded in time; one that runs out sets TQ_DEVERR_TIMEOUT, after which the CTA waits (bounded)
// for the MMAs it issued and frees its tensor memory.
#include "mma_e4m3.cuh"
#include "search_topk.cuh"
#include "tcgen05.cuh"

namespace tq {
namespace {

constexpr int kQ = 16;                      // queries per CTA
constexpr int kN = 4 * kQ;                  // B rows (D columns) per family: query x piece
constexpr int kRows = 128;                  // database rows per tile
constexpr int kScorers = 256;               // warps 0-7: D -> scores -> top-k
// Expander groups of 4 warps (warps 8, 9, ..): one at 1 MSE bit (2 bit vectors per row), one per
// MMA warp from 2 bits up, where a tile's 3-5 vectors cycle through its MMA warp's two A slots and
// one group waiting on those would leave the other MMA warp idle (4 bits: 91 -> 68 ms measured).
template <int P>
struct StRoles {
    static constexpr int kGroups = P == 1 ? 1 : 2;
    static constexpr int kExpanders = 128 * kGroups;
    static constexpr int kThreads = kScorers + kExpanders + 64;   // + two MMA warps (even and odd tiles)
};
constexpr int kQG = kQ / 2;                 // queries scored by each half of the scorers
constexpr int kSlots = 4;                   // A slots, one bit vector each: 0-1 even tiles, 2-3 odd tiles
constexpr int kSlotCols = 64;               // up to 8 words x 8 columns
constexpr int kDCols = 2 * kN;              // a D buffer: MSE then QJL columns
constexpr int kSlot0 = 2 * kDCols;          // first A slot column
constexpr int kTmemCols = 512;
constexpr uint32_t kIdesc = tc::idesc_e4m3(kN);

template <int P, int W>
struct StCfg {
    static constexpr int T = 1 << (P - 1);   // Walsh terms
    static constexpr int K = 32 * W;         // k per bit vector
    static constexpr int kBm = kN * T * K;   // MSE B bytes
    static constexpr int kBq = kN * K;       // QJL B bytes
    static constexpr int kStateOff = (kBm + kBq + 127) / 128 * 128;
    static constexpr int kUsed = kStateOff + (int)sizeof(SearchStateT<kQ>);
    // at least 120 KB: one CTA per SM, since each allocates all 512 TMEM columns
    static constexpr int kSmem = kUsed > 120 * 1024 ? kUsed : 120 * 1024;
    static_assert(kUsed <= 227 * 1024, "shared memory");
    static_assert(2 * kQ * K <= kQ * kCand, "prologue scratch (queries, projections) fits the candidate scores");
};

using u64 = unsigned long long;
__device__ __forceinline__ u64 pk2(float x, float y) {
    u64 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(x), "f"(y));
    return r;
}
__device__ __forceinline__ float2 upk2(u64 r) {
    float2 v;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
    return v;
}
__device__ __forceinline__ u64 mul2(u64 a, u64 b) {
    u64 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ u64 fma2(u64 a, u64 b, u64 c) {
    u64 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// AND of p over the 128 scorer threads of a query half (named barrier bar), which also orders
// their shared-memory accesses around it.
__device__ __forceinline__ bool half_and(bool p, int bar) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\tbar.red.and.pred po, %2, 128, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(bar)
        : "memory");
    return r != 0;
}
// Query h's merge by the scorers of its half g (rank r in the half; named barrier 1 + g).
template <int NQ>
__device__ __forceinline__ void half_merge(SearchStateT<NQ>& st, int h, int k, int g, int r) {
    if (g == 0) merge_candidates<NQ, 128, 1>(st, h, k, r);
    else merge_candidates<NQ, 128, 2>(st, h, k, r);
}

template <int P, int W>
__global__ void __launch_bounds__(StRoles<P>::kThreads, 1) search_tc_kernel(const SearchArgs a) {
    using C = StCfg<P, W>;
    constexpr int T = C::T, K = C::K;
    constexpr int kThreadsSt_ = StRoles<P>::kThreads, kExpanders = StRoles<P>::kExpanders;
    constexpr int kGroups = StRoles<P>::kGroups;
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* img = sm;
    SearchStateT<kQ>& st = *reinterpret_cast<SearchStateT<kQ>*>(sm + C::kStateOff);
    __shared__ __align__(8) uint64_t a_full[kSlots], a_free[kSlots], d_full[2], d_free[2], drain[2];
    __shared__ uint32_t s_tmem, s_merge;
    __shared__ int s_abort, s_drained;
    __shared__ int s_e0[2][kQ];
    // per query pair (h, h + 1): [0] = 2^-e0 (MSE) of both, c0 sum q' of both; [1] = 2 kq 2^-e0 (QJL) of
    // both, -kq sum u of both
    __shared__ float4 s_cst2[kQ / 2][2];
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int nv = qjl ? T + 1 : T;   // bit vectors per row
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t q0 = (int64_t)kQ * blockIdx.y;
    const int nqt = (int)min((int64_t)kQ, a.nq - q0);
    const int64_t c0 = (int64_t)blockIdx.x * a.chunk, cend = min(a.n, c0 + a.chunk);
    const int ntile = (int)((cend - c0 + kRows - 1) / kRows);

    // ---- prologue: the queries (scratch in the candidate buffers), barriers, tensor memory
    float* qv = &st.cs[0][0];
    float* uv = qv + kQ * K;
    for (int e = tid; e < kQ * K; e += kThreadsSt_) {
        const int h = e / K, j = e - h * K;
        const bool ok = h < nqt;
        qv[e] = (ok && j < prm.d) ? a.qrot[(size_t)(q0 + h) * prm.d + j] : 0.f;
        uv[e] = (qjl && ok && j < prm.m) ? a.qproj[(size_t)(q0 + h) * prm.m + j] : 0.f;
    }
    if (tid == 0) {
        for (int s = 0; s < kSlots; ++s) {
            tc::mbar_init(&a_full[s], 4);   // the 4 warps of the expander group of the slot's tiles
            tc::mbar_init(&a_free[s], 1);
        }
        for (int u = 0; u < 2; ++u) {
            tc::mbar_init(&d_full[u], 1);
            tc::mbar_init(&d_free[u], kScorers / 32);
        }
        tc::mbar_init(&drain[0], 1);
        tc::mbar_init(&drain[1], 1);
        tc::mbar_init_fence();
        s_abort = 0;
        s_merge = 0;
        s_drained = 1;
    }
    if (warp == 0) tc::tmem_alloc<kTmemCols>(&s_tmem);
    __syncthreads();
    {   // per query: column exponents and sums (warp w takes queries w, w + 10)
        float kmax = 0.f;
#pragma unroll
        for (int t = 0; t < T; ++t) kmax = fmaxf(kmax, fabsf(prm.kappa[t]));
        for (int h = warp; h < kQ; h += kThreadsSt_ / 32) {
            float mq = 0.f, sq = 0.f, mu = 0.f, su = 0.f;
            for (int j = lane; j < K; j += 32) {
                const float x = qv[h * K + j], u = uv[h * K + j];
                mq = fmaxf(mq, fabsf(x));
                sq += x;
                mu = fmaxf(mu, fabsf(u));
                su += u;
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
                sq += __shfl_xor_sync(0xffffffffu, sq, o);
                mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
                su += __shfl_xor_sync(0xffffffffu, su, o);
            }
            if (lane == 0) {
                const int em = column_exponent(128.f * kmax * mq), eu = column_exponent(128.f * mu);
                s_e0[0][h] = em;
                s_e0[1][h] = eu;
                float* c = reinterpret_cast<float*>(&s_cst2[h >> 1][0]);
                const int o = h & 1;
                c[o] = ldexpf(1.f, -em);
                c[2 + o] = prm.c0 * sq;
                c[4 + o] = 2.f * prm.qjl_scale * ldexpf(1.f, -eu);
                c[6 + o] = -prm.qjl_scale * su;
            }
        }
    }
    __syncthreads();
    // B: vector v (terms, then the signs), query h, coordinate j -> piece pc in row 32 (h / 8) + 8 pc +
    // h % 8 (each half's D columns piece-major, so the epilogue meets query pairs in adjacent registers)
    for (int e = tid; e < (T + 1) * kQ * K; e += kThreadsSt_) {
        const int v = e / (kQ * K), r = e - v * (kQ * K), h = r / K, j = r - h * K;
        const bool isq = v == T;
        const int k = 32 * (j >> 5) + tc::expanded_k(j & 31);
        const float val = isq ? uv[h * K + j] : prm.kappa[v] * qv[h * K + j];
        float x = ldexpf(val * tc::expanded_scale(j & 31), s_e0[isq ? 1 : 0][h]);
        unsigned char* fam = img + (isq ? C::kBm : 0);
        const int kk = isq ? k : v * K + k, ktot = isq ? K : T * K;
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
            const uint32_t b = to_e4m3(x);
            fam[tc::kmajor8(32 * (h >> 3) + 8 * pc + (h & 7), kk, ktot)] = (unsigned char)b;
            x = (x - from_e4m3(b)) * 16.f;
        }
    }
    tc::fence_proxy_async();
    __syncthreads();
    if (tid < kQ) {   // the scratch is dead: the top-k state starts empty
        st.nb[tid] = 0;
        st.cnt[tid] = 0;
        st.ts[tid] = -INFINITY;
        st.ti[tid] = INT_MAX;
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;

    if (warp < kScorers / 32) {
        // ---------------------------------------------------------------- scorers
        // group g = warp / 4 scores queries 8 g .. 8 g + 7 of the rows of TMEM lanes 32 (warp % 4) ..
        const int g = warp >> 2, rl = 32 * (warp & 3) + lane;
        const uint32_t lane_tmem = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        // the next tile's norms of this thread's row, raw (converted when used, so the loads stay in
        // flight for a tile); rows past the chunk read row c0 and are never reported
        uint16_t nn = 0, nr = 0;
        auto load = [&](int t) {
            const int64_t row = c0 + (int64_t)t * kRows + rl;
            const size_t rr = (size_t)(row < cend ? row : c0);
            nn = __ldg(a.norm + rr);
            if (qjl) nr = __ldg(a.rnorm + rr);
        };
        // scores of this thread's row of tile tp against the group's 8 queries, from D buffer tp % 2
        // (query pairs in packed fp32x2 arithmetic)
        float est[kQG];
        auto score = [&](int tp, float n, float rho, bool ok) -> bool {
            const int buf = tp & 1;
            if (ok) ok = tc::mbar_wait(&d_full[buf], (uint32_t)((tp >> 1) & 1));
            ok = __all_sync(0xffffffffu, ok);
            tc::fence_after();
            if (ok) {
                const uint32_t d = lane_tmem + (uint32_t)(buf * kDCols + 32 * g);   // [piece][query] of this half
                float dm[32], dq[32];
                tc::tmem_ld32(d, dm);
                if (qjl) tc::tmem_ld32(d + kN, dq);
                tc::wait_ld();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&d_free[buf]);   // D is in registers: the buffer is free
                const u64 n2 = pk2(n, n), r2 = pk2(rho, rho), s16 = pk2(1.f / 16.f, 1.f / 16.f);
#pragma unroll
                for (int pp = 0; pp < kQG / 2; ++pp) {
                    const float4 cm = s_cst2[4 * g + pp][0], cq = s_cst2[4 * g + pp][1];
                    const int i = 2 * pp;   // the pair's columns: 8 pc + i, 8 pc + i + 1
                    u64 m = fma2(pk2(dm[24 + i], dm[25 + i]), s16, pk2(dm[16 + i], dm[17 + i]));
                    m = fma2(m, s16, pk2(dm[8 + i], dm[9 + i]));
                    m = fma2(m, s16, pk2(dm[i], dm[i + 1]));
                    u64 e = mul2(n2, fma2(pk2(cm.x, cm.y), m, pk2(cm.z, cm.w)));
                    if (qjl) {
                        u64 u = fma2(pk2(dq[24 + i], dq[25 + i]), s16, pk2(dq[16 + i], dq[17 + i]));
                        u = fma2(u, s16, pk2(dq[8 + i], dq[9 + i]));
                        u = fma2(u, s16, pk2(dq[i], dq[i + 1]));
                        e = fma2(r2, fma2(pk2(cq.x, cq.y), u, pk2(cq.z, cq.w)), e);
                    }
                    const float2 ev = upk2(e);
                    est[2 * pp] = ev.x;
                    est[2 * pp + 1] = ev.y;
                }
            }
            return ok;
        };
        // Appends the scored row (index idx, -1: none) where it beats one of the group's queries' k-th
        // best.  Every listed row precedes the tile (rows are scanned in increasing order), so "beats"
        // is a strictly greater score.  A query whose buffer could overflow with the next tile is
        // flagged in s_merge.
        auto append = [&](int64_t idx) {
            uint32_t pass = 0u;
            if (idx >= 0) {   // the 8 thresholds first (they change only in merges), one vote
                const float4 t0 = reinterpret_cast<const float4*>(st.ts)[2 * g];
                const float4 t1 = reinterpret_cast<const float4*>(st.ts)[2 * g + 1];
                pass = (uint32_t)(est[0] > t0.x) | ((uint32_t)(est[1] > t0.y) << 1) | ((uint32_t)(est[2] > t0.z) << 2) |
                       ((uint32_t)(est[3] > t0.w) << 3) | ((uint32_t)(est[4] > t1.x) << 4) |
                       ((uint32_t)(est[5] > t1.y) << 5) | ((uint32_t)(est[6] > t1.z) << 6) |
                       ((uint32_t)(est[7] > t1.w) << 7);
                const int lim = nqt - kQG * g;
                pass &= lim >= kQG ? 0xFFu : lim > 0 ? (1u << lim) - 1u : 0u;
            }
            if (!__any_sync(0xffffffffu, pass != 0u)) return;
#pragma unroll
            for (int i = 0; i < kQG; ++i) {
                const int h = kQG * g + i;
                const bool ph = (pass >> i) & 1u;
                const unsigned bal = __ballot_sync(0xffffffffu, ph);
                if (bal) {
                    int base = 0;
                    if (lane == 0) {
                        base = atomicAdd(&st.cnt[h], __popc(bal));
                        if (base + __popc(bal) > kCand - kRows) atomicOr(&s_merge, 1u << h);
                    }
                    base = __shfl_sync(0xffffffffu, base, 0);
                    if (ph) {
                        const int pos = base + __popc(bal & ((1u << lane) - 1u));
                        st.cs[h][pos] = est[i];
                        st.ci[h][pos] = (int)idx;
                    }
                }
            }
        };

        // the query half's 128 threads meet once per tile (named barrier 1 + g): merge decisions are
        // uniform, and appends and merges of its queries do not overlap
        const int hr = tid - 128 * g, hbar = 1 + g, hlo = kQG * g, hhi = min(nqt, kQG * g + kQG);
        const uint32_t hmask = 0xFFu << (kQG * g);
        bool ok = true;
        load(0);
        for (int t = 0; t < ntile; ++t) {
            const float n = half_bits_to_float(nn), rho = qjl ? half_bits_to_float(nr) : 0.f;
            const int64_t row = c0 + (int64_t)t * kRows + rl;
            if (t + 1 < ntile) load(t + 1);
            ok = score(t, n, rho, ok);
            if (ok) append(row < cend ? row : -1);
            if (!half_and(ok, hbar)) {
                ok = false;
                break;
            }
            const uint32_t mm = *(volatile uint32_t*)&s_merge & hmask;
            if (mm) {
                for (int h = hlo; h < hhi; ++h)
                    if ((mm >> h) & 1u) half_merge(st, h, a.k, g, hr);
                if (hr == 0) atomicAnd(&s_merge, ~hmask);
                half_and(true, hbar);
            }
        }
        if (ok) {
            for (int h = hlo; h < hhi; ++h)
                if (st.cnt[h] > 0) half_merge(st, h, a.k, g, hr);
        } else if (hr == 0) {
            *(volatile int*)&s_abort = 1;
        }
        for (int h = hlo; h < hhi; ++h) {
            const size_t base = ((size_t)(q0 + h) * a.nchunk + blockIdx.x) * a.k;
            for (int t = hr; t < a.k; t += 128) {
                const bool have = ok && t < st.nb[h];
                a.cand_s[base + t] = have ? st.bs[h][t] : -INFINITY;
                a.cand_i[base + t] = have ? st.bi[h][t] : INT_MAX;
            }
        }
    } else if (warp < (kScorers + kExpanders) / 32) {
        // ---------------------------------------------------------------- expanders
        // group e = (warp - 8) / 4 takes tiles e, e + kGroups, .. (with two groups: the tiles of MMA warp
        // e); warp 8 + 4 e + q writes TMEM lanes 32 q .. 32 q + 31: every bit vector of those rows
        const int e = (warp - kScorers / 32) >> 2, q = warp & 3, rl = 32 * q + lane;
        const uint32_t lane_tmem = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t npl[P * W], nsg[W];   // the next tile's codes of this thread's row
        // rows past the chunk repeat row c0: their scores are never reported
        auto load = [&](int t) {
            const int64_t row = c0 + (int64_t)t * kRows + rl;
            const size_t rr = (size_t)(row < cend ? row : c0);
            const uint32_t* pl = a.planes + rr * (P * W);
#pragma unroll
            for (int i = 0; i < P * W; ++i) npl[i] = __ldg(pl + i);
            if (qjl) {
                const uint32_t* sg = a.signs + rr * W;
#pragma unroll
                for (int i = 0; i < W; ++i) nsg[i] = __ldg(sg + i);
            } else {
#pragma unroll
                for (int i = 0; i < W; ++i) nsg[i] = 0u;
            }
        };
        bool ok = true;
        if (e < ntile) load(e);
        for (int t = e; t < ntile && ok; t += kGroups) {
            if (__any_sync(0xffffffffu, *(volatile int*)&s_abort != 0)) break;
            uint32_t pl[P * W], sg[W];
#pragma unroll
            for (int i = 0; i < P * W; ++i) pl[i] = npl[i];
#pragma unroll
            for (int i = 0; i < W; ++i) sg[i] = nsg[i];
            if (t + kGroups < ntile) load(t + kGroups);
            // tile t's bit vectors into the A slots of its MMA warp (t % 2), alternately
            for (int v = 0; v < nv; ++v) {
                const int sw = (t >> 1) * nv + v, slot = 2 * (t & 1) + (sw & 1), use = sw >> 1;
                if (use >= 1) ok = tc::mbar_wait(&a_free[slot], (uint32_t)((use - 1) & 1));
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                tc::fence_after();
                uint32_t w[W];
#pragma unroll
                for (int wd = 0; wd < W; ++wd) {
                    uint32_t x = 0u;
                    if (v == T) {
                        x = sg[wd];
                    } else {
#pragma unroll
                        for (int p = 0; p < P; ++p)
                            if ((odd_mask(v) >> p) & 1) x ^= pl[p * W + wd];
                    }
                    w[wd] = x;
                }
                tc::store_bits<W>(lane_tmem + (uint32_t)(kSlot0 + slot * kSlotCols), w);
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&a_full[slot]);
            }
        }
        if (!ok && lane == 0) *(volatile int*)&s_abort = 1;
    } else {
        // ---------------------------------------------------------------- MMA issue (lane 0 of the last two warps)
        const int mw = warp - (kScorers + kExpanders) / 32;   // issues tiles mw, mw + 2, ... into D buffer mw and A slots 2 mw, 2 mw + 1
        if (lane == 0) {
            const uint32_t bimg = tc::smem_u32(img);
            const uint64_t bm0 = tc::kmajor_desc(bimg, (uint32_t)(T * K * 8));
            const uint64_t bq0 = tc::kmajor_desc(bimg + C::kBm, (uint32_t)(K * 8));
            bool issued = false, ok = true;
            for (int t = mw; t < ntile && ok; t += 2) {
                if (*(volatile int*)&s_abort) break;
                const int buf = mw;
                if (t >= 2 && !tc::mbar_wait(&d_free[buf], (uint32_t)(((t - 2) >> 1) & 1))) {
                    ok = false;
                    break;
                }
                tc::fence_after();
                for (int v = 0; v < nv; ++v) {
                    const int sw = (t >> 1) * nv + v, slot = 2 * mw + (sw & 1);
                    if (!tc::mbar_wait(&a_full[slot], (uint32_t)((sw >> 1) & 1))) {
                        ok = false;
                        break;
                    }
                    tc::fence_after();
                    const bool isq = v == T;
                    const uint32_t dcol = tmem + (uint32_t)(buf * kDCols + (isq ? kN : 0));
                    const uint32_t acol = tmem + (uint32_t)(kSlot0 + slot * kSlotCols);
#pragma unroll
                    for (int wd = 0; wd < W; ++wd) {
                        const uint64_t bd = isq ? bq0 + (uint64_t)(16 * wd) : bm0 + (uint64_t)(16 * (v * W + wd));
                        tc::mma_e4m3_ts<kIdesc>(dcol, acol + 8 * wd, bd, (wd == 0 && (v == 0 || isq)) ? 0u : 1u);
                    }
                    tc::commit(&a_free[slot]);
                    issued = true;
                }
                if (ok) tc::commit(&d_full[buf]);
            }
            if (!ok) *(volatile int*)&s_abort = 1;
            // every MMA issued has completed before the tensor memory is freed
            if (issued) {
                tc::commit(&drain[mw]);
                if (!tc::mbar_wait(&drain[mw], 0u)) s_drained = 0;
            }
        }
        __syncwarp();
    }
    tc::fence_before();
    __syncthreads();
    if (tid == 0 && s_abort) set_error(a.err, TQ_DEVERR_TIMEOUT);
    tc::fence_after();
    // an MMA that outlived the bounded drain still writes this memory: it is then left allocated
    if (warp == 0 && s_drained) tc::tmem_dealloc<kTmemCols>(tmem);
}

template <int P, int W>
cudaError_t run_tc(const SearchArgs& a, cudaStream_t s) {
    using C = StCfg<P, W>;
    cudaError_t e = cudaFuncSetAttribute(search_tc_kernel<P, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)a.nchunk, (unsigned)((a.nq + kQ - 1) / kQ));
    search_tc_kernel<P, W><<<grid, StRoles<P>::kThreads, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool search_tc_ok(const tq_ctx* c) {
    const Params& p = c->prm;
    return c->kernel_path != TQ_PATH_CUDA_CORE && (p.W == 4 || p.W == 7 || p.W == 8) && (!p.qjl || p.Ws == p.W) &&
           p.odd_walsh && p.P >= 1 && p.P <= 3 && c->d_hi == 0;
}

cudaError_t launch_search_tc(SearchArgs& a, int sms, cudaStream_t s) {
    // Chunks per query group: one CTA per SM runs, so pick the count whose rounds of CTAs come
    // closest to an even split of the work (within 1 %, the fewest chunks: every chunk refills its
    // top-k lists), at most what the workspace holds and at least 4 tiles per chunk.
    const int64_t groups = (a.nq + kQ - 1) / kQ, tiles = (a.n + kRows - 1) / kRows;
    int64_t maxc = a.nchunk;
    if (maxc > tiles / 4) maxc = tiles / 4;
    if (maxc < 1) maxc = 1;
    double best = 1e30;
    int64_t pick = 1;
    for (int64_t c = 1; c <= maxc; ++c) {
        const double cost = (double)((groups * c + sms - 1) / sms) / (double)c;
        if (cost < best * 0.99) {
            best = cost;
            pick = c;
        }
    }
    const int64_t per = (tiles + pick - 1) / pick;
    a.chunk = (int)(per * kRows);
    a.nchunk = (int)((a.n + a.chunk - 1) / a.chunk);
    switch (a.prm.P * 16 + a.prm.W) {
        case 16 + 4: return run_tc<1, 4>(a, s);
        case 16 + 7: return run_tc<1, 7>(a, s);
        case 16 + 8: return run_tc<1, 8>(a, s);
        case 32 + 4: return run_tc<2, 4>(a, s);
        case 32 + 7: return run_tc<2, 7>(a, s);
        case 32 + 8: return run_tc<2, 8>(a, s);
        case 48 + 4: return run_tc<3, 4>(a, s);
        case 48 + 7: return run_tc<3, 7>(a, s);
        case 48 + 8: return run_tc<3, 8>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
