// Attention logits on the 5th-generation tensor cores (tcgen05.mma kind::f8f6f4 with the A
// operand in tensor memory) for 96 < d <= 128 (m <= 128 in PROD mode) and 1..3 MSE bits.
//
// Pages: juejin.cn post section 三 and csdn tutorial section QJL (the asymmetric estimator);
// the arithmetic per key is that of the CUDA-core kernels in k_attn.cu, rearranged as a small
// dense contraction per tile of 128 keys:
//   Walsh form (host_setup.cpp): <Pi q, c[idx]> = c0 sum_j q'_j + sum_t kappa_t M_t with M_t the
//   sum of q' over the set bits of x_t, the XOR of the planes in term t; <S q, 2 sign - 1> =
//   2 M_u - sum_j u_j.  So per key we need masked sums of T + 1 bit vectors of 128 bits against
//   the 4 query heads of a GQA quad:  D[key][column] = sum_k A[key][k] B[k][column].
//
// A (128 keys x K, in TMEM): every bit becomes one e4m3 byte.  Bits 2 and 3 of a byte are, as
//   e4m3, exactly 2^-7 and 2^-6 (subnormal 4 x 2^-9, and the smallest normal), so masking a
//   shifted copy of a 32-bit word with 0x04040404 or 0x08080808 yields 4 coordinates at once:
//   register c of word x is ((x >> s_c) & mask_c), byte i holding coordinate 8 i + ((c + 2) & 7)
//   of the word with value 2^-7 (c even) or 2^-6 (c odd).  Eleven ALU operations per 32
//   coordinates; tcgen05.st writes the registers as TMEM columns (4 k per 32-bit column).
// B (K x 16 columns, shared memory, K-major no-swizzle core matrices): column 4 h + pc is piece
//   pc of query head h, value x 2^(e0_h) x (2^7 or 2^6, undoing the A scale); four e4m3 pieces
//   x = b0 + b1/16 + b2/256 + b3/4096 carry ~16 bits.  Built once per group by
//   tc_image_kernel, with the epilogue constants, and copied into shared memory per CTA.
// D (fp32, TMEM): 16 columns per mma warp; the MSE blocks sum, and so do the QJL ones.
//
// One CTA per SM owns a contiguous range of 128-key tiles and runs them through a pipeline of
// specialised warps that meet only at mbarriers (all waits bounded; a timeout sets
// TQ_DEVERR_TIMEOUT and stops every role):
//   producer warp  bulk asynchronous copies of each tile's fields (planes, signs, norms,
//                  residual norms; lengths rounded up to 8 keys, inside the cache since its
//                  capacity is a multiple of 8) into a ring of shared-memory stages;
//   16 worker warps warp w expands word w / 4 of every bit vector of keys 32 (w % 4) .. + 31
//                  (its TMEM lanes) into the tile's A buffer, and kLag tiles later finishes
//                  head w / 4 of those keys from D (fp32) into logits;
//   mma warps      kSplit warps per bit vector, each issuing its share of the vector's 4
//                  tcgen05.mma (K = 32 each) into its own 16 D columns and committing (a single
//                  thread spends ~70 cycles per mma issue, so the issue is spread over warps); at a
//                  group change they drain their mma and the first loads the group's B.
// TMEM holds kNB tile buffers (A and D), so expansion, mma and the epilogue of different tiles
// overlap.
#include "mma_e4m3.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kTile = 128;
constexpr int kWorkers = 16;                      // warps 0..15
constexpr int kProducerWarp = kWorkers;           // then one mma warp per bit vector
constexpr int kSuspendNs = 20000;     // suspend-time hint of one try_wait
constexpr int kWaitLimit = 1 << 16;   // tries before a wait gives up (bounded by ~1.3 s)

template <int P>
struct TcCfg {
    static constexpr int T = 1 << (P - 1);      // Walsh terms
    static constexpr int NV = T + 1;            // bit vectors per key (terms, then signs)
    static constexpr int kSplit = 1;                // mma warps per bit vector (each its K share)
    static constexpr int NI = NV * kSplit;          // mma warps
    static constexpr int kThreads = (kWorkers + 1 + NI) * 32;
    static constexpr int kACols = NV * 32;      // A: NV x 4 words x 8 columns (4 e4m3 each)
    static constexpr int kDCols = NI * 16;      // D: 16 columns per mma warp
    static constexpr int kBufCols = kACols + kDCols;
    static constexpr int kNB = 512 / kBufCols >= 4 ? 4 : 512 / kBufCols;   // TMEM tile buffers
    static constexpr int kLag = kNB - 1;        // tiles between a tile's expansion and its finish
    static constexpr int kSignOff = kTile * P * 16;
    static constexpr int kNormOff = kSignOff + kTile * 16;
    static constexpr int kRnormOff = kNormOff + kTile * 2;
    static constexpr int kStageBytes = kRnormOff + kTile * 2;
    // enough stages to fill more than half of shared memory: one CTA (and its 512 TMEM
    // columns) per SM
    static constexpr int kStages = (120 * 1024 + kStageBytes - 1) / kStageBytes;
    static constexpr int kBmBytes = 16 * T * 128;   // MSE B: 16 columns x T*128 k
    static constexpr int kBqBytes = 16 * 128;       // QJL B: 16 columns x 128 k
    static constexpr int kConstOff = kBmBytes + kBqBytes;
    static constexpr int kImgBytes = (kConstOff + 64 + 127) / 128 * 128;
    static constexpr int kImgOff = kStages * kStageBytes;
    static constexpr int kSmem = kImgOff + kImgBytes;
    static_assert(kStageBytes % 128 == 0, "stage alignment");
    static_assert(kNB >= 2 && kNB * kBufCols <= 512, "TMEM budget");
    static_assert(kLag < kStages, "the producer must run ahead of the finish");
    static constexpr int kMaxStages = 32;
    static_assert(kStages <= kMaxStages, "barrier array");
};

struct TcArgs {
    Params prm;
    const float* qrot;
    const float* qproj;
    int B, Hq, Hkv, G, quads, ngroups;
    KeyCache k;
    float scale;
    float* logits;
    unsigned char* img;
    int* err;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void bar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}
// Waits for the phase with the given parity to complete.  Each try_wait may suspend the thread
// for up to kSuspendNs (it resumes as soon as the phase completes), so waiting warps do not
// spin on the issue slots; false after kWaitLimit tries (~1 s).
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
    for (int it = 0; it < kWaitLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
            : "memory");
        if (done) return true;
    }
    return false;
}

// K-major no-swizzle operand: core matrices of 8 rows x 16 bytes, LBO = 128 B along K,
// SBO = sbo bytes between 8-row groups; descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
           ((uint64_t)1 << 46);
}
// byte offset of element (row r, k) in a [rows x ktot] 8-bit K-major operand
__host__ __device__ __forceinline__ uint32_t kmajor8(int r, int k, int ktot) {
    return (uint32_t)(((r >> 3) * (ktot >> 4) + (k >> 4)) * 128 + (r & 7) * 16 + (k & 15));
}

// kind::f8f6f4: D f32, A and B e4m3, N = 16, M = 128
constexpr uint32_t kIdesc = (1u << 4) | ((16u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(kIdesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar)));
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
    uint32_t r[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void bar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void bar_init_n(uint64_t* bar, int n) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(n));
}

// The 8 A registers of one 32-bit bit-vector word (see the file comment).
__device__ __forceinline__ void expand_word(uint32_t x, uint32_t (&r)[8]) {
    const uint32_t y = x >> 2, z = x >> 4, u = x << 2;
    r[0] = x & 0x04040404u;
    r[1] = x & 0x08080808u;
    r[2] = y & 0x04040404u;
    r[3] = y & 0x08080808u;
    r[4] = z & 0x04040404u;
    r[5] = z & 0x08080808u;
    r[6] = u & 0x04040404u;
    r[7] = u & 0x08080808u;
}

__device__ __forceinline__ int group_len(const TcArgs& a, int g) {
    const int L = a.k.len[g / (a.Hkv * a.quads)];
    return L < 0 ? 0 : (L > a.k.cap ? (int)a.k.cap : L);
}

struct Cursor {
    int g, L, k0;
};

__device__ Cursor seek(const TcArgs& a, int64_t u) {
    Cursor c{0, 0, 0};
    for (; c.g < a.ngroups; ++c.g) {
        c.L = group_len(a, c.g);
        const int64_t n = (c.L + kTile - 1) / kTile;
        if (u < n) {
            c.k0 = (int)(u * kTile);
            return c;
        }
        u -= n;
    }
    c.L = 0;
    return c;
}

__device__ __forceinline__ void next_tile(const TcArgs& a, Cursor& c) {
    c.k0 += kTile;
    while (c.k0 >= c.L && c.g < a.ngroups) {
        ++c.g;
        c.k0 = 0;
        c.L = c.g < a.ngroups ? group_len(a, c.g) : 0;
    }
}

template <int P>
__device__ void issue_tile(const TcArgs& a, const Cursor& c, unsigned char* st, uint64_t* bar) {
    using C = TcCfg<P>;
    const int b = c.g / (a.Hkv * a.quads), kvh = (c.g / a.quads) % a.Hkv;
    const size_t row = ((size_t)b * a.Hkv + kvh) * (size_t)a.k.cap + (size_t)c.k0;
    const int nk = min(kTile, c.L - c.k0);
    const uint32_t nc = (uint32_t)((nk + 7) & ~7);
    const bool qjl = a.prm.qjl != 0;
    const uint32_t bp = nc * P * 16, bs = qjl ? nc * 16 : 0u, bn = nc * 2, br = qjl ? nc * 2 : 0u;
    bar_expect_tx(bar, bp + bs + bn + br);
    bulk_copy(st, a.k.planes + row * (P * 4), bp, bar);
    if (qjl) bulk_copy(st + C::kSignOff, a.k.signs + row * 4, bs, bar);
    bulk_copy(st + C::kNormOff, a.k.norm + row, bn, bar);
    if (qjl) bulk_copy(st + C::kRnormOff, a.k.rnorm + row, br, bar);
}

struct GroupPos {
    int nh;
    size_t qrow0;
};
__device__ __forceinline__ GroupPos group_pos(const TcArgs& a, int g) {
    const int b = g / (a.Hkv * a.quads), kvh = (g / a.quads) % a.Hkv, quad = g % a.quads;
    const int hbase = kvh * a.G + 4 * quad;
    return GroupPos{min(4, kvh * a.G + a.G - hbase), (size_t)b * a.Hq + hbase};
}

// ------------------------------------------------------------------ per-group B image

template <int P>
__global__ void __launch_bounds__(128) tc_image_kernel(const TcArgs a) {
    using C = TcCfg<P>;
    constexpr int T = C::T;
    __shared__ float sq_[4][128], su_[4][128];
    __shared__ float red[4][4][4];   // [warp][head][mq, sq, mu, su]
    __shared__ int e0[2][4];
    __shared__ float sums[2][4];
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupPos gp = group_pos(a, g);
    unsigned char* img = a.img + (size_t)g * C::kImgBytes;
    for (int e = tid; e < 4 * 128; e += 128) {
        const int h = e >> 7, j = e & 127;
        sq_[h][j] = (h < gp.nh && j < prm.d) ? a.qrot[(gp.qrow0 + h) * prm.d + j] : 0.f;
        su_[h][j] = (qjl && h < gp.nh && j < prm.m) ? a.qproj[(gp.qrow0 + h) * prm.m + j] : 0.f;
    }
    __syncthreads();
    for (int h = 0; h < 4; ++h) {
        const float x = sq_[h][tid], u = su_[h][tid];
        float mq = fabsf(x), s = x, mu = fabsf(u), su = u;
        for (int o = 16; o > 0; o >>= 1) {
            mq = fmaxf(mq, __shfl_xor_sync(0xffffffffu, mq, o));
            s += __shfl_xor_sync(0xffffffffu, s, o);
            mu = fmaxf(mu, __shfl_xor_sync(0xffffffffu, mu, o));
            su += __shfl_xor_sync(0xffffffffu, su, o);
        }
        if (lane == 0) {
            red[warp][h][0] = mq;
            red[warp][h][1] = s;
            red[warp][h][2] = mu;
            red[warp][h][3] = su;
        }
    }
    __syncthreads();
    if (tid < 4) {
        const int h = tid;
        float mq = 0.f, s = 0.f, mu = 0.f, su = 0.f;
        for (int w = 0; w < 4; ++w) {
            mq = fmaxf(mq, red[w][h][0]);
            s += red[w][h][1];
            mu = fmaxf(mu, red[w][h][2]);
            su += red[w][h][3];
        }
        float kmax = 0.f;
        for (int t = 0; t < T; ++t) kmax = fmaxf(kmax, fabsf(prm.kappa[t]));
        // largest B magnitude (x 2^7) lands in [128, 256)
        e0[0][h] = column_exponent(128.f * kmax * mq);
        e0[1][h] = column_exponent(128.f * mu);
        sums[0][h] = s;
        sums[1][h] = su;
    }
    __syncthreads();
    // B bytes: (family, column n, k); k -> (term or sign vector v, word wd, register c, byte i)
    constexpr int kM = 16 * T * 128, kQ = 16 * 128;
    for (int e = tid; e < kM + kQ; e += 128) {
        const bool isq = e >= kM;
        const int ee = isq ? e - kM : e, ktot = isq ? 128 : T * 128;
        const int n = ee / ktot, kk = ee % ktot;
        const int v = kk >> 7, k = kk & 127, wd = k >> 5, c = (k >> 2) & 7, i = k & 3;
        const int j = 32 * wd + 8 * i + ((c + 2) & 7);
        const int h = n >> 2, pc = n & 3;
        const float f = (c & 1) ? 64.f : 128.f;
        const float x = isq ? su_[h][j] : prm.kappa[v] * sq_[h][j];
        const uint32_t byte = piece(x * f, e0[isq ? 1 : 0][h], pc);
        img[(isq ? kM : 0) + kmajor8(n, kk, ktot)] = (unsigned char)byte;
    }
    if (tid < 16) {
        float* cst = reinterpret_cast<float*>(img + C::kConstOff);
        const int h = tid & 3, which = tid >> 2;
        float val;
        if (which == 0) val = ldexpf(1.f, -e0[0][h]);
        else if (which == 1) val = ldexpf(1.f, -e0[1][h]);
        else if (which == 2) val = prm.c0 * sums[0][h];
        else val = -prm.qjl_scale * sums[1][h];
        cst[tid] = val;
    }
}

// ------------------------------------------------------------------ scoring

// Word wd of every bit vector of key `row` into A (the thread's TMEM lanes, column base a_tmem).
template <int P>
__device__ __forceinline__ void expand_tile(const TcArgs& a, const unsigned char* st, uint32_t a_tmem, int row,
                                            int wd) {
    using C = TcCfg<P>;
    constexpr int T = C::T;
    uint32_t pw[P];
#pragma unroll
    for (int p = 0; p < P; ++p) pw[p] = *reinterpret_cast<const uint32_t*>(st + row * (P * 16) + p * 16 + wd * 4);
#pragma unroll
    for (int v = 0; v < T; ++v) {
        uint32_t x = 0u;
#pragma unroll
        for (int p = 0; p < P; ++p)
            if ((odd_mask(v) >> p) & 1) x ^= pw[p];
        uint32_t r[8];
        expand_word(x, r);
        tmem_st8(a_tmem + (v * 4 + wd) * 8, r);
    }
    if (a.prm.qjl) {
        uint32_t r[8];
        expand_word(*reinterpret_cast<const uint32_t*>(st + C::kSignOff + row * 16 + wd * 4), r);
        tmem_st8(a_tmem + (T * 4 + wd) * 8, r);
    }
}

// Shared-memory descriptors of the B blocks read by mma warp (v, kh): K-steps wd of its share.
template <int P>
__device__ __forceinline__ void b_descs(int v, int kh, uint32_t bimg, uint64_t (&bd)[4]) {
    using C = TcCfg<P>;
    constexpr int T = C::T;
    const uint32_t bsrc = v < T ? bimg + v * 4 * 256 : bimg + C::kBmBytes;
    const uint32_t sbo = v < T ? T * 128 * 8 : 128 * 8;
#pragma unroll
    for (int k = 0; k < 4 / C::kSplit; ++k) bd[k] = smem_desc(bsrc + (kh * (4 / C::kSplit) + k) * 256, sbo);
}

// The mma of warp (v, kh) for one tile buffer: A columns of vector v, its D block.
template <int P>
__device__ __forceinline__ void issue_share(int v, int kh, uint32_t buf_tmem, const uint64_t (&bd)[4]) {
    using C = TcCfg<P>;
    constexpr int K = 4 / C::kSplit;
    const uint32_t d = buf_tmem + C::kACols + 16 * (v * C::kSplit + kh);
#pragma unroll
    for (int k = 0; k < K; ++k) mma_ts(d, buf_tmem + (v * 4 + kh * K + k) * 8, bd[k], k ? 1u : 0u);
}

// Logit of key `row` for head h of the tile's quad, from D (column base d_tmem, this thread's lanes).
// Per-group values a worker needs to finish tiles of head h.
struct FinishGroup {
    int g, nh;
    size_t qrow0;
    float fm, fq, cq, cu;   // 2^-e0 (MSE, QJL), c0 sum q', -kq sum u
};

template <int P>
__device__ __forceinline__ void finish_group(const TcArgs& a, int g, int h, FinishGroup& F) {
    using C = TcCfg<P>;
    const GroupPos gp = group_pos(a, g);
    const float* cst = reinterpret_cast<const float*>(a.img + (size_t)g * C::kImgBytes + C::kConstOff);
    F.g = g;
    F.nh = gp.nh;
    F.qrow0 = gp.qrow0;
    F.fm = __ldg(cst + h);
    F.fq = __ldg(cst + 4 + h);
    F.cq = __ldg(cst + 8 + h);
    F.cu = __ldg(cst + 12 + h);
}

// Finishing a tile is split so that its TMEM loads overlap other work: finish_load issues the
// loads of the D blocks (head h, this thread's lanes), finish_store waits for them and writes the
// logit of key `row`.
template <int P>
struct FinishRegs {
    float dm[TcCfg<P>::T * TcCfg<P>::kSplit][4];
    float dq[TcCfg<P>::kSplit][4];
};

template <int P>
__device__ __forceinline__ void finish_load(const TcArgs& a, uint32_t d_tmem, int h, FinishRegs<P>& R) {
    using C = TcCfg<P>;
    constexpr int T = C::T, KS = C::kSplit;
#pragma unroll
    for (int i = 0; i < T * KS; ++i) tmem_ld4(d_tmem + 16 * i + 4 * h, R.dm[i]);
#pragma unroll
    for (int i = 0; i < KS; ++i) {
        if (a.prm.qjl) tmem_ld4(d_tmem + 16 * (T * KS + i) + 4 * h, R.dq[i]);
        else R.dq[i][0] = R.dq[i][1] = R.dq[i][2] = R.dq[i][3] = 0.f;
    }
}

template <int P>
__device__ __forceinline__ void finish_store(const TcArgs& a, const unsigned char* st, FinishRegs<P>& R,
                                             const Cursor& c, const FinishGroup& F, int row, int h) {
    using C = TcCfg<P>;
    constexpr int T = C::T, KS = C::kSplit;
    const bool qjl = a.prm.qjl != 0;
    const float n = half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kNormOff)[row]);
    const float rho = qjl ? half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kRnormOff)[row]) : 0.f;
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 1; i < T * KS; ++i)
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) R.dm[0][pc] += R.dm[i][pc];
#pragma unroll
    for (int i = 1; i < KS; ++i)
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) R.dq[0][pc] += R.dq[i][pc];
    const int key = c.k0 + row;
    // pieces: sum_pc D[pc] 16^-pc, then the column scale 2^-e0
    const float m = F.fm * fmaf(R.dm[0][3], 1.f / 4096.f, fmaf(R.dm[0][2], 1.f / 256.f, fmaf(R.dm[0][1], 1.f / 16.f, R.dm[0][0])));
    float est = n * (F.cq + m);
    if (qjl) {
        const float qv =
            F.fq * fmaf(R.dq[0][3], 1.f / 4096.f, fmaf(R.dq[0][2], 1.f / 256.f, fmaf(R.dq[0][1], 1.f / 16.f, R.dq[0][0])));
        est = fmaf(rho, fmaf(2.f * a.prm.qjl_scale, qv, F.cu), est);
    }
    if (key < c.L && h < F.nh) a.logits[(F.qrow0 + h) * (size_t)a.k.cap + key] = a.scale * est;
}

// Position in a ring of N slots: slot and the parity of its current use.
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance() {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

struct Shared {
    uint64_t full[TcCfg<1>::kMaxStages], empty[TcCfg<1>::kMaxStages];
    uint64_t a_ready[4], d_full[4], buf_free[4];
    uint64_t img_bar, drained, drain[16];
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool aborted(const Shared& S) { return *(volatile const int*)&S.abort != 0; }
__device__ __forceinline__ void abort_all(Shared& S, int* err) {
    *(volatile int*)&S.abort = 1;
    set_error(err, TQ_DEVERR_TIMEOUT);
}

template <int P>
__global__ void __launch_bounds__(TcCfg<P>::kThreads, 1) logits_tc_kernel(const TcArgs a) {
    using C = TcCfg<P>;
    extern __shared__ __align__(1024) unsigned char sm[];
    __shared__ __align__(8) Shared S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (blockIdx.x == 0 && tid == 0)
        for (int b = 0; b < a.B; ++b)
            if (a.k.len[b] < 0 || a.k.len[b] > a.k.cap) set_error(a.err, TQ_DEVERR_LEN_RANGE);
    int64_t total = 0;
    for (int g = 0; g < a.ngroups; ++g) total += (group_len(a, g) + kTile - 1) / kTile;
    const int64_t lo = total * blockIdx.x / gridDim.x, hi = total * (blockIdx.x + 1) / gridDim.x, n = hi - lo;
    if (n <= 0) return;   // uniform over the CTA, before any allocation

    unsigned char* img_buf = sm + C::kImgOff;
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) {
            bar_init_n(&S.full[s], 1);
            bar_init_n(&S.empty[s], kWorkers);
        }
        for (int b = 0; b < C::kNB; ++b) {
            bar_init_n(&S.a_ready[b], kWorkers);
            bar_init_n(&S.d_full[b], C::NI);
            bar_init_n(&S.buf_free[b], kWorkers);
        }
        bar_init_n(&S.img_bar, 1);
        bar_init_n(&S.drained, C::NI);
        for (int v = 0; v < C::NI; ++v) bar_init_n(&S.drain[v], 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kProducerWarp + 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&S.tmem)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = S.tmem;
    bool drained = true;

    if (warp == kProducerWarp) {
        if (lane == 0) {
            Cursor c = seek(a, lo);
            Ring<C::kStages> r;
            int64_t t = 0;
            for (; t < n && !aborted(S); ++t) {
                // a stage's previous tile must be finished (its empty phase) before the refill
                if (t >= C::kStages && !bar_wait(&S.empty[r.slot], r.phase ^ 1u)) {
                    abort_all(S, a.err);
                    break;
                }
                issue_tile<P>(a, c, sm + r.slot * C::kStageBytes, &S.full[r.slot]);
                next_tile(a, c);
                r.advance();
            }
            // let every copy issued land before the CTA can leave (the last one of each stage)
            for (int k = 0; k < C::kStages && k < t; ++k) {
                // stage r.slot - 1 - k holds tile t - 1 - k; its full phase is that tile's use
                const int64_t u = t - 1 - k;
                drained &= bar_wait(&S.full[(int)(u % C::kStages)], (uint32_t)((u / C::kStages) & 1));
            }
        }
    } else if (warp > kProducerWarp) {
        const int w = warp - kProducerWarp - 1;   // mma warp: bit vector v, K share kh
        const int v = w / C::kSplit, kh = w % C::kSplit;
        if (lane == 0) {
            Cursor c = seek(a, lo);
            int cur_group = -1, nswitch = 0, ndrain = 0;
            bool issued_any = false;
            const bool active = v < C::T || a.prm.qjl;
            uint64_t bd[4];
            b_descs<P>(v, kh, smem_u32(img_buf), bd);   // the B buffer is fixed; its contents follow the group
            Ring<C::kNB> rb;
            for (int64_t i = 0; i < n && !aborted(S); ++i, rb.advance()) {
                const int b = rb.slot;
                if (c.g != cur_group) {
                    // every mma warp drains (its mma read the old B), the first one reloads B
                    bool ok = true;
                    if (nswitch > 0) {
                        if (issued_any) {
                            mma_commit(&S.drain[w]);
                            ok = bar_wait(&S.drain[w], (uint32_t)(ndrain++ & 1));
                        }
                        bar_arrive(&S.drained);
                        if (ok && w == 0) ok = bar_wait(&S.drained, (uint32_t)((nswitch - 1) & 1));
                    }
                    if (ok && w == 0) {
                        bar_expect_tx(&S.img_bar, C::kImgBytes);
                        bulk_copy(img_buf, a.img + (size_t)c.g * C::kImgBytes, C::kImgBytes, &S.img_bar);
                    }
                    if (!ok || !bar_wait(&S.img_bar, (uint32_t)(nswitch & 1))) {
                        abort_all(S, a.err);
                        break;
                    }
                    cur_group = c.g;
                    ++nswitch;
                }
                if (!bar_wait(&S.a_ready[b], rb.phase)) {
                    abort_all(S, a.err);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;");
                if (active) {
                    issue_share<P>(v, kh, tmem + b * C::kBufCols, bd);
                    issued_any = true;
                }
                mma_commit(&S.d_full[b]);
                next_tile(a, c);
            }
            if (issued_any) {   // every mma issued has completed before the CTA can leave
                mma_commit(&S.drain[w]);
                drained &= bar_wait(&S.drain[w], (uint32_t)(ndrain++ & 1));
            }
        }
    } else {
        // workers: expand tile i, finish tile i - kLag
        const int row = 32 * (warp & 3) + lane, part = warp >> 2;
        const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
        Cursor ce = seek(a, lo), cf = ce;
        FinishGroup F;
        F.g = -1;
        FinishRegs<P> R;
        Ring<C::kStages> se, sf;   // stages of the expanded and of the finished tile
        Ring<C::kNB> be, bf;       // TMEM buffers of the expanded and of the finished tile
        for (int64_t i = 0; i < n + C::kLag; ++i) {
            if (aborted(S)) break;
            const bool do_e = i < n, do_f = i >= C::kLag;
            // expand tile i: loads, ALU and TMEM stores issued, completion awaited further down
            if (do_e) {
                bool okw = bar_wait(&S.full[se.slot], se.phase);
                if (okw && i >= C::kNB) okw = bar_wait(&S.buf_free[be.slot], be.phase ^ 1u);
                if (!okw) {
                    abort_all(S, a.err);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;");
                expand_tile<P>(a, sm + se.slot * C::kStageBytes, tmem + lane_off + be.slot * C::kBufCols, row, part);
            }
            // finish tile i - kLag: its TMEM loads go out while the stores above drain
            if (do_f) {
                if (!bar_wait(&S.d_full[bf.slot], bf.phase)) {
                    abort_all(S, a.err);
                    break;
                }
                asm volatile("tcgen05.fence::after_thread_sync;");
                finish_load<P>(a, tmem + lane_off + bf.slot * C::kBufCols + C::kACols, part, R);
            }
            if (do_e) {
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0) bar_arrive(&S.a_ready[be.slot]);
                next_tile(a, ce);
                se.advance();
                be.advance();
            }
            if (do_f) {
                if (cf.g != F.g) finish_group<P>(a, cf.g, part, F);
                finish_store<P>(a, sm + sf.slot * C::kStageBytes, R, cf, F, row, part);
                asm volatile("tcgen05.fence::before_thread_sync;");
                __syncwarp();
                if (lane == 0) {
                    bar_arrive(&S.buf_free[bf.slot]);
                    bar_arrive(&S.empty[sf.slot]);
                }
                next_tile(a, cf);
                sf.advance();
                bf.advance();
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    const bool ok = __syncthreads_and(drained && !aborted(S)) != 0;
    if (!ok) {
        if (!__syncthreads_and(drained)) return;   // something may still write TMEM or shared memory
    }
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == kProducerWarp + 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
}

template <int P>
cudaError_t run_tc(const TcArgs& a, int device, cudaStream_t s) {
    using C = TcCfg<P>;
    static int grid = 0;
    if (!grid) {
        cudaError_t e = cudaFuncSetAttribute(logits_tc_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
        if (e != cudaSuccess) return e;
        int sms = 148;
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
        grid = sms;   // one CTA per SM: each allocates all 512 TMEM columns
    }
    tc_image_kernel<P><<<a.ngroups, 128, 0, s>>>(a);
    logits_tc_kernel<P><<<grid, C::kThreads, C::kSmem, s>>>(a);
    return cudaGetLastError();
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool logits_tc_supported(const tq_ctx* kc) {
    const Params& p = kc->prm;
    return p.W == 4 && (!p.qjl || p.Ws == 4) && p.odd_walsh && p.P >= 1 && p.P <= 3;
}

bool logits_tc_ok(const tq_ctx* kc, const KeyCache& k) {
    const bool qjl = kc->prm.qjl != 0;
    return logits_tc_supported(kc) && k.cap % 8 == 0 && aligned16(k.planes) && aligned16(k.norm) &&
           (!qjl || (aligned16(k.signs) && aligned16(k.rnorm)));
}

size_t logits_tc_image_bytes(int B, int Hq, int Hkv) {
    const int quads = (Hq / Hkv + 3) / 4;
    return (size_t)B * Hkv * quads * TcCfg<3>::kImgBytes;
}

cudaError_t launch_logits_tc(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                             const KeyCache& k, float scale, float* logits, void* image, cudaStream_t s) {
    TcArgs a{};
    a.prm = kc->prm;
    a.qrot = qrot;
    a.qproj = qproj;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.quads = (a.G + 3) / 4;
    a.ngroups = B * Hkv * a.quads;
    a.k = k;
    a.scale = scale;
    a.logits = logits;
    a.img = static_cast<unsigned char*>(image);
    a.err = kc->derr;
    switch (kc->prm.P) {
        case 1: return run_tc<1>(a, kc->device, s);
        case 2: return run_tc<2>(a, kc->device, s);
        case 3: return run_tc<3>(a, kc->device, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
