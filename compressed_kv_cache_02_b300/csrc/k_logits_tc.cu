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
//   coordinates; one 32-column tcgen05.st writes a bit vector (4 k per 32-bit column).
// B (K x 16 columns, shared memory, K-major no-swizzle core matrices): column 4 h + pc is piece
//   pc of query head h, value x 2^(e0_h) x (2^7 or 2^6, undoing the A scale); four e4m3 pieces
//   x = b0 + b1/16 + b2/256 + b3/4096 carry ~16 bits.  Built once per group by
//   tc_image_kernel, with the epilogue constants, and copied into shared memory per CTA.
// D (fp32, TMEM): 16 MSE columns (the T terms accumulate) and 16 QJL columns.
//
// logits_tc_kernel: a CTA of 4 warps owns a chunk of keys of one (batch, KV head, head quad) and
// walks it in tiles of 128 keys, one key per thread (= TMEM lane).  Per tile: the next tile's codes
// are copied (cp.async) into the other of two stages; each thread builds its key's bit vectors,
// waits until the previous tile's MMAs are done, finishes that tile from D (its previous key's
// logits), expands the new vectors into A and, after one CTA barrier, one thread issues the tile's
// mma (4 per bit vector) and a commit.  A (32 columns per vector) and D (32 columns) fit 128 TMEM
// columns (256 at 3 MSE bits), so up to 4 (2) CTAs share an SM and interleave their tiles on the
// tensor pipe: the small mma (N = 16) are bound by the issue rate of the tensor pipe (about one
// per 32 cycles per SM measured), not by its arithmetic.  Every wait is bounded in time; one that
// runs out sets TQ_DEVERR_TIMEOUT.
#include "mma_e4m3.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kTile = 128;
constexpr int kSuspendNs = 20000;                 // suspend-time hint of one try_wait
constexpr uint64_t kWaitNs = 1000000000ull;       // a wait gives up after one second

template <int P>
struct TcCfg {
    static constexpr int T = 1 << (P - 1);      // Walsh terms
    static constexpr int NV = T + 1;            // bit vectors per key (terms, then signs)
    static constexpr int kSignOff = kTile * P * 16;
    static constexpr int kNormOff = kSignOff + kTile * 16;
    static constexpr int kRnormOff = kNormOff + kTile * 2;
    static constexpr int kStageBytes = kRnormOff + kTile * 2;
    static constexpr int kBmBytes = 16 * T * 128;   // MSE B: 16 columns x T*128 k
    static constexpr int kBqBytes = 16 * 128;       // QJL B: 16 columns x 128 k
    static constexpr int kConstOff = kBmBytes + kBqBytes;
    static constexpr int kImgBytes = (kConstOff + 64 + 127) / 128 * 128;
    static_assert(kStageBytes % 128 == 0, "stage alignment");
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

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity to complete.  Each try_wait may suspend the thread
// for up to kSuspendNs (it resumes as soon as the phase completes); false once kWaitNs of
// wall-clock time (the GPU's global timer) have passed.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
    const uint64_t t0 = global_ns();
    for (;;) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
            : "=r"(done)
            : "r"(smem_u32(bar)), "r"(parity), "n"(kSuspendNs)
            : "memory");
        if (done) return true;
        if (global_ns() - t0 > kWaitNs) return false;
    }
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

// The tile's bit vectors of key `row`: the T Walsh terms (XOR of their planes), then the signs.
template <int P>
__device__ __forceinline__ void load_vectors(const unsigned char* st, int row, bool qjl, uint4 (&x)[TcCfg<P>::NV]) {
    using C = TcCfg<P>;
    constexpr int T = C::T;
    uint4 pl[P];
#pragma unroll
    for (int p = 0; p < P; ++p) pl[p] = *reinterpret_cast<const uint4*>(st + row * (P * 16) + p * 16);
#pragma unroll
    for (int v = 0; v < T; ++v) {
        x[v] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int p = 0; p < P; ++p)
            if ((odd_mask(v) >> p) & 1) {
                x[v].x ^= pl[p].x;
                x[v].y ^= pl[p].y;
                x[v].z ^= pl[p].z;
                x[v].w ^= pl[p].w;
            }
    }
    x[T] = qjl ? *reinterpret_cast<const uint4*>(st + C::kSignOff + row * 16) : make_uint4(0u, 0u, 0u, 0u);
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// ------------------------------------------------------------------ scoring, one CTA per chunk

constexpr int kT2Threads = 128;
constexpr int kT2ChunkMax = 2048;

#ifndef TQ_LOGITS_TC_BUFFERS
#define TQ_LOGITS_TC_BUFFERS 1
#endif

template <int P>
struct Tc2Cfg {
    using C = TcCfg<P>;
    static constexpr int kACols = 32 * C::NV;                       // A: one 32-column slot per vector
    static constexpr int kBufCols = kACols + 32;                    // A and D (16 MSE + 16 QJL columns)
    // two A + D buffers where they fit 256 columns (the MMAs of one tile then overlap the next
    // tile's expansion and the finish of the one before), else one
    static constexpr int NB = (TQ_LOGITS_TC_BUFFERS >= 2 && 2 * kBufCols <= 256) ? 2 : 1;
    static constexpr int kTmemCols = (NB * kBufCols <= 128) ? 128 : 256;
    static constexpr int kStageOff = C::kImgBytes;                  // B image, then two code stages
    static constexpr int kSmemUsed = kStageOff + 2 * C::kStageBytes;
    // dynamic shared memory requested: caps the CTAs per SM at 512 / kTmemCols
    static constexpr int kSmem = kTmemCols == 128 ? 52 * 1024 : 100 * 1024;
    static_assert(kSmemUsed <= kSmem, "shared memory layout");
};

__device__ __forceinline__ void cp_async16_tc(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

// Codes of the keys [k0, k0 + nk) of the cache rows starting at `row` into a stage (TcCfg
// lays them out), 16-byte cp.async pieces, one commit group.  The norm fields are copied in whole
// 16-byte pieces (8 keys), which stay inside the cache because its capacity is a multiple of 8.
template <int P>
__device__ __forceinline__ void stage_codes(const TcArgs& a, size_t row, int nk, unsigned char* st, bool qjl) {
    using C = TcCfg<P>;
    const int npl = nk * P, nsg = qjl ? nk : 0, nn = (nk + 7) / 8, nr = qjl ? nn : 0;
    const uint4* pl = reinterpret_cast<const uint4*>(a.k.planes + row * (P * 4));
    const uint4* sg = reinterpret_cast<const uint4*>(a.k.signs + row * 4);
    const uint4* nm = reinterpret_cast<const uint4*>(a.k.norm + row);
    const uint4* rn = reinterpret_cast<const uint4*>(a.k.rnorm + row);
    for (int e = threadIdx.x; e < npl + nsg + nn + nr; e += kT2Threads) {
        if (e < npl) cp_async16_tc(st + 16 * e, pl + e);
        else if (e < npl + nsg) cp_async16_tc(st + C::kSignOff + 16 * (e - npl), sg + (e - npl));
        else if (e < npl + nsg + nn) cp_async16_tc(st + C::kNormOff + 16 * (e - npl - nsg), nm + (e - npl - nsg));
        else cp_async16_tc(st + C::kRnormOff + 16 * (e - npl - nsg - nn), rn + (e - npl - nsg - nn));
    }
    asm volatile("cp.async.commit_group;");
}

template <int P>
__global__ void __launch_bounds__(kT2Threads) logits_tc_kernel(const TcArgs a, int chunk) {
    using C = TcCfg<P>;
    using K2 = Tc2Cfg<P>;
    constexpr int T = C::T;
    constexpr int NB = K2::NB;
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* img = sm;
    unsigned char* stages = sm + K2::kStageOff;
    __shared__ __align__(8) uint64_t s_mma[NB];   // buffer u: the MMAs of its latest tile are done
    __shared__ uint32_t s_tmem;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int bh = blockIdx.y, b = bh / a.Hkv;
    const int g = bh * a.quads + blockIdx.z;   // (batch, KV head, quad) as group_pos numbers them
    const int L = checked_len(a.k.len, b, a.k.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * chunk;
    if (i0 >= L) return;
    const int nkeys = (int)(min((int64_t)L, i0 + chunk) - i0);
    const int ntile = (nkeys + kTile - 1) / kTile;
    const GroupPos gp = group_pos(a, g);
    const bool qjl = a.prm.qjl != 0;
    const size_t row0 = (size_t)bh * a.k.cap + (size_t)i0;

    for (int e = tid; e < C::kImgBytes / 16; e += kT2Threads)
        cp_async16_tc(img + 16 * e, a.img + (size_t)g * C::kImgBytes + 16 * e);
    stage_codes<P>(a, row0, min(kTile, nkeys), stages, qjl);
    if (tid == 0) {
        for (int u = 0; u < NB; ++u) bar_init_n(&s_mma[u], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "n"(K2::kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = s_tmem;
    const uint32_t lane_tmem = tmem + ((uint32_t)(32 * warp) << 16);
    const uint32_t bimg = smem_u32(img);
    const uint64_t bm0 = smem_desc(bimg, T * 128 * 8), bq0 = smem_desc(bimg + C::kBmBytes, 128 * 8);
    const float k2 = 2.f * a.prm.qjl_scale;
    float cst[16];
    // this thread's key of the tiles in flight: norm, residual norm, index (-1: none); `newer` is
    // the latest tile's, `older` the one before (two buffers)
    struct KeyState {
        float n, rho;
        int key;
    };
    KeyState older{0.f, 0.f, -1}, newer{0.f, 0.f, -1};
    bool ok = true;

    // logits of this thread's key of a tile whose MMAs (on buffer u) are done
    auto finish = [&](int u, const KeyState& ks) {
        const uint32_t d = lane_tmem + (uint32_t)(u * K2::kBufCols + K2::kACols);
        float dm[16], dq[16];
        tmem_ld16(d, dm);
        if (qjl) tmem_ld16(d + 16, dq);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        if (ks.key < 0) return;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float m = cst[h] * fmaf(dm[4 * h + 3], 1.f / 4096.f,
                                          fmaf(dm[4 * h + 2], 1.f / 256.f, fmaf(dm[4 * h + 1], 1.f / 16.f, dm[4 * h])));
            float est = ks.n * (cst[8 + h] + m);
            if (qjl) {
                const float qv = cst[4 + h] * fmaf(dq[4 * h + 3], 1.f / 4096.f,
                                                   fmaf(dq[4 * h + 2], 1.f / 256.f, fmaf(dq[4 * h + 1], 1.f / 16.f, dq[4 * h])));
                est = fmaf(ks.rho, fmaf(k2, qv, cst[12 + h]), est);
            }
            if (h < gp.nh) a.logits[(gp.qrow0 + h) * (size_t)a.k.cap + (size_t)(i0 + ks.key)] = a.scale * est;
        }
    };
    // waits (every thread, CTA-uniform outcome) for the MMAs of the tile that used buffer u last
    auto wait_buffer = [&](int u, int tile) -> bool {
        const bool w = bar_wait(&s_mma[u], (uint32_t)((tile / NB) & 1));
        if (!__syncthreads_and(w)) return false;
        asm volatile("tcgen05.fence::after_thread_sync;");
        return true;
    };

    for (int t = 0; t < ntile && ok; ++t) {
        const int u = t % NB;
        unsigned char* st = stages + (t & 1) * C::kStageBytes;
        if (t + 1 < ntile)
            stage_codes<P>(a, row0 + (size_t)(t + 1) * kTile, min(kTile, nkeys - (t + 1) * kTile),
                           stages + ((t + 1) & 1) * C::kStageBytes, qjl);
        else
            asm volatile("cp.async.commit_group;");
        asm volatile("cp.async.wait_group 1;");
        asm volatile("fence.proxy.async.shared::cta;");   // the image is read by the tensor cores
        __syncthreads();
        if (t == 0) {
#pragma unroll
            for (int i = 0; i < 16; ++i) cst[i] = reinterpret_cast<const float*>(img + C::kConstOff)[i];
        }
        // this thread's key of tile t: its bit vectors and norms
        const int key = t * kTile + tid;
        const bool valid = key < nkeys;
        uint4 x[C::NV];
        load_vectors<P>(st, tid, qjl, x);
        const float n = valid ? half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kNormOff)[tid]) : 0.f;
        const float rho = (valid && qjl) ? half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kRnormOff)[tid]) : 0.f;
        // buffer u was last used by tile t - NB: wait for its MMAs, finish it
        if (t >= NB) {
            if (!wait_buffer(u, t - NB)) {
                ok = false;
                break;
            }
            finish(u, NB == 2 ? older : newer);
        }
        const uint32_t abuf = (uint32_t)(u * K2::kBufCols);
#pragma unroll
        for (int v = 0; v < C::NV; ++v) {
            if (v == T && !qjl) break;
            uint32_t r[32];
            const uint32_t w4[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
#pragma unroll
            for (int wd = 0; wd < 4; ++wd) {
                uint32_t e8[8];
                expand_word(w4[wd], e8);
#pragma unroll
                for (int c = 0; c < 8; ++c) r[8 * wd + c] = e8[c];
            }
            tmem_st32(lane_tmem + abuf + 32 * v, r);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;");
        __syncthreads();
        if (tid == 0) {
            asm volatile("tcgen05.fence::after_thread_sync;");
            const uint32_t dm_t = tmem + abuf + K2::kACols, dq_t = dm_t + 16;
#pragma unroll
            for (int v = 0; v < T; ++v)
#pragma unroll
                for (int wd = 0; wd < 4; ++wd)
                    mma_ts(dm_t, tmem + abuf + 32 * v + 8 * wd, bm0 + (uint64_t)((v * 4 + wd) * 16),
                           (v == 0 && wd == 0) ? 0u : 1u);
            if (qjl) {
#pragma unroll
                for (int wd = 0; wd < 4; ++wd)
                    mma_ts(dq_t, tmem + abuf + 32 * T + 8 * wd, bq0 + (uint64_t)(wd * 16), wd == 0 ? 0u : 1u);
            }
            mma_commit(&s_mma[u]);
        }
        older = newer;
        newer = KeyState{n, rho, valid ? key : -1};
    }
    asm volatile("cp.async.wait_all;");
    // the tiles still in flight, oldest first
    if (ok && NB == 2 && ntile >= 2) {
        ok = wait_buffer((ntile - 2) % NB, ntile - 2);
        if (ok) finish((ntile - 2) % NB, older);
    }
    if (ok) {
        ok = wait_buffer((ntile - 1) % NB, ntile - 1);
        if (ok) finish((ntile - 1) % NB, newer);
    }
    if (!ok) {
        if (tid == 0) set_error(a.err, TQ_DEVERR_TIMEOUT);
        return;   // an MMA may still be in flight: the TMEM allocation is left to the context teardown
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(K2::kTmemCols));
}

template <int P>
cudaError_t run_tc(const TcArgs& a, cudaStream_t s) {
    using K2 = Tc2Cfg<P>;
    cudaError_t e = cudaFuncSetAttribute(logits_tc_kernel<P>, cudaFuncAttributeMaxDynamicSharedMemorySize, K2::kSmem);
    if (e != cudaSuccess) return e;
    // keys per CTA: the largest power of two in [256, kT2ChunkMax] giving two rounds of CTAs
    int chunk = kT2ChunkMax;
    while (chunk > 256 && (int64_t)a.ngroups * ((a.k.cap + chunk - 1) / chunk) < 148 * 8) chunk >>= 1;
    const int nchunk = (int)((a.k.cap + chunk - 1) / chunk);
    tc_image_kernel<P><<<a.ngroups, 128, 0, s>>>(a);
    dim3 grid(nchunk, a.B * a.Hkv, a.quads);
    logits_tc_kernel<P><<<grid, kT2Threads, K2::kSmem, s>>>(a, chunk);
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
        case 1: return run_tc<1>(a, s);
        case 2: return run_tc<2>(a, s);
        case 3: return run_tc<3>(a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
