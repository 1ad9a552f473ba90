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
// One CTA per SM owns a contiguous range of 128-key tiles.  Tile i goes to worker group i % 4;
// the groups run independently and meet the shared producer only at mbarriers (every wait is
// bounded; a timeout sets TQ_DEVERR_TIMEOUT and stops every role):
//   per group (128 TMEM columns: two 32-column A slots and two 32-column D buffers, and a
//   ring of shared-memory stages)
//     4 worker warps  warp q owns keys 32 q .. 32 q + 31 of the group's tiles (its TMEM lanes):
//                  it expands the tile's bit vectors one at a time into the next free A slot,
//                  then finishes the group's previous tile from its D buffer into logits;
//     1 mma warp   bulk asynchronous copies of the group's tiles (one per field: planes, signs,
//                  norms, residual norms; lengths rounded up to 8 keys, inside the cache since
//                  its capacity is a multiple of 8) into the stage ring, refilling a stage once
//                  the workers have released the tile two back (its D buffer, hence its stage);
//                  per bit vector 4 tcgen05.mma (K = 32) from the slot into the tile's D (16
//                  MSE columns, the T terms accumulating, and 16 QJL columns), a commit that
//                  frees the slot when they complete, and per tile a commit that fills D.
//                  Issue costs its thread ~70 cycles per mma, so four groups issue in parallel.
//                  At a change of (batch, KV head, quad) it drains its mma and loads the
//                  group's B image into its own buffer.
#include "mma_e4m3.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kTile = 128;
constexpr int kGroups = 4;                        // worker groups (tiles in flight x2)
constexpr int kWorkerWarps = 4 * kGroups;         // warps 0..15: group w / 4, lanes 32 (w % 4)
constexpr int kMmaWarp0 = kWorkerWarps;           // warps 16..19: the groups' mma (and copy) warps
constexpr int kThreads = (kMmaWarp0 + kGroups) * 32;
constexpr int kGroupCols = 128;                   // TMEM columns per group
constexpr int kSuspendNs = 20000;     // suspend-time hint of one try_wait
constexpr int kWaitLimit = 1 << 16;   // tries before a wait gives up (bounded by ~1.3 s)

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
    static constexpr int kMaxStages = 8;        // per group
    // each group's stage ring fills its share of what the images leave of ~200 KB (one CTA and
    // its 512 TMEM columns per SM)
    static constexpr int kStagesFit = (200 * 1024 - kGroups * kImgBytes) / (kGroups * kStageBytes);
    static constexpr int kStages = kStagesFit > kMaxStages ? kMaxStages : kStagesFit;
    static constexpr int kImgOff = kGroups * kStages * kStageBytes;
    static constexpr int kSmem = kImgOff + kGroups * kImgBytes;
    static_assert(kStageBytes % 128 == 0, "stage alignment");
    static_assert(kStages >= 3, "the producer must run ahead of the finish");
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

// One bit vector into the 32 columns of an A slot: word wd -> columns 8 wd .. 8 wd + 7.
__device__ __forceinline__ void expand_vector(const uint4& x, uint32_t slot_tmem) {
    uint32_t r[8];
    expand_word(x.x, r);
    tmem_st8(slot_tmem, r);
    expand_word(x.y, r);
    tmem_st8(slot_tmem + 8, r);
    expand_word(x.z, r);
    tmem_st8(slot_tmem + 16, r);
    expand_word(x.w, r);
    tmem_st8(slot_tmem + 24, r);
}

// Per-group values a worker needs to finish tiles.
struct FinishGroup {
    int g, nh;
    size_t qrow0;
    const float4* c;   // 2^-e0 (MSE) x4, 2^-e0 (QJL) x4, c0 sum q' x4, -kq sum u x4 (shared memory)
};

// Called by a whole warp: the group's position and its 16 epilogue constants into the warp's
// own shared-memory slot.
template <int P>
__device__ __forceinline__ void finish_group(const TcArgs& a, int g, float* warp_cst, FinishGroup& F) {
    using C = TcCfg<P>;
    const GroupPos gp = group_pos(a, g);
    F.g = g;
    F.nh = gp.nh;
    F.qrow0 = gp.qrow0;
    const int lane = threadIdx.x & 31;
    __syncwarp();   // every lane is done with the previous group's constants
    if (lane < 16) warp_cst[lane] = __ldg(reinterpret_cast<const float*>(a.img + (size_t)g * C::kImgBytes + C::kConstOff) + lane);
    __syncwarp();
    F.c = reinterpret_cast<const float4*>(warp_cst);
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

// Logits of key `row` for the 4 heads of the tile's quad from its D buffer.
template <int P>
__device__ __forceinline__ void finish_tile(const TcArgs& a, const unsigned char* st, uint32_t d_tmem,
                                            const Cursor& c, const FinishGroup& F, int row) {
    using C = TcCfg<P>;
    const bool qjl = a.prm.qjl != 0;
    float dm[16], dq[16];
    tmem_ld16(d_tmem, dm);
    if (qjl) tmem_ld16(d_tmem + 16, dq);
    const float n = half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kNormOff)[row]);
    const float rho = qjl ? half_bits_to_float(reinterpret_cast<const uint16_t*>(st + C::kRnormOff)[row]) : 0.f;
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
    const int key = c.k0 + row;
    if (key >= c.L) return;
    const float k2 = 2.f * a.prm.qjl_scale;
    const float4 fm4 = F.c[0], fq4 = F.c[1], cq4 = F.c[2], cu4 = F.c[3];
    const float fm[4] = {fm4.x, fm4.y, fm4.z, fm4.w}, fq[4] = {fq4.x, fq4.y, fq4.z, fq4.w};
    const float cq[4] = {cq4.x, cq4.y, cq4.z, cq4.w}, cu[4] = {cu4.x, cu4.y, cu4.z, cu4.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        // pieces: sum_pc D[pc] 16^-pc, then the column scale 2^-e0
        const float m = fm[h] * fmaf(dm[4 * h + 3], 1.f / 4096.f,
                                     fmaf(dm[4 * h + 2], 1.f / 256.f, fmaf(dm[4 * h + 1], 1.f / 16.f, dm[4 * h])));
        float est = n * (cq[h] + m);
        if (qjl) {
            const float qv = fq[h] * fmaf(dq[4 * h + 3], 1.f / 4096.f,
                                          fmaf(dq[4 * h + 2], 1.f / 256.f, fmaf(dq[4 * h + 1], 1.f / 16.f, dq[4 * h])));
            est = fmaf(rho, fmaf(k2, qv, cu[h]), est);
        }
        if (h < F.nh) a.logits[(F.qrow0 + h) * (size_t)a.k.cap + key] = a.scale * est;
    }
}

// Position in a ring of N slots: slot and the parity of its current use; `step` slots per move.
template <int N>
struct Ring {
    int slot = 0;
    uint32_t phase = 0;
    __device__ __forceinline__ void advance(int step = 1) {
        slot += step;
        if (slot >= N) {
            slot -= N;
            phase ^= 1u;
        }
    }
};

struct Group {
    uint64_t full[8];   // the group's stage ring
    uint64_t slot_ready[2], slot_free[2], d_full[2], d_free[2], img_bar, drain_bar;
};

struct Shared {
    Group grp[kGroups];
    float cst[kWorkerWarps][16];   // per worker warp: the epilogue constants of its current group
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool aborted(const Shared& S) { return *(volatile const int*)&S.abort != 0; }
__device__ __forceinline__ void abort_all(Shared& S, int* err) {
    *(volatile int*)&S.abort = 1;
    set_error(err, TQ_DEVERR_TIMEOUT);
}

template <int P>
__global__ void __launch_bounds__(kThreads, 1) logits_tc_kernel(const TcArgs a) {
    using C = TcCfg<P>;
    constexpr int T = C::T;
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
    const bool qjl = a.prm.qjl != 0;
    const int nv = qjl ? C::NV : T;   // bit vectors scored per key

    if (tid == 0) {
        for (int g = 0; g < kGroups; ++g) {
            Group& G = S.grp[g];
            for (int s = 0; s < C::kStages; ++s) bar_init_n(&G.full[s], 1);
            for (int k = 0; k < 2; ++k) {
                bar_init_n(&G.slot_ready[k], 4);
                bar_init_n(&G.slot_free[k], 1);
                bar_init_n(&G.d_full[k], 1);
                bar_init_n(&G.d_free[k], 4);
            }
            bar_init_n(&G.img_bar, 1);
            bar_init_n(&G.drain_bar, 1);
        }
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(smem_u32(&S.tmem)));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = S.tmem;
    bool drained = true;

    if (warp >= kMmaWarp0) {
        const int g = warp - kMmaWarp0;
        Group& G = S.grp[g];
        if (lane == 0 && g < n) {
            Cursor c = seek(a, lo + g);
            unsigned char* img = sm + C::kImgOff + g * C::kImgBytes;
            const uint32_t bimg = smem_u32(img);
            const uint32_t base = tmem + g * kGroupCols;
            // B descriptors: the buffer is fixed (its contents follow the group); a K step of 32
            // bytes is +256 B of start address, +16 in the descriptor's 16-byte address field
            const uint64_t bm0 = smem_desc(bimg, T * 128 * 8), bq0 = smem_desc(bimg + C::kBmBytes, 128 * 8);
            int cur_group = -1, nimg = 0, ndrain = 0;
            bool issued_any = false;
            Ring<2> sa, db;
            // copies: the group's first kStages tiles now, then one refill per tile
            unsigned char* ring = sm + g * C::kStages * C::kStageBytes;
            const int64_t ntiles = (n - g + kGroups - 1) / kGroups;
            Cursor cp = c;
            Ring<C::kStages> rp;
            int64_t copied = 0;
            for (; copied < ntiles && copied < C::kStages; ++copied) {
                issue_tile<P>(a, cp, ring + rp.slot * C::kStageBytes, &G.full[rp.slot]);
                for (int s = 0; s < kGroups; ++s) next_tile(a, cp);
                rp.advance();
            }
            int64_t k = 0;   // the group's tile count
            for (int64_t i = g; i < n && !aborted(S); i += kGroups, ++k) {
                if (c.g != cur_group) {   // drain the mma that read the old B, then load this group's
                    bool ok = true;
                    if (issued_any) {
                        mma_commit(&G.drain_bar);
                        ok = bar_wait(&G.drain_bar, (uint32_t)(ndrain++ & 1));
                    }
                    if (ok) {
                        bar_expect_tx(&G.img_bar, C::kImgBytes);
                        bulk_copy(img, a.img + (size_t)c.g * C::kImgBytes, C::kImgBytes, &G.img_bar);
                        ok = bar_wait(&G.img_bar, (uint32_t)(nimg++ & 1));
                    }
                    if (!ok) {
                        abort_all(S, a.err);
                        break;
                    }
                    cur_group = c.g;
                }
                if (k >= 2) {
                    if (!bar_wait(&G.d_free[db.slot], db.phase ^ 1u)) {
                        abort_all(S, a.err);
                        break;
                    }
                    // tile k - 2 is finished: its stage takes the next tile
                    if (copied < ntiles) {
                        issue_tile<P>(a, cp, ring + rp.slot * C::kStageBytes, &G.full[rp.slot]);
                        for (int s = 0; s < kGroups; ++s) next_tile(a, cp);
                        rp.advance();
                        ++copied;
                    }
                }
                const uint32_t d = base + 64 + 32 * db.slot;
                bool ok = true;
#pragma unroll
                for (int v = 0; v < C::NV; ++v) {
                    if (v == T && !qjl) break;
                    if (!bar_wait(&G.slot_ready[sa.slot], sa.phase)) {
                        ok = false;
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;");
                    const uint32_t a_t = base + 32 * sa.slot;
                    const uint32_t dd = v < T ? d : d + 16;
                    const uint64_t b0 = v < T ? bm0 + (uint64_t)(v * 4 * 16) : bq0;
#pragma unroll
                    for (int wd = 0; wd < 4; ++wd)
                        mma_ts(dd, a_t + 8 * wd, b0 + (uint64_t)(wd * 16), (wd == 0 && (v == 0 || v == T)) ? 0u : 1u);
                    mma_commit(&G.slot_free[sa.slot]);
                    issued_any = true;
                    sa.advance();
                }
                if (!ok) {
                    abort_all(S, a.err);
                    break;
                }
                mma_commit(&G.d_full[db.slot]);
                db.advance();
                for (int s = 0; s < kGroups; ++s) next_tile(a, c);
            }
            if (issued_any) {   // every mma issued has completed before the CTA can leave
                mma_commit(&G.drain_bar);
                drained &= bar_wait(&G.drain_bar, (uint32_t)(ndrain++ & 1));
            }
            // and every copy issued has landed (the last use of each stage)
            for (int j = 0; j < C::kStages && j < copied; ++j) {
                const int64_t u = copied - 1 - j;
                drained &= bar_wait(&G.full[(int)(u % C::kStages)], (uint32_t)((u / C::kStages) & 1));
            }
        }
    } else {
        // worker warp: group g, keys (TMEM lanes) 32 q .. 32 q + 31
        const int g = warp >> 2, q = warp & 3, row = 32 * q + lane;
        Group& G = S.grp[g];
        const unsigned char* ring = sm + g * C::kStages * C::kStageBytes;
        const uint32_t lane_off = (uint32_t)(32 * q) << 16;
        const uint32_t base = tmem + lane_off + g * kGroupCols;
        if (g < n) {
            Cursor ce = seek(a, lo + g), cf = ce;
            FinishGroup F;
            F.g = -1;
            Ring<C::kStages> se, sf;
            Ring<2> sa, db;
            int64_t u = 0;   // A slot uses so far
            const int64_t ntiles = (n - g + kGroups - 1) / kGroups;   // this group's tiles
            for (int64_t k = 0; k <= ntiles; ++k) {
                if (aborted(S)) break;
                if (k < ntiles) {   // expand tile k: one bit vector per A slot
                    bool okw = bar_wait(&G.full[se.slot], se.phase);
                    uint4 x[C::NV];
                    if (okw) load_vectors<P>(ring + se.slot * C::kStageBytes, row, qjl, x);
#pragma unroll
                    for (int v = 0; v < C::NV; ++v) {
                        if (!okw || (v == T && !qjl)) break;
                        // the slot's previous vector must be consumed by its mma
                        if (u >= 2) okw = bar_wait(&G.slot_free[sa.slot], sa.phase ^ 1u);
                        if (!okw) break;
                        asm volatile("tcgen05.fence::after_thread_sync;");
                        expand_vector(x[v], base + 32 * sa.slot);
                        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
                        asm volatile("tcgen05.fence::before_thread_sync;");
                        __syncwarp();
                        if (lane == 0) bar_arrive(&G.slot_ready[sa.slot]);
                        sa.advance();
                        ++u;
                    }
                    if (!okw) {
                        abort_all(S, a.err);
                        break;
                    }
                    for (int s = 0; s < kGroups; ++s) next_tile(a, ce);
                    se.advance();
                }
                if (k >= 1) {   // finish tile k - 1
                    if (!bar_wait(&G.d_full[db.slot], db.phase)) {
                        abort_all(S, a.err);
                        break;
                    }
                    asm volatile("tcgen05.fence::after_thread_sync;");
                    if (cf.g != F.g) finish_group<P>(a, cf.g, S.cst[warp], F);
                    finish_tile<P>(a, ring + sf.slot * C::kStageBytes, base + 64 + 32 * db.slot, cf, F, row);
                    asm volatile("tcgen05.fence::before_thread_sync;");
                    __syncwarp();
                    if (lane == 0) bar_arrive(&G.d_free[db.slot]);   // frees D and the tile's stage
                    db.advance();
                    for (int s = 0; s < kGroups; ++s) next_tile(a, cf);
                    sf.advance();
                }
            }
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    const bool ok = __syncthreads_and(drained && !aborted(S)) != 0;
    if (!ok) {
        if (!__syncthreads_and(drained)) return;   // something may still write TMEM or shared memory
    }
    asm volatile("tcgen05.fence::after_thread_sync;");
    if (warp == kMmaWarp0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
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
    logits_tc_kernel<P><<<grid, kThreads, C::kSmem, s>>>(a);
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
