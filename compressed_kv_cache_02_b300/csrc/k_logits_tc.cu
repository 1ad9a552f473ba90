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
#include "tcgen05.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kTile = 128;
constexpr uint32_t kIdesc = tc::idesc_e4m3(16);   // M 128, N 16 (4 heads x 4 pieces), K 32

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
    __shared__ __align__(16) unsigned char img[C::kImgBytes];   // built here, then copied out whole
    const Params& prm = a.prm;
    const bool qjl = prm.qjl != 0;
    const int g = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const GroupPos gp = group_pos(a, g);
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
    // B bytes: (family, head h, k) -> its 4 pieces (one chain) in columns 4 h .. 4 h + 3;
    // k -> (term or sign vector v, word wd, register c, byte i)
    constexpr int kM = 16 * T * 128, kMk = T * 128;
    for (int e = tid; e < 4 * (kMk + 128); e += 128) {
        const bool isq = e >= 4 * kMk;
        const int ee = isq ? e - 4 * kMk : e, ktot = isq ? 128 : kMk;
        const int h = ee / ktot, kk = ee % ktot;
        const int v = kk >> 7, k = kk & 127, wd = k >> 5, c = (k >> 2) & 7, i = k & 3;
        const int j = 32 * wd + 8 * i + ((c + 2) & 7);
        const float f = (c & 1) ? 64.f : 128.f;
        const float val = isq ? su_[h][j] : prm.kappa[v] * sq_[h][j];
        float x = ldexpf(val * f, e0[isq ? 1 : 0][h]);   // pieces b0 + b1/16 + b2/256 + b3/4096
        unsigned char* fam = img + (isq ? kM : 0);
#pragma unroll
        for (int pc = 0; pc < 4; ++pc) {
            const uint32_t b = to_e4m3(x);
            fam[tc::kmajor8(4 * h + pc, kk, ktot)] = (unsigned char)b;
            x = (x - from_e4m3(b)) * 16.f;
        }
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
    __syncthreads();
    uint4* out = reinterpret_cast<uint4*>(a.img + (size_t)g * C::kImgBytes);
    for (int e = tid; e < C::kImgBytes / 16; e += 128) out[e] = reinterpret_cast<const uint4*>(img)[e];
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

// ------------------------------------------------------------------ scoring, one CTA per chunk

constexpr int kT2Threads = 128;
constexpr int kT2ChunkMax = 2048;

template <int P>
struct Tc2Cfg {
    using C = TcCfg<P>;
    static constexpr int kACols = 32 * C::NV;                       // A: one 32-column slot per vector
    static constexpr int kBufCols = kACols + 32;                    // A and D (16 MSE + 16 QJL columns)
    static constexpr int kTmemCols = kBufCols <= 128 ? 128 : 256;
    static constexpr int kStageOff = C::kImgBytes;                  // B image, then two code stages
    static constexpr int kSmemUsed = kStageOff + 2 * C::kStageBytes;
    // dynamic shared memory requested: caps the CTAs per SM at 512 / kTmemCols
    static constexpr int kSmem = kTmemCols == 128 ? 52 * 1024 : 100 * 1024;
    static_assert(kSmemUsed <= kSmem, "shared memory layout");
};

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
    static_assert(kT2Threads >= kTile && kT2Threads >= 48, "one thread per sign row; norms by warps 0 and 1");
    const int t = threadIdx.x;
    for (int e = t; e < npl; e += kT2Threads) tc::cp_async16(st + 16 * e, pl + e);
    if (t < nsg) tc::cp_async16(st + C::kSignOff + 16 * t, sg + t);   // nsg <= kTile = kT2Threads
    if (t < nn) tc::cp_async16(st + C::kNormOff + 16 * t, nm + t);
    else if (t - 32 >= 0 && t - 32 < nr) tc::cp_async16(st + C::kRnormOff + 16 * (t - 32), rn + (t - 32));
    asm volatile("cp.async.commit_group;");
}

template <int P>
__global__ void __launch_bounds__(kT2Threads) logits_tc_kernel(const TcArgs a, int chunk) {
    using C = TcCfg<P>;
    using K2 = Tc2Cfg<P>;
    constexpr int T = C::T;
    extern __shared__ __align__(128) unsigned char sm[];
    unsigned char* img = sm;
    unsigned char* stages = sm + K2::kStageOff;
    __shared__ __align__(8) uint64_t s_mma, s_drain;   // the latest tile's MMAs are done; all MMAs are done
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
        tc::cp_async16(img + 16 * e, a.img + (size_t)g * C::kImgBytes + 16 * e);
    stage_codes<P>(a, row0, min(kTile, nkeys), stages, qjl);
    if (tid == 0) {
        tc::mbar_init(&s_mma, 1);
        tc::mbar_init(&s_drain, 1);
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc<K2::kTmemCols>(&s_tmem);
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_tmem = tmem + ((uint32_t)(32 * warp) << 16);
    const uint32_t bimg = tc::smem_u32(img);
    const uint64_t bm0 = tc::kmajor_desc(bimg, T * 128 * 8), bq0 = tc::kmajor_desc(bimg + C::kBmBytes, 128 * 8);
    const float k2 = 2.f * a.prm.qjl_scale;
    float* lrow = a.logits + gp.qrow0 * (size_t)a.k.cap + (size_t)i0;   // logits of this chunk's first key, head 0
    float cst[16];
    // this thread's key of the tile in flight: norm, residual norm, index (-1: none)
    float pn = 0.f, pr = 0.f;
    int pkey = -1;
    bool ok = true;

    // logits of this thread's key of the tile whose MMAs are done
    auto finish = [&]() {
        const uint32_t d = lane_tmem + (uint32_t)K2::kACols;
        float dm[16], dq[16];
        tc::tmem_ld16(d, dm);
        if (qjl) tc::tmem_ld16(d + 16, dq);
        tc::wait_ld();
        if (pkey < 0) return;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const float m = cst[h] * fmaf(dm[4 * h + 3], 1.f / 4096.f,
                                          fmaf(dm[4 * h + 2], 1.f / 256.f, fmaf(dm[4 * h + 1], 1.f / 16.f, dm[4 * h])));
            float est = pn * (cst[8 + h] + m);
            if (qjl) {
                const float qv = cst[4 + h] * fmaf(dq[4 * h + 3], 1.f / 4096.f,
                                                   fmaf(dq[4 * h + 2], 1.f / 256.f, fmaf(dq[4 * h + 1], 1.f / 16.f, dq[4 * h])));
                est = fmaf(pr, fmaf(k2, qv, cst[12 + h]), est);
            }
            if (h < gp.nh) lrow[(size_t)h * a.k.cap + pkey] = a.scale * est;
        }
    };
    // waits (every thread, CTA-uniform outcome) for the MMAs of tile t
    auto wait_tile = [&](int t) -> bool {
        const bool w = tc::mbar_wait(&s_mma, (uint32_t)(t & 1));
        if (!__syncthreads_and(w)) return false;
        tc::fence_after();
        return true;
    };

    for (int t = 0; t < ntile; ++t) {
        unsigned char* st = stages + (t & 1) * C::kStageBytes;
        if (t + 1 < ntile)
            stage_codes<P>(a, row0 + (size_t)(t + 1) * kTile, min(kTile, nkeys - (t + 1) * kTile),
                           stages + ((t + 1) & 1) * C::kStageBytes, qjl);
        else
            asm volatile("cp.async.commit_group;");
        asm volatile("cp.async.wait_group 1;");
        tc::fence_proxy_async();   // the image is read by the tensor cores
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
        // A and D are reused: wait for tile t - 1's MMAs, finish it
        if (t >= 1) {
            if (!wait_tile(t - 1)) {
                ok = false;
                break;
            }
            finish();
        }
#pragma unroll
        for (int v = 0; v < C::NV; ++v) {
            if (v == T && !qjl) break;
            const uint32_t w4[4] = {x[v].x, x[v].y, x[v].z, x[v].w};
            tc::store_bits<4>(lane_tmem + 32 * v, w4);
        }
        tc::wait_st();
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after();
            const uint32_t dm_t = tmem + K2::kACols, dq_t = dm_t + 16;
#pragma unroll
            for (int v = 0; v < T; ++v)
#pragma unroll
                for (int wd = 0; wd < 4; ++wd)
                    tc::mma_e4m3_ts<kIdesc>(dm_t, tmem + 32 * v + 8 * wd, bm0 + (uint64_t)((v * 4 + wd) * 16),
                                            (v == 0 && wd == 0) ? 0u : 1u);
            if (qjl) {
#pragma unroll
                for (int wd = 0; wd < 4; ++wd)
                    tc::mma_e4m3_ts<kIdesc>(dq_t, tmem + 32 * T + 8 * wd, bq0 + (uint64_t)(wd * 16), wd == 0 ? 0u : 1u);
            }
            tc::commit(&s_mma);
        }
        pn = n;
        pr = rho;
        pkey = valid ? key : -1;
    }
    asm volatile("cp.async.wait_all;");
    if (ok) {
        ok = wait_tile(ntile - 1);
        if (ok) finish();
    }
    bool drained = true;
    if (!ok) {   // a wait ran out: flag it, and let every MMA this CTA issued finish (bounded)
        if (tid == 0) {
            set_error(a.err, TQ_DEVERR_TIMEOUT);
            tc::commit(&s_drain);
        }
        drained = __syncthreads_and(tid != 0 || tc::mbar_wait(&s_drain, 0u));
    }
    tc::fence_before();
    __syncthreads();
    // an MMA that outlived the bounded drain still writes this memory: it is then left allocated
    if (warp == 0 && drained) tc::tmem_dealloc<K2::kTmemCols>(tmem);
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
