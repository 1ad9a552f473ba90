// Bulk quantization on the 5th-generation tensor cores (tcgen05.mma, TMEM accumulators) for
// bf16 rows with d = m = 128: the dense rotation and JL projection of batched keys.
//
// Pages: juejin.cn post section 二 and csdn tutorial sections PolarQuant / QJL (rotate, code,
// residual, signs); the arithmetic is that of quantize_kernel (k_quantize.cu), only the two
// d x d products move to tensor cores:
//   phase 1  Y = X Pi^T          A = the tile's x rows (bf16, exact), B = Pi as 2 bf16 pieces
//                                (hi + mid; what they leave is below 2^-18 of each entry, so u
//                                moves by ~3e-7, far inside the 1e-5 band of the code parity
//                                rule), both accumulated into one TMEM accumulator (128 columns).
//   epilogue n = ||x||, n16, u = y / n, idx, bit planes, r' = y - n16 c[idx], ||r'||.
//   phase 2  Z = r' (S Pi^T)^T   A = r' split into bf16 hi and lo, B = S Pi^T as 2 bf16 pieces,
//                                all products but lo x the second piece into one accumulator (z
//                                moves by a few 1e-6 of ||x||, inside the 1e-5 band of the sign
//                                rule); sign_j = [z_j > 0].
// Pi and S Pi^T stay resident in shared memory (4 x 32 KB), so one CTA per SM walks the tiles of
// 128 rows.  The scalar quantizer (quantize_tc2_kernel, ordinary and split contexts) and the
// polar encoder (polar_tc2_kernel) run two 8-warp groups per CTA, each on its own tile with its
// own x buffer and TMEM accumulator, r' held in tensor memory as the phase-2 A operand, so one
// group's epilogue overlaps the other's MMAs.  Operands in shared memory use the K-major no-swizzle
// core-matrix layout (8 rows x 16 bytes per core matrix; LBO = 128 B between core matrices along
// K, SBO = 2048 B between 8-row groups).  One thread per group issues the MMAs; tcgen05.commit
// signals an mbarrier whose waits are bounded in time (TQ_DEVERR_TIMEOUT).
#include <cuda_bf16.h>

#include <cstring>
#include <vector>

#include "tcgen05.cuh"
#include "tq_device.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr int kTcThreads = 512;   // two groups of 8 warps; 2 threads per row of a group's tile, 64 coordinates each
constexpr int kTile = 128;
constexpr uint32_t kMatBytes = 128 * 128 * 2;   // one 128 x 128 bf16 operand
constexpr int kPieces = 2;                      // bf16 pieces of Pi and of S Pi^T
constexpr uint32_t kSmemB = 2 * kPieces * kMatBytes;   // Pi pieces then S Pi^T pieces (128 KB)

__host__ __device__ constexpr uint32_t kmajor_off(int r, int k) {
    return (uint32_t)(((r >> 3) * 16 + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)(2048 >> 4) << 32) |
           ((uint64_t)1 << 46);
}

// kind::f16: D f32, A and B bf16, both K-major, N = 128, M = 128
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

__device__ __forceinline__ void mma_bf16(uint32_t tmem, uint64_t da, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(tmem),
        "l"(da), "l"(db), "r"(kIdesc), "r"(accumulate));
}

// D (+)= A (B_0 + B_1)^T: 8 K-steps of 16 per piece, every step into the same accumulator.  The
// descriptors of later K-steps and pieces differ only in the start-address field (16-byte units),
// which stays below 2^14 for any shared-memory offset.
__device__ __forceinline__ void issue_pieces(uint32_t tmem, uint32_t a_saddr, uint32_t b_saddr, bool accumulate) {
    const uint64_t da = smem_desc(a_saddr), db = smem_desc(b_saddr);
#pragma unroll 1
    for (int p = 0; p < kPieces; ++p)
#pragma unroll
        for (int s = 0; s < 8; ++s)
            mma_bf16(tmem, da + (uint64_t)(s * 16), db + (uint64_t)((p * kMatBytes + s * 256) >> 4),
                     (accumulate || p > 0 || s > 0) ? 1u : 0u);
}

// The 32 coordinates [32 part, 32 part + 32) of this thread's row from the accumulator at tmem_row.
__device__ __forceinline__ void load_row_part(uint32_t tmem_row, int part, float (&y)[32]) {
    float v0[16], v1[16];
    tc::tmem_ld16(tmem_row + 32 * part, v0);
    tc::tmem_ld16(tmem_row + 32 * part + 16, v1);
    asm volatile("tcgen05.wait::ld.sync.aligned;");
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        y[j] = v0[j];
        y[16 + j] = v1[j];
    }
}

struct TcArgs {
    Params prm;
    const uint16_t* x;       // bf16 rows
    int64_t n, ld_x;
    const uint4* bops;       // 6 pre-laid-out 128 x 128 bf16 operands (Pi pieces, S Pi^T pieces)
    uint32_t* planes;
    uint32_t* signs;
    uint16_t* norm;
    uint16_t* rnorm;
    int* err;
};


// ---------------------------------------------------------------- two tiles in flight
// The CTA is split into two groups of 8 warps that each take every other tile, so one group's
// CUDA-core epilogue runs while the other group's MMAs do.  Per group: one x buffer (the next
// tile's rows are copied into it as
// soon as the current tile's Y = X Pi^T is done), a 128-column accumulator D (Y, then Z) and a
// 128-column A operand in tensor memory holding r' as bf16 hi (columns 0..63) and lo (64..127),
// so the projection Z = r' (S Pi^T)^T reads A from tensor memory (kind::f16, A in TMEM) and no
// shared-memory r' buffer is needed; the two groups use all 512 columns.  Warp w of group g owns
// TMEM lanes 32 (w % 4).. (rows) and coordinates 64 (w / 4 % 2).. in two passes of 32.
constexpr int kTc2Groups = 2;
constexpr int kTc2GThreads = kTcThreads / kTc2Groups;   // 256
constexpr uint32_t kSmemTc2 = kSmemB + kTc2Groups * kMatBytes + kTc2Groups * 4 * kTile * sizeof(float);

__device__ __forceinline__ bool group_and(bool v, int id) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "n"(kTc2GThreads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t db, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(db), "r"(kIdesc), "r"(accumulate));
}

// D = A_hi (B_0 + B_1)^T + A_lo B_0^T, A in tensor memory (8 columns per K-step of 16), B in shared
// memory.  The product left out, A_lo B_1^T, has entries below 2^-9 |r'| times 2^-9 |S Pi^T| each:
// about 2^-18 ||r'|| in z (4e-6 of ||r'||), inside the 1e-5 ||x|| band of the sign rule.
__device__ __forceinline__ void issue_pieces_ta(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_saddr) {
    const uint64_t db = smem_desc(b_saddr);
#pragma unroll 1
    for (int ap = 0; ap < 2; ++ap)
#pragma unroll 1
        for (int p = 0; p < kPieces - ap; ++p)
#pragma unroll
            for (int s = 0; s < 8; ++s)
                mma_bf16_ts(d_tmem, a_tmem + 64 * ap + 8 * s, db + (uint64_t)((p * kMatBytes + s * 256) >> 4),
                            (ap > 0 || p > 0 || s > 0) ? 1u : 0u);
}

// The x rows of `tile` into sXg (cp.async by the group's threads, zeros beyond n), one commit group.
__device__ __forceinline__ void stage_x_group(const TcArgs& a, int tile, unsigned char* sXg, int gtid) {
    const int64_t r0 = (int64_t)tile * kTile;
    const int nvalid = (int)min((int64_t)kTile, a.n - r0);
    for (int e = gtid; e < kTile * 16; e += kTc2GThreads) {
        const int r = e >> 4, kc = e & 15;
        unsigned char* dst = sXg + kmajor_off(r, 8 * kc);
        if (r < nvalid) tc::cp_async16(dst, a.x + (size_t)(r0 + r) * a.ld_x + 8 * kc);
        else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
    }
    asm volatile("cp.async.commit_group;");
}

// Codes of a thread's 32 coordinates y with an odd-symmetric NB-bit table (thr: the 2^NB - 1
// thresholds, cen: the 2^NB centroids, shared memory): a sign (y > 0, the middle threshold being 0)
// and magnitude bits of |y| against the upper half of the table, the lower planes mirrored on the
// negative side word-wise.  Each decision a > b is the sign bit of b - a (exact in sign; +0 on a
// tie), shifted into its plane word from the top, coordinate 31 first.  pw[0..NB-1] receive the
// planes, y the residual y - n16 c[idx], rs its squared norm.  The decisions agree with ordered
// comparisons except where |y| equals a threshold exactly.
template <int NB>
__device__ __forceinline__ void sym_codes(float (&y)[32], float nrm, float n16, float nv, const float* thr,
                                          const float* cen, uint32_t* pw, float& rs) {
    constexpr int H = 1 << (NB - 1);   // first index of the upper half
    uint32_t sg = 0u, mw[3] = {0u, 0u, 0u};
    if constexpr (NB == 1) {
        const float cm = cen[1];
#pragma unroll
        for (int c = 31; c >= 0; --c) {
            const float yc = nrm > 0.f ? y[c] : 0.f;
            const float dz = 0.f - yc;   // negative iff yc > 0 (+0 for yc = +-0)
            sg = __funnelshift_l(__float_as_uint(dz), sg, 1);
            const float r = fmaf(n16, copysignf(cm, dz), y[c]);   // y - n16 c, c = +-cm with the sign of yc
            y[c] = r;
            rs = fmaf(r, r, rs);
        }
    } else {
        float ts[H - 1];
#pragma unroll
        for (int k = 0; k + 1 < H; ++k) ts[k] = thr[H + k] * nv;
        float cm[NB == 4 ? 1 : H];
        if constexpr (NB < 4) {
#pragma unroll
            for (int k = 0; k < H; ++k) cm[k] = cen[H + k];
        }
#pragma unroll
        for (int c = 31; c >= 0; --c) {
            const float yc = nrm > 0.f ? y[c] : 0.f;
            const float av = fabsf(yc);
            const float dz = 0.f - yc;
            sg = __funnelshift_l(__float_as_uint(dz), sg, 1);
            float mag;
            if constexpr (NB == 2) {
                const float d0 = ts[0] - av;
                mw[0] = __funnelshift_l(__float_as_uint(d0), mw[0], 1);
                mag = d0 < 0.f ? cm[1] : cm[0];
            } else if constexpr (NB == 3) {
                const float d1 = ts[1] - av;
                const bool m1 = d1 < 0.f;
                const float d0 = (m1 ? ts[2] : ts[0]) - av;
                mw[1] = __funnelshift_l(__float_as_uint(d1), mw[1], 1);
                mw[0] = __funnelshift_l(__float_as_uint(d0), mw[0], 1);
                const bool m0 = d0 < 0.f;
                mag = m1 ? (m0 ? cm[3] : cm[2]) : (m0 ? cm[1] : cm[0]);
            } else {   // 3 magnitude bits by binary search, the magnitude from the table
                const float d2 = ts[3] - av;
                const bool m2 = d2 < 0.f;
                const float d1 = (m2 ? ts[5] : ts[1]) - av;
                const bool m1 = d1 < 0.f;
                const float d0 = (m2 ? (m1 ? ts[6] : ts[4]) : (m1 ? ts[2] : ts[0])) - av;
                const bool m0 = d0 < 0.f;
                mw[2] = __funnelshift_l(__float_as_uint(d2), mw[2], 1);
                mw[1] = __funnelshift_l(__float_as_uint(d1), mw[1], 1);
                mw[0] = __funnelshift_l(__float_as_uint(d0), mw[0], 1);
                mag = cen[H + (m2 ? 4 : 0) + (m1 ? 2 : 0) + (m0 ? 1 : 0)];
            }
            const float r = fmaf(n16, copysignf(mag, dz), y[c]);
            y[c] = r;
            rs = fmaf(r, r, rs);
        }
    }
    pw[NB - 1] = sg;
#pragma unroll
    for (int p = 0; p + 1 < NB; ++p) pw[p] = mw[p] ^ ~sg;
}

// SYM: the table (for SPLIT, both tables) is odd-symmetric, c_k = -c_{2^P-1-k}: codes by sym_codes.
// SPLIT: a split context, each coordinate word coded with P or, below d_hi, P + 1 bits from its own
// table (P = 0 when not SYM: the width is then read at run time and the tables searched in order).
template <int P, bool SYM, bool SPLIT = false>
__global__ void __launch_bounds__(kTcThreads, 1) quantize_tc2_kernel(const TcArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ __align__(8) uint64_t mbar[kTc2Groups], s_drain[kTc2Groups];
    __shared__ uint32_t s_tmem;
    __shared__ int s_drained;
    __shared__ float s_thr[kMaxLevels], s_cen[kMaxLevels], s_thr_hi[kMaxLevels], s_cen_hi[kMaxLevels];
    const Params& prm = a.prm;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp >> 3, gw = warp & 7, q = gw & 3, hh = gw >> 2, gtid = tid & (kTc2GThreads - 1);
    const int row = 32 * q + lane, bar_id = 1 + g;
    const bool leader = gtid == 0;
    unsigned char* sB = sm;
    unsigned char* sX = sm + kSmemB + g * kMatBytes;
    float* s_xn = reinterpret_cast<float*>(sm + kSmemB + kTc2Groups * kMatBytes) + g * 4 * kTile;   // [2][128]
    float* s_rs = s_xn + 2 * kTile;                                                                  // [2][128]
    const int ntiles = (int)((a.n + kTile - 1) / kTile);
    if (tid < kMaxLevels) {
        s_thr[tid] = prm.thresholds[tid];
        s_cen[tid] = prm.centroids[tid];
        if (SPLIT) {
            s_thr_hi[tid] = prm.thresholds_hi[tid];
            s_cen_hi[tid] = prm.centroids_hi[tid];
        }
    }
    for (int e = tid; e < (int)((prm.qjl ? kSmemB : kSmemB / 2) / 16); e += kTcThreads) tc::cp_async16(sB + 16 * e, a.bops + e);
    asm volatile("cp.async.commit_group;");
    int tile = kTc2Groups * blockIdx.x + g;
    if (tile < ntiles) stage_x_group(a, tile, sX, gtid);
    else asm volatile("cp.async.commit_group;");   // an empty group keeps the wait counts alike
    if (tid == 0) {
        for (int i = 0; i < kTc2Groups; ++i) {
            tc::mbar_init(&mbar[i], 1);
            tc::mbar_init(&s_drain[i], 1);
        }
        s_drained = 1;
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc<512>(&s_tmem);
    asm volatile("cp.async.wait_group 1;");   // this thread's share of the B operands has landed
    asm volatile("fence.proxy.async.shared::cta;");
    tc::fence_before();
    __syncthreads();   // both groups' shares: the B operands are whole before either group's MMAs
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t d_col = tmem + 256 * g, a_col = d_col + 128;
    const uint32_t d_row = d_col + lane_off, a_row = a_col + lane_off;
    uint32_t phase = 0;
    bool ok = true;

    for (; tile < ntiles && ok; tile += kTc2Groups * gridDim.x) {
        const int64_t r0 = (int64_t)tile * kTile;
        const int nvalid = (int)min((int64_t)kTile, a.n - r0);
        asm volatile("cp.async.wait_group 0;");   // this tile's rows (and, at first, the B operands)
        asm volatile("fence.proxy.async.shared::cta;");
        tc::fence_before();
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");
        tc::fence_after();
        if (leader) {   // phase 1: Y = X Pi^T
            issue_pieces(d_col, tc::smem_u32(sX), tc::smem_u32(sB), false);
            tc::commit(&mbar[g]);
        }
        {   // ||x||^2 partial over this thread's 64 coordinates while the MMAs run
            float xs = 0.f;
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                const uint4 w = *reinterpret_cast<const uint4*>(sX + kmajor_off(row, 64 * hh + 8 * kc));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16_bits_to_float(ws[i] & 0xffffu), hi = bf16_bits_to_float(ws[i] >> 16);
                    xs = fmaf(lo, lo, xs);
                    xs = fmaf(hi, hi, xs);
                }
            }
            s_xn[hh * kTile + row] = xs;
        }
        ok = group_and(tc::mbar_wait(&mbar[g], phase), bar_id);   // also: the x reads are done
        phase ^= 1u;
        if (!ok) break;
        tc::fence_after();
        const int next = tile + kTc2Groups * gridDim.x;
        if (next < ntiles) stage_x_group(a, next, sX, gtid);   // lands while this tile finishes
        const float nrm = sqrtf(s_xn[row] + s_xn[kTile + row]);
        const float n16 = half_bits_to_float(float_to_half_bits(nrm));
        const float nv = nrm > 0.f ? nrm : 1.f;
        const int64_t grow = r0 + row;
        const bool valid = row < nvalid;
        float rs = 0.f;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int part = 2 * hh + pass;
            float y[32];
            load_row_part(d_row, part, y);
            uint32_t pw[kFastBits] = {};
            const bool hi = SPLIT && 32 * part < prm.d_hi;   // this word's coordinates take P + 1 bits
            if constexpr (SPLIT && SYM) {   // the word's table is the P- or (P+1)-bit one, both symmetric
                if (hi) sym_codes<P + 1>(y, nrm, n16, nv, s_thr_hi, s_cen_hi, pw, rs);
                else sym_codes<P>(y, nrm, n16, nv, s_thr, s_cen, pw, rs);
            } else if constexpr (SPLIT) {
                const int nb = prm.P + (hi ? 1 : 0);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float yc = nrm > 0.f ? y[c] : 0.f;
                    int idx = 0;
#pragma unroll
                    for (int b = kFastBits - 1; b >= 0; --b)
                        if (b < nb) {
                            const int k = idx + (1 << b) - 1;
                            const bool up = yc > (hi ? s_thr_hi[k] : s_thr[k]) * nv;
                            idx += up ? (1 << b) : 0;
                            pw[b] |= (up ? 1u : 0u) << c;
                        }
                    const float r = y[c] - n16 * (hi ? s_cen_hi[idx] : s_cen[idx]);
                    y[c] = r;
                    rs = fmaf(r, r, rs);
                }
            } else if constexpr (SYM) {
                sym_codes<P>(y, nrm, n16, nv, s_thr, s_cen, pw, rs);
            } else if constexpr (P <= 3) {
                constexpr int NT = (1 << P) - 1;
                float ts[NT], cv[NT + 1];
#pragma unroll
                for (int k = 0; k < NT; ++k) ts[k] = s_thr[k] * nv;
#pragma unroll
                for (int k = 0; k <= NT; ++k) cv[k] = s_cen[k];
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float yc = nrm > 0.f ? y[c] : 0.f;
                    float cen;
                    if constexpr (P == 1) {
                        const bool up = yc > ts[0];
                        pw[0] |= (up ? 1u : 0u) << c;
                        cen = up ? cv[1] : cv[0];
                    } else if constexpr (P == 2) {
                        const bool u1 = yc > ts[1];
                        const bool u0 = yc > (u1 ? ts[2] : ts[0]);
                        pw[1] |= (u1 ? 1u : 0u) << c;
                        pw[0] |= (u0 ? 1u : 0u) << c;
                        cen = u1 ? (u0 ? cv[3] : cv[2]) : (u0 ? cv[1] : cv[0]);
                    } else {
                        const bool u2 = yc > ts[3];
                        const bool u1 = yc > (u2 ? ts[5] : ts[1]);
                        const float t0 = u2 ? (u1 ? ts[6] : ts[4]) : (u1 ? ts[2] : ts[0]);
                        const bool u0 = yc > t0;
                        pw[2] |= (u2 ? 1u : 0u) << c;
                        pw[1] |= (u1 ? 1u : 0u) << c;
                        pw[0] |= (u0 ? 1u : 0u) << c;
                        const float clo = u1 ? (u0 ? cv[3] : cv[2]) : (u0 ? cv[1] : cv[0]);
                        const float chi = u1 ? (u0 ? cv[7] : cv[6]) : (u0 ? cv[5] : cv[4]);
                        cen = u2 ? chi : clo;
                    }
                    const float r = y[c] - n16 * cen;
                    y[c] = r;
                    rs = fmaf(r, r, rs);
                }
            } else {
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const float yc = nrm > 0.f ? y[c] : 0.f;
                    int idx = 0;
#pragma unroll
                    for (int b = P - 1; b >= 0; --b) {
                        const int k = idx + (1 << b) - 1;
                        const bool up = yc > s_thr[k] * nv;
                        idx += up ? (1 << b) : 0;
                        pw[b] |= (up ? 1u : 0u) << c;
                    }
                    const float r = y[c] - n16 * s_cen[idx];
                    y[c] = r;
                    rs = fmaf(r, r, rs);
                }
            }
            if (valid) {
                if constexpr (SPLIT && SYM) {   // P planes, then the top plane of the words below d_hi
#pragma unroll
                    for (int p = 0; p < P; ++p) a.planes[(size_t)grow * prm.row_words + p * 4 + part] = pw[p];
                    if (hi) a.planes[(size_t)grow * prm.row_words + P * 4 + part] = pw[P];
                } else if constexpr (SPLIT) {
                    for (int p = 0; p < prm.P; ++p) a.planes[(size_t)grow * prm.row_words + p * 4 + part] = pw[p];
                    if (hi) {
                        const uint32_t top = prm.P == 1 ? pw[1] : (prm.P == 2 ? pw[2] : pw[3]);
                        a.planes[(size_t)grow * prm.row_words + prm.P * 4 + part] = top;
                    }
                } else {
#pragma unroll
                    for (int p = 0; p < P; ++p) a.planes[(size_t)grow * prm.row_words + p * 4 + part] = pw[p];
                }
            }
            if (prm.qjl) {   // r' as bf16 hi and lo into the A operand
                uint32_t h[16], l[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const __nv_bfloat162 hp = __floats2bfloat162_rn(y[2 * i], y[2 * i + 1]);
                    h[i] = *reinterpret_cast<const uint32_t*>(&hp);
                    const float h0 = __uint_as_float(h[i] << 16), h1 = __uint_as_float(h[i] & 0xffff0000u);
                    const __nv_bfloat162 lp = __floats2bfloat162_rn(y[2 * i] - h0, y[2 * i + 1] - h1);
                    l[i] = *reinterpret_cast<const uint32_t*>(&lp);
                }
                tc::tmem_st16(a_row + 16 * part, h);
                tc::tmem_st16(a_row + 64 + 16 * part, l);
            }
        }
        if (!prm.qjl) {   // MSE mode: no residual sketch
            if (valid && hh == 0) {
                const uint16_t nh = float_to_half_bits(nrm);
                a.norm[grow] = nh;
                if (__hisinf(__ushort_as_half(nh))) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
            }
            tc::fence_before();
            continue;   // the next iteration's group barrier orders these TMEM reads before its MMAs
        }
        s_rs[hh * kTile + row] = rs;
        tc::wait_st();
        tc::fence_before();
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");   // Y read, A written
        if (leader) {   // phase 2: Z = r' (S Pi^T)^T, A from tensor memory
            tc::fence_after();
            issue_pieces_ta(d_col, a_col, tc::smem_u32(sB) + kPieces * kMatBytes);
            tc::commit(&mbar[g]);
        }
        ok = group_and(tc::mbar_wait(&mbar[g], phase), bar_id);
        phase ^= 1u;
        if (!ok) break;
        tc::fence_after();
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int part = 2 * hh + pass;
            float z[32];
            load_row_part(d_row, part, z);
            uint32_t sw = 0u;   // bit c = [z_c > 0]: the sign bit of 0 - z_c (+0 for z_c = +-0)
#pragma unroll
            for (int c = 31; c >= 0; --c) sw = __funnelshift_l(__float_as_uint(0.f - z[c]), sw, 1);
            if (valid) a.signs[(size_t)grow * 4 + part] = sw;
        }
        if (valid && hh == 0) {
            const uint16_t nh = float_to_half_bits(nrm);
            const uint16_t rh = float_to_half_bits(sqrtf(s_rs[row] + s_rs[kTile + row]));
            a.norm[grow] = nh;
            a.rnorm[grow] = rh;
            if (__hisinf(__ushort_as_half(nh)) || __hisinf(__ushort_as_half(rh))) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
        }
        tc::fence_before();
    }
    asm volatile("cp.async.wait_all;");
    if (!ok) {   // a wait ran out: flag it, and let every MMA this group issued finish (bounded)
        if (leader) {
            set_error(a.err, TQ_DEVERR_TIMEOUT);
            tc::commit(&s_drain[g]);
        }
        if (!group_and(!leader || tc::mbar_wait(&s_drain[g], 0u), bar_id) && leader) s_drained = 0;
    }
    tc::fence_before();
    __syncthreads();
    // an MMA that outlived the bounded drain still writes this memory: it is then left allocated
    if (warp == 0 && s_drained) tc::tmem_dealloc<512>(tmem);
}

// ---------------------------------------------------------------- polar-angle encoder
// The recursive polar encoder (k_polar.cu; csdn tutorial, section 将笛卡尔积坐标转为极坐标, and
// freelamp article, section 技术突破：极坐标量化) with its two d x d products on the tensor cores, for
// bf16 rows at d = 128 (7 levels, 127 angles): phase 1 Y = X Pi^T as above; the epilogue runs the
// polar transform — each 32 consecutive coordinates are the subtree of one level-5 node, so levels
// 1-5 are thread-local and one thread per row combines the 4 level-5 radii into levels 6 and 7 —
// codes each angle against its level's thresholds, packs the code stream, rebuilds y_hat
// top-down from the stored fp16 radius and the centroids' cos / sin, and with QJL projects
// r' = y - y_hat as in phase 2 above (r = Pi^T r', so S r = (S Pi^T) r').
// The angle codes need neither the angles nor the radii themselves: a level-1 code is the index of
// the uniform sector holding (y_2i, y_2i+1), found by halving the turn (sector_code); a level-l
// angle atan2(r_hi, r_lo) in [0, pi/2] passes threshold t exactly when R_hi > tan^2(t) R_lo, with R
// the squared radii, which add up the tree without square roots (level_code).  Both decide as the
// angle comparisons do, up to float rounding at a threshold.
constexpr int kPolarTcLevels = 7;
constexpr int kCodeStride = 132;   // bytes per row of the code stream in shared memory (33 words: no bank conflicts)
constexpr float kTanPi8 = 0.41421356237309504880f;   // tan(pi / 8)

struct PolarTcArgs {
    const uint16_t* x;
    int64_t n, ld_x;
    const uint4* bops;
    const float* cs;          // [level][32]: cos then sin of the level's 2^B centroids
    uint32_t* codes;
    uint16_t* r16;
    uint32_t* signs;
    uint16_t* rnorm;
    int* err;
    int cw;                   // code words per row
    float tau[kPolarTcLevels - 1][15];   // levels 2..7: tan^2 of the ascending thresholds (uniform indices)
};

// Level-1 code: #{k >= 1 : psi > 2 pi k / 2^B} for psi = atan2(hi, lo) taken in [0, 2 pi).  Halving
// the turn: psi > pi is hi < 0, after which the point turns by pi; the remaining angle exceeds
// pi / 2 when x < 0, after which the point turns by pi / 2; it then exceeds pi / 4 when y > x,
// after which it turns by pi / 4 (scaled by sqrt 2); last, it exceeds pi / 8 when
// y > tan(pi / 8) x.  Signed zeros fall as atan2 puts them (hi = -0 counts as the upper
// half-plane, as atan2(-0, lo) in {-0, pi} does after the wrap).
template <int B>
__device__ __forceinline__ int sector_code(float lo, float hi) {
    const bool s1 = hi < 0.f;
    if constexpr (B == 1) return s1 ? 1 : 0;
    const float x1 = s1 ? -lo : lo, y1 = s1 ? -hi : hi;
    const bool s2 = x1 < 0.f;
    int c = (s1 ? 2 : 0) + (s2 ? 1 : 0);
    if constexpr (B == 2) return c;
    const float x2 = s2 ? y1 : x1, y2 = s2 ? -x1 : y1;
    const bool s3 = y2 > x2;
    c = 2 * c + (s3 ? 1 : 0);
    if constexpr (B == 3) return c;
    const float x3 = s3 ? x2 + y2 : x2, y3 = s3 ? y2 - x2 : y2;
    return 2 * c + (y3 > kTanPi8 * x3 ? 1 : 0);
}

// Level-l code (l >= 2): #{k : atan2(r_hi, r_lo) > t_k}, t_k in (0, pi/2), from the squared radii:
// the angle passes t_k iff R_hi / R_lo > tan^2 t_k (the ratio is +inf for R_lo = 0 < R_hi and NaN
// for 0 / 0, whose angle atan2(0, 0) = 0 passes nothing).  The tan^2 t_k ascend, so the count is a
// B-step binary search (the step for bit b deciding bit b of the code); tau indices are compile-
// time constants, the thresholds picked by selects.
template <int B>
__device__ __forceinline__ int level_code(float Rlo, float Rhi, const float* tau) {
    const float qv = __fdividef(Rhi, Rlo);
    if constexpr (B == 1) {
        return qv > tau[0] ? 1 : 0;
    } else if constexpr (B == 2) {
        const bool u1 = qv > tau[1];
        const bool u0 = qv > (u1 ? tau[2] : tau[0]);
        return (u1 ? 2 : 0) + (u0 ? 1 : 0);
    } else if constexpr (B == 3) {
        const bool u2 = qv > tau[3];
        const bool u1 = qv > (u2 ? tau[5] : tau[1]);
        const bool u0 = qv > (u2 ? (u1 ? tau[6] : tau[4]) : (u1 ? tau[2] : tau[0]));
        return (u2 ? 4 : 0) + (u1 ? 2 : 0) + (u0 ? 1 : 0);
    } else {
        const bool u3 = qv > tau[7];
        const bool u2 = qv > (u3 ? tau[11] : tau[3]);
        const float t1 = u3 ? (u2 ? tau[13] : tau[9]) : (u2 ? tau[5] : tau[1]);
        const bool u1 = qv > t1;
        const float t0 = u3 ? (u2 ? (u1 ? tau[14] : tau[12]) : (u1 ? tau[10] : tau[8]))
                            : (u2 ? (u1 ? tau[6] : tau[4]) : (u1 ? tau[2] : tau[0]));
        const bool u0 = qv > t0;
        return (u3 ? 8 : 0) + (u2 ? 4 : 0) + (u1 ? 2 : 0) + (u0 ? 1 : 0);
    }
}

// The polar encoder runs two tiles in flight per CTA, as quantize_tc2_kernel: two 8-warp groups,
// each with its own x buffer, accumulator D and A operand (r' hi and lo) in tensor memory.  A
// thread owns 64 coordinates of its row (two level-5 subtrees, taken in two passes); the thread
// holding the row's first half adds levels 6 and 7.  The codes use the group's spent x buffer as
// scratch, so the next tile's rows are copied in once they are packed and, with QJL, y_hat has
// been rebuilt: during the projection and the signs.  Per group six 128-float slots: x-norm
// partials (0, 1), the squared level-5 radii of parts 0..3 (2..5), then the r'-norm partials (2, 3).
constexpr uint32_t kSmemPolar2 = kSmemB + kTc2Groups * kMatBytes + kTc2Groups * 6 * kTile * sizeof(float);

template <int B, bool QJL>
__global__ void __launch_bounds__(kTcThreads, 1) polar_tc2_kernel(const PolarTcArgs a) {
    extern __shared__ __align__(128) unsigned char sm[];
    __shared__ __align__(8) uint64_t mbar[kTc2Groups], s_drain[kTc2Groups];
    __shared__ uint32_t s_tmem;
    __shared__ int s_drained;
    __shared__ float s_cs[kPolarTcLevels * 32];   // indexed by code per lane: shared, not parameter space
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = warp >> 3, gw = warp & 7, q = gw & 3, hh = gw >> 2, gtid = tid & (kTc2GThreads - 1);
    const int row = 32 * q + lane, bar_id = 1 + g;
    const bool leader = gtid == 0;
    unsigned char* sB = sm;
    unsigned char* sX = sm + kSmemB + g * kMatBytes;
    float* s_part = reinterpret_cast<float*>(sm + kSmemB + kTc2Groups * kMatBytes) + g * 6 * kTile;
    const int ntiles = (int)((a.n + kTile - 1) / kTile);
    if (QJL && tid < kPolarTcLevels * 32) s_cs[tid] = a.cs[tid];
    for (int e = tid; e < (int)((QJL ? kSmemB : kSmemB / 2) / 16); e += kTcThreads) tc::cp_async16(sB + 16 * e, a.bops + e);
    asm volatile("cp.async.commit_group;");
    auto stage = [&](int t) {   // the x rows of tile t into this group's buffer, one commit group
        const int64_t r0 = (int64_t)t * kTile;
        const int nv = (int)min((int64_t)kTile, a.n - r0);
        for (int e = gtid; e < kTile * 16; e += kTc2GThreads) {
            const int r = e >> 4, kc = e & 15;
            unsigned char* dst = sX + kmajor_off(r, 8 * kc);
            if (r < nv) tc::cp_async16(dst, a.x + (size_t)(r0 + r) * a.ld_x + 8 * kc);
            else *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        asm volatile("cp.async.commit_group;");
    };
    int tile = kTc2Groups * blockIdx.x + g;
    if (tile < ntiles) stage(tile);
    else asm volatile("cp.async.commit_group;");   // an empty group keeps the wait counts alike
    if (tid == 0) {
        for (int i = 0; i < kTc2Groups; ++i) {
            tc::mbar_init(&mbar[i], 1);
            tc::mbar_init(&s_drain[i], 1);
        }
        s_drained = 1;
        tc::mbar_init_fence();
    }
    if (warp == 0) tc::tmem_alloc<512>(&s_tmem);
    asm volatile("cp.async.wait_group 1;");   // this thread's share of the B operands has landed
    asm volatile("fence.proxy.async.shared::cta;");
    tc::fence_before();
    __syncthreads();   // both groups' shares: the B operands (and the cos/sin table) are whole
    tc::fence_after();
    const uint32_t tmem = s_tmem;
    const uint32_t lane_off = (uint32_t)(32 * q) << 16;
    const uint32_t d_col = tmem + 256 * g, a_col = d_col + 128;
    const uint32_t d_row = d_col + lane_off, a_row = a_col + lane_off;
    const float* cs = s_cs;
    uint32_t phase = 0;
    bool ok = true;

    for (; tile < ntiles && ok; tile += kTc2Groups * gridDim.x) {
        const int64_t r0 = (int64_t)tile * kTile;
        const int nvalid = (int)min((int64_t)kTile, a.n - r0);
        const int next = tile + kTc2Groups * gridDim.x;
        asm volatile("cp.async.wait_group 0;");
        asm volatile("fence.proxy.async.shared::cta;");
        tc::fence_before();
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");
        tc::fence_after();
        if (leader) {   // phase 1: Y = X Pi^T
            issue_pieces(d_col, tc::smem_u32(sX), tc::smem_u32(sB), false);
            tc::commit(&mbar[g]);
        }
        {   // ||x||^2 partial over this thread's 64 coordinates while the MMAs run
            float xs = 0.f;
#pragma unroll
            for (int kc = 0; kc < 8; ++kc) {
                const uint4 w = *reinterpret_cast<const uint4*>(sX + kmajor_off(row, 64 * hh + 8 * kc));
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float lo = bf16_bits_to_float(ws[i] & 0xffffu), hi = bf16_bits_to_float(ws[i] >> 16);
                    xs = fmaf(lo, lo, xs);
                    xs = fmaf(hi, hi, xs);
                }
            }
            s_part[hh * kTile + row] = xs;
        }
        ok = group_and(tc::mbar_wait(&mbar[g], phase), bar_id);   // also: the x reads are done
        phase ^= 1u;
        if (!ok) break;
        tc::fence_after();
        const float nrm = sqrtf(s_part[row] + s_part[kTile + row]);
        const int64_t grow = r0 + row;
        const bool valid = row < nvalid;
        unsigned char* code = sX + row * kCodeStride;   // this row's 127 angle codes (the x buffer is spent)
        // levels 1-5 of this thread's two level-5 subtrees (part p = 2 hh + pass; level-l node i of
        // subtree p is global node (32 >> l) p + i, at stream position 128 - (256 >> l) + that)
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int part = 2 * hh + pass;
            float y[32];
            load_row_part(d_row, part, y);
            float rad[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float lo = y[2 * i], hi = y[2 * i + 1];
                rad[i] = fmaf(lo, lo, hi * hi);
                code[16 * part + i] = (unsigned char)sector_code<B>(lo, hi);
            }
#pragma unroll
            for (int l = 2; l <= 5; ++l) {
                const int nodes = 32 >> l, pos = 128 - (256 >> l) + nodes * part;
#pragma unroll
                for (int i = 0; i < nodes; ++i) {
                    const float lo = rad[2 * i], hi = rad[2 * i + 1];
                    rad[i] = lo + hi;
                    code[pos + i] = (unsigned char)level_code<B>(lo, hi, a.tau[l - 2]);
                }
            }
            s_part[(2 + part) * kTile + row] = rad[0];
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");   // level-5 radii visible
        if (hh == 0) {   // levels 6 and 7 of the row
            const float r5[4] = {s_part[2 * kTile + row], s_part[3 * kTile + row], s_part[4 * kTile + row],
                                 s_part[5 * kTile + row]};
#pragma unroll
            for (int i = 0; i < 2; ++i) code[124 + i] = (unsigned char)level_code<B>(r5[2 * i], r5[2 * i + 1], a.tau[4]);
            code[126] = (unsigned char)level_code<B>(r5[0] + r5[1], r5[2] + r5[3], a.tau[5]);
        }
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");   // every code written
        // pack: word w holds stream bits 32 w .. 32 w + 31, stream bit t being bit t - B an of code
        // an = t / B; the codes from a0 = 32 w / B on are laid side by side in a 64-bit window
        // (code a0 + k at bit B k), whose bits sh .. sh + 31 (sh = 32 w - B a0) are the word
        for (int w = hh; w < a.cw; w += 2) {
            const int a0 = 32 * w / B, sh = 32 * w - B * a0;
            constexpr int K = (31 + B - 1) / B + 1;
            uint64_t win = 0u;
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (a0 + k < 127) win |= (uint64_t)code[a0 + k] << (B * k);
            if (valid) a.codes[(size_t)grow * a.cw + w] = (uint32_t)(win >> sh);
        }
        const uint16_t nh = float_to_half_bits(nrm);
        if (valid && hh == 0) {
            a.r16[grow] = nh;
            if (__hisinf(__ushort_as_half(nh))) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
        }
        if constexpr (!QJL) {
            asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");   // codes read
            if (next < ntiles) stage(next);
            tc::fence_before();
            continue;
        }
        // y_hat top-down from the stored radius: root -> level 6 -> the part's level-5 node -> its
        // subtree; r' = y - y_hat into the A operand as bf16 hi and lo
        float rs = 0.f;
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int part = 2 * hh + pass;
            float y[32];
            load_row_part(d_row, part, y);
            float rho = half_bits_to_float(nh);
            {
                const int c7 = code[126], c6 = code[124 + (part >> 1)];
                rho *= (part >> 1) ? cs[6 * 32 + 16 + c7] : cs[6 * 32 + c7];
                rho *= (part & 1) ? cs[5 * 32 + 16 + c6] : cs[5 * 32 + c6];
            }
            float rad[16];
            rad[0] = rho;
#pragma unroll
            for (int l = 5; l >= 2; --l) {   // node i of level l -> children 2 i, 2 i + 1 of level l - 1
                const int nodes = 32 >> l, pos = 128 - (256 >> l) + nodes * part;
#pragma unroll
                for (int i = nodes - 1; i >= 0; --i) {
                    const int c = code[pos + i];
                    const float r = rad[i];
                    rad[2 * i] = r * cs[(l - 1) * 32 + c];
                    rad[2 * i + 1] = r * cs[(l - 1) * 32 + 16 + c];
                }
            }
            uint32_t h[16], lo16[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const int c = code[16 * part + i];
                const float r0v = y[2 * i] - rad[i] * cs[c], r1v = y[2 * i + 1] - rad[i] * cs[16 + c];
                rs = fmaf(r0v, r0v, rs);
                rs = fmaf(r1v, r1v, rs);
                const __nv_bfloat162 hp = __floats2bfloat162_rn(r0v, r1v);
                h[i] = *reinterpret_cast<const uint32_t*>(&hp);
                const float h0 = __uint_as_float(h[i] << 16), h1 = __uint_as_float(h[i] & 0xffff0000u);
                const __nv_bfloat162 lp = __floats2bfloat162_rn(r0v - h0, r1v - h1);
                lo16[i] = *reinterpret_cast<const uint32_t*>(&lp);
            }
            tc::tmem_st16(a_row + 16 * part, h);
            tc::tmem_st16(a_row + 64 + 16 * part, lo16);
        }
        s_part[(2 + hh) * kTile + row] = rs;   // the level-5 slots were last read before the code barrier
        tc::wait_st();
        tc::fence_before();
        asm volatile("bar.sync %0, %1;" ::"r"(bar_id), "n"(kTc2GThreads) : "memory");   // codes read, A written
        if (next < ntiles) stage(next);   // the code scratch is free: the next tile's rows land meanwhile
        if (leader) {   // phase 2: Z = r' (S Pi^T)^T, A from tensor memory
            tc::fence_after();
            issue_pieces_ta(d_col, a_col, tc::smem_u32(sB) + kPieces * kMatBytes);
            tc::commit(&mbar[g]);
        }
        ok = group_and(tc::mbar_wait(&mbar[g], phase), bar_id);
        phase ^= 1u;
        if (!ok) break;
        tc::fence_after();
#pragma unroll 1
        for (int pass = 0; pass < 2; ++pass) {
            const int part = 2 * hh + pass;
            float z[32];
            load_row_part(d_row, part, z);
            uint32_t sw = 0u;   // bit c = [z_c > 0]: the sign bit of 0 - z_c (+0 for z_c = +-0)
#pragma unroll
            for (int c = 31; c >= 0; --c) sw = __funnelshift_l(__float_as_uint(0.f - z[c]), sw, 1);
            if (valid) a.signs[(size_t)grow * 4 + part] = sw;
        }
        if (valid && hh == 0) {
            const uint16_t rh = float_to_half_bits(sqrtf(s_part[2 * kTile + row] + s_part[3 * kTile + row]));
            a.rnorm[grow] = rh;
            if (__hisinf(__ushort_as_half(rh))) set_error(a.err, TQ_DEVERR_NORM_OVERFLOW);
        }
        tc::fence_before();
    }
    asm volatile("cp.async.wait_all;");
    if (!ok) {   // a wait ran out: flag it, and let every MMA this group issued finish (bounded)
        if (leader) {
            set_error(a.err, TQ_DEVERR_TIMEOUT);
            tc::commit(&s_drain[g]);
        }
        if (!group_and(!leader || tc::mbar_wait(&s_drain[g], 0u), bar_id) && leader) s_drained = 0;
    }
    tc::fence_before();
    __syncthreads();
    // an MMA that outlived the bounded drain still writes this memory: it is then left allocated
    if (warp == 0 && s_drained) tc::tmem_dealloc<512>(tmem);
}

}  // namespace

bool quantize_tc_supported(const tq_ctx* c, int dtype, const void* x, int64_t n, int64_t ld_x) {
    return c->bops != nullptr && c->P <= kFastBits && c->kernel_path != TQ_PATH_CUDA_CORE && dtype == TQ_BF16 && n >= 4096 &&
           (ld_x % 8) == 0 && (reinterpret_cast<uintptr_t>(x) % 16) == 0;
}

// Host layout of the four B operands (Pi pieces hi, mid, then S Pi^T pieces hi, mid): element
// (i, j) of each 128 x 128 matrix at kmajor_off(i, j); St NULL leaves the last two zero.
void build_tc_operands(const float* Pi, const float* St, std::vector<uint16_t>& out) {
    out.assign(2 * kPieces * 128 * 128, 0);
    auto bf16_rne = [](float v) -> uint16_t {
        uint32_t u;
        std::memcpy(&u, &v, 4);
        const uint32_t lsb = (u >> 16) & 1u;
        return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
    };
    auto bf16_val = [](uint16_t b) -> float {
        uint32_t u = (uint32_t)b << 16;
        float v;
        std::memcpy(&v, &u, 4);
        return v;
    };
    for (int which = 0; which < (St ? 2 : 1); ++which)
        for (int i = 0; i < 128; ++i)
            for (int j = 0; j < 128; ++j) {
                const float v = which == 0 ? Pi[i * 128 + j] : St[i * 128 + j];
                const uint16_t h = bf16_rne(v);
                const uint16_t m = bf16_rne(v - bf16_val(h));
                const uint16_t piece[kPieces] = {h, m};
                for (int p = 0; p < kPieces; ++p)
                    out[((size_t)(kPieces * which + p) * 128 * 128 * 2 + kmajor_off(i, j)) / 2] = piece[p];
            }
}

cudaError_t launch_quantize_tc(const tq_ctx* c, const void* x, int64_t n, int64_t ld_x, uint32_t* planes,
                               uint32_t* signs, uint16_t* norm, uint16_t* rnorm, cudaStream_t s) {
    TcArgs a{};
    a.prm = c->prm;
    a.x = static_cast<const uint16_t*>(x);
    a.n = n;
    a.ld_x = ld_x;
    a.bops = reinterpret_cast<const uint4*>(c->bops);
    a.planes = planes;
    a.signs = signs;
    a.norm = norm;
    a.rnorm = rnorm;
    a.err = c->derr;
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, c->device);
    const int64_t ntiles = (n + kTile - 1) / kTile;
    // two tiles in flight per CTA (quantize_tc2_kernel)
    const int64_t pairs = (ntiles + kTc2Groups - 1) / kTc2Groups;
    const int grid2 = (int)(pairs < sms ? pairs : sms);
    auto run2 = [&](auto kernel) -> cudaError_t {
        cudaError_t e2 = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemTc2);
        if (e2 != cudaSuccess) return e2;
        kernel<<<grid2, kTcThreads, kSmemTc2, s>>>(a);
        return cudaSuccess;
    };
    cudaError_t e = cudaErrorInvalidValue;
    const bool sym = c->prm.odd_walsh != 0;
    if (c->prm.d_hi > 0) {
        if (c->prm.split_walsh && c->prm.P == 1) e = run2(quantize_tc2_kernel<1, true, true>);
        else if (c->prm.split_walsh && c->prm.P == 2) e = run2(quantize_tc2_kernel<2, true, true>);
        else if (c->prm.split_walsh && c->prm.P == 3) e = run2(quantize_tc2_kernel<3, true, true>);
        else e = run2(quantize_tc2_kernel<0, false, true>);
    }
    else if (c->prm.P == 1) e = sym ? run2(quantize_tc2_kernel<1, true>) : run2(quantize_tc2_kernel<1, false>);
    else if (c->prm.P == 2) e = sym ? run2(quantize_tc2_kernel<2, true>) : run2(quantize_tc2_kernel<2, false>);
    else if (c->prm.P == 3) e = sym ? run2(quantize_tc2_kernel<3, true>) : run2(quantize_tc2_kernel<3, false>);
    else if (c->prm.P == 4) e = sym ? run2(quantize_tc2_kernel<4, true>) : run2(quantize_tc2_kernel<4, false>);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace tq

namespace tq {

cudaError_t launch_polar_tc(const PolarTcLaunch& L, cudaStream_t s) {
    PolarTcArgs a{};
    a.x = static_cast<const uint16_t*>(L.x);
    a.n = L.n;
    a.ld_x = L.ld_x;
    a.bops = reinterpret_cast<const uint4*>(L.bops);
    a.cs = L.cs;
    a.codes = L.codes;
    a.r16 = L.r16;
    a.signs = L.signs;
    a.rnorm = L.rnorm;
    a.err = L.err;
    a.cw = L.cw;
    for (int l = 0; l + 1 < kPolarTcLevels; ++l)
        for (int t = 0; t < 15; ++t) a.tau[l][t] = L.tau[l][t];
    int sms = 148;
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, L.device);
    const int64_t ntiles = (L.n + kTile - 1) / kTile;
    const int64_t pairs = (ntiles + kTc2Groups - 1) / kTc2Groups;   // two tiles in flight per CTA
    const int grid = (int)(pairs < sms ? pairs : sms);
    auto run = [&](auto kernel) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemPolar2);
        if (e != cudaSuccess) return e;
        kernel<<<grid, kTcThreads, kSmemPolar2, s>>>(a);
        return cudaGetLastError();
    };
    switch (L.bits * 2 + (L.qjl ? 1 : 0)) {
        case 2: return run(polar_tc2_kernel<1, false>);
        case 3: return run(polar_tc2_kernel<1, true>);
        case 4: return run(polar_tc2_kernel<2, false>);
        case 5: return run(polar_tc2_kernel<2, true>);
        case 6: return run(polar_tc2_kernel<3, false>);
        case 7: return run(polar_tc2_kernel<3, true>);
        case 8: return run(polar_tc2_kernel<4, false>);
        case 9: return run(polar_tc2_kernel<4, true>);
    }
    return cudaErrorInvalidValue;
}

}  // namespace tq
