// Softmax-weighted sum of MSE-coded values on the 5th-generation tensor cores (tcgen05.mma
// kind::f8f6f4, A in tensor memory) for 96 < d <= 128 and 1..3 value bits.
//
// Pages: nonndazone.ru essay, section 2 (keys and values are both cached and compressed); the
// softmax-weighted sum of the values is the attention step after the logits of the juejin.cn post,
// section 三.  The arithmetic is that of values_coded128_kernel (k_attn.cu), rearranged as a small
// dense contraction per block of 32 keys:
//   Walsh form of the value table (host_setup.cpp): c(idx) = c0 + sum_t kappa_t x_t(idx), x_t the
//   parity of the index bits in the t-th odd subset.  With w_i = exp(l_i - M) n_i (n_i the value's
//   fp16 norm, M the chunk's largest logit of the head),
//     sum_i w_i v_hat_i[j] = c0 sum_i w_i + sum_t kappa_t sum_i w_i x_t(idx_ij)
//   and the last sum is D_t[j][h] = sum_k A_t[j][k] B[k][h]: A_t the 0/1 bits of term t (coordinate
//   j = TMEM lane, key k), B the weights of the 4 query heads of the GQA quad.
//
// A (TMEM, per term 8 columns = 32 keys): the value rows are stored key-major, so each warp turns
//   the 32 keys' plane words of its 32 coordinates (one word per key) into per-coordinate 32-key
//   masks with a 5-round shuffle transpose, XORs the planes of each term, and expands every mask
//   into e4m3 bytes by shift-and-mask: register c byte i holds key 8 i + ((c + 2) & 7) as 2^-7 (c
//   even) or 2^-6 (c odd) (bits 2 and 3 of an e4m3 byte), eleven ALU operations per mask.
// B (shared memory, 32 keys x 16 columns, K-major no-swizzle): column 4 h + pc holds piece pc of
//   head h's weight, scaled by 2^7 or 2^6 to undo A's scale and by 2^-e (e from the chunk's largest
//   norm) so it fits e4m3; four pieces b0 + b1/16 + b2/256 + b3/4096 carry ~16 bits.
// D (TMEM, fp32): 16 columns per term, accumulated over the CTA's whole chunk of keys.
// The softmax uses two passes over the chunk (its logits staged in shared memory): the maximum
// first, then the weights, so the accumulators never need rescaling.  Per CTA: a chunk of up to
// kVChunkMax keys of one (batch, KV head, head quad); 4 warps (warp q: coordinates 32 q .. 32 q +
// 31, TMEM lanes 32 q ..); blocks of 32 keys through two A slots / B tiles / value stages; one
// thread issues the MMAs, tcgen05.commit frees a slot; every wait is bounded in time.  Output: the
// chunk's partial state (max, sum of exp, weighted sum in the value context's rotated basis) for
// attn_combine_kernel.
#include "mma_e4m3.cuh"
#include "tcgen05.cuh"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr uint32_t kVIdesc = tc::idesc_e4m3(16);   // M 128 (coordinates), N 16 (4 heads x 4 pieces), K 32 keys
constexpr int kVThreads = 128;                   // worker threads (4 warps); one more warp issues the MMAs
constexpr int kVChunkMax = 2048;                  // logits staged: 4 x 2048 floats = 32 KB
constexpr int kVSlots = 2;
constexpr int kVTmemCols = 128;                   // D: T x 16 columns, A slots: 2 x T x 8 (T <= 4)
// dynamic shared memory per CTA: sized so that at most 4 CTAs share an SM (4 x 128 TMEM columns)
constexpr size_t kVSmem = 52 * 1024;

struct VtcArgs {
    const float* logits;
    int B, Hq, Hkv, G, d;
    int64_t cap;
    const int32_t* len;
    int chunk, nchunk;
    int* err;
    const uint32_t* vplanes;   // [rows][P][4]
    const uint16_t* vnorm;
    float c0;
    float kappa[4];
    float* partials;
};

// 32 x 32 bit transposes across the warp, N matrices at once (their rounds interleaved so the
// shuffles overlap): on entry lane i holds row i of each (bit j = element (i, j)); on exit lane j
// holds column j (bit i = element (i, j)).  Five rounds; in round s lanes exchange with lane ^ s
// the half-blocks of size s that cross the diagonal.
template <int N>
__device__ __forceinline__ void transpose32(uint32_t (&x)[N], int lane) {
    const uint32_t m[5] = {0x0000FFFFu, 0x00FF00FFu, 0x0F0F0F0Fu, 0x33333333u, 0x55555555u};
#pragma unroll
    for (int r = 0; r < 5; ++r) {
        const int s = 16 >> r;
        uint32_t y[N];
#pragma unroll
        for (int n = 0; n < N; ++n) y[n] = __shfl_xor_sync(0xffffffffu, x[n], s);
        // lanes with bit s clear keep their low half-blocks and take the partner's low half-blocks
        // into their high ones; lanes with bit s set the mirror image
#pragma unroll
        for (int n = 0; n < N; ++n)
            x[n] = (lane & s) ? ((x[n] & ~m[r]) | ((y[n] >> s) & m[r])) : ((x[n] & m[r]) | ((y[n] << s) & ~m[r]));
    }
}

// Exact value of an e4m3 byte (hardware conversion through binary16, which holds every e4m3 value).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}

struct VShared {
    uint64_t ready[kVSlots];      // the 4 worker warps have written A and B of a block
    uint64_t slot_free[kVSlots];  // the block's MMAs are done (tcgen05.commit)
    uint64_t done;                // every MMA of the chunk is done
    uint32_t tmem;
    int abort;
    float red[4][8];
};

__device__ __forceinline__ void workers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// A bounded wait that also gives up at once once the CTA has aborted; on a time-out it records the
// abort (the CTA then runs to its end without further waiting and sets TQ_DEVERR_TIMEOUT).
__device__ __forceinline__ void wait_or_abort(VShared& S, uint64_t* bar, uint32_t parity) {
    if (*(volatile int*)&S.abort) return;
    if (!tc::mbar_wait(bar, parity)) *(volatile int*)&S.abort = 1;
}

template <int P>
__global__ void __launch_bounds__(kVThreads + 32) values_tc_kernel(const VtcArgs a) {
    constexpr int T = 1 << (P - 1);       // Walsh terms of a symmetric P-bit table
    constexpr int ROW = P * 4;            // words per value row
    constexpr int kStages = 3;            // value-row stages (prefetch distance 1)
    extern __shared__ __align__(128) unsigned char sm[];
    float* s_l = reinterpret_cast<float*>(sm);                                   // [4][kVChunkMax]
    float* s_n = s_l + 4 * kVChunkMax;                                           // [kVChunkMax] fp16 norms (half used)
    unsigned char* s_b = reinterpret_cast<unsigned char*>(s_n + kVChunkMax);     // [kVSlots][512]
    uint32_t* s_v = reinterpret_cast<uint32_t*>(s_b + kVSlots * 512);            // [kStages][32][ROW]
    __shared__ __align__(8) VShared S;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool worker = warp < 4;
    const int bh = blockIdx.y, b = bh / a.Hkv, kvh = bh - b * a.Hkv;
    const int L = checked_len(a.len, b, a.cap, a.err);
    const int64_t i0 = (int64_t)blockIdx.x * a.chunk;
    if (i0 >= L) return;
    const int hbase = kvh * a.G + 4 * blockIdx.z;
    const int nh = min(4, kvh * a.G + a.G - hbase);
    const int64_t iend = min((int64_t)L, i0 + a.chunk);
    const int nkeys = (int)(iend - i0);
    const int nblk = (nkeys + 31) / 32;
    const size_t rowbase = (size_t)bh * a.cap;
    const float* lg = a.logits + ((size_t)b * a.Hq + hbase) * a.cap;

    if (tid == 0) {
        for (int s = 0; s < kVSlots; ++s) {
            tc::mbar_init(&S.ready[s], 4);
            tc::mbar_init(&S.slot_free[s], 1);
        }
        tc::mbar_init(&S.done, 1);
        S.abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tc::tmem_alloc<kVTmemCols>(&S.tmem);
    }
    // pass 1 (worker warps): the chunk's logits (-inf beyond the keys and heads) and value norms
    // into shared memory, the maxima
    float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
    float nmax = 0.f;
    if (worker) {
        // asynchronous 4-byte copies (no load latency in the issuing threads), then the maxima
        // from shared memory; the norms travel as fp16 pairs, which the launcher's conditions (an
        // even capacity, a 4-byte aligned norm array; i0 is a multiple of 512) keep aligned and
        // inside the sequence's rows
        uint16_t* s_nh = reinterpret_cast<uint16_t*>(s_n);
#pragma unroll
        for (int h = 0; h < 4; ++h)
            if (h < nh)
                for (int i = tid; i < nkeys; i += kVThreads)
                    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(tc::smem_u32(s_l + h * kVChunkMax + i)),
                                 "l"(lg + (size_t)h * a.cap + i0 + i));
        for (int i = tid; i < (nkeys + 1) / 2; i += kVThreads)
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(tc::smem_u32(s_nh + 2 * i)),
                         "l"(a.vnorm + rowbase + i0 + 2 * i));
        asm volatile("cp.async.commit_group;");
        asm volatile("cp.async.wait_all;");
        workers_sync();
#pragma unroll
        for (int h = 0; h < 4; ++h)
            for (int i = tid; i < a.chunk; i += kVThreads) {
                float v = -INFINITY;
                if (h < nh && i < nkeys) v = s_l[h * kVChunkMax + i];
                else s_l[h * kVChunkMax + i] = -INFINITY;
                mx[h] = fmaxf(mx[h], v);
            }
        for (int i = tid; i < nkeys; i += kVThreads) nmax = fmaxf(nmax, half_bits_to_float(s_nh[i]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
            for (int h = 0; h < 4; ++h) mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], o));
            nmax = fmaxf(nmax, __shfl_xor_sync(0xffffffffu, nmax, o));
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h) S.red[h][warp] = mx[h];
            S.red[0][4 + warp] = nmax;
        }
    }
    asm volatile("tcgen05.fence::before_thread_sync;");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;");
    const uint32_t tmem = S.tmem;

    if (!worker) {
        // the MMA warp: per block, once the workers have written its A and B, T mma and a commit
        if (lane == 0) {
            for (int j = 0; j < nblk; ++j) {
                const int slot = j % kVSlots;
                wait_or_abort(S, &S.ready[slot], (uint32_t)((j / kVSlots) & 1));
                if (*(volatile int*)&S.abort) break;
                asm volatile("tcgen05.fence::after_thread_sync;");
                const uint64_t bd = tc::kmajor_desc(tc::smem_u32(s_b + slot * 512), 256);   // 16 rows x 32 k
#pragma unroll
                for (int t = 0; t < T; ++t)
                    tc::mma_e4m3_ts<kVIdesc>(tmem + 16 * t, tmem + 16 * T + slot * 8 * T + 8 * t, bd, j > 0 ? 1u : 0u);
                tc::commit(&S.slot_free[slot]);
            }
            tc::commit(&S.done);   // completes once every MMA issued before it has
        }
        __syncwarp();
    } else {
        float M[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) M[h] = fmaxf(fmaxf(S.red[h][0], S.red[h][1]), fmaxf(S.red[h][2], S.red[h][3]));
        nmax = fmaxf(fmaxf(S.red[0][4], S.red[0][5]), fmaxf(S.red[0][6], S.red[0][7]));
        // B values: w n 2^-e with 2^-e n_max in [1/2, 1), times 2^7 or 2^6
        int e = 0;
        frexpf(nmax, &e);
        const float nscale = ldexpf(1.f, -e);
        // this thread's weights: key kq = tid / 4 of each block, head hq = tid % 4
        const int kq = tid >> 2, hq = tid & 3;
        const int kperm = 4 * ((kq + 6) & 7) + (kq >> 3);     // its position along K (A's byte order)
        const float kscale = (((kq + 6) & 7) & 1) ? 64.f : 128.f;
        float lsum = 0.f, wsum = 0.f;   // sum of exp(l - M) and of exp(l - M) n for head hq
        const uint32_t a_tmem = tmem + ((uint32_t)(32 * warp) << 16) + 16 * T;   // A slots after D
        auto stage_rows = [&](int j) {   // value rows of block j into stage j % kStages
            const int k0 = 32 * j, n = min(32, nkeys - k0);
            const uint4* src = reinterpret_cast<const uint4*>(a.vplanes + (rowbase + i0 + k0) * ROW);
            uint4* dst = reinterpret_cast<uint4*>(s_v + (j % kStages) * 32 * ROW);
            for (int q = tid; q < n * P; q += kVThreads) tc::cp_async16(dst + q, src + q);
            asm volatile("cp.async.commit_group;");
        };
        stage_rows(0);
        for (int j = 0; j < nblk; ++j) {
            const int slot = j % kVSlots;
            // rows of block j + 1 into stage (j + 1) % 3, last read by block j - 2's transposes,
            // which every worker finished before the barrier of block j - 1
            if (j + 1 < nblk) stage_rows(j + 1);
            else asm volatile("cp.async.commit_group;");
            // A and B of this slot were read by block j - 2's MMAs
            if (j >= kVSlots) wait_or_abort(S, &S.slot_free[slot], (uint32_t)(((j / kVSlots) - 1) & 1));
            asm volatile("tcgen05.fence::after_thread_sync;");
            // weights of block j -> B tile (4 e4m3 pieces per head)
            {
                const int k = 32 * j + kq;
                const bool valid = k < nkeys && hq < nh;
                const float ex = valid ? __expf(s_l[hq * kVChunkMax + k] - M[hq]) : 0.f;
                const float vn = valid ? half_bits_to_float(reinterpret_cast<const uint16_t*>(s_n)[k]) : 0.f;
                lsum += ex;
                wsum = fmaf(ex, vn, wsum);
                float x = ex * vn * nscale * kscale;
                unsigned char* bt = s_b + slot * 512;
#pragma unroll
                for (int pc = 0; pc < 4; ++pc) {
                    const uint32_t byte = to_e4m3(x);
                    bt[tc::kmajor8(4 * hq + pc, kperm, 32)] = (unsigned char)byte;
                    x = (x - e4m3_value(byte)) * 16.f;
                }
            }
            asm volatile("cp.async.wait_group 1;");   // block j's rows have landed (j + 1's may not)
            asm volatile("fence.proxy.async.shared::cta;");
            workers_sync();
            // A: this warp's 32 coordinates x the block's 32 keys, per term
            {
                const uint32_t* rows = s_v + (j % kStages) * 32 * ROW;
                uint32_t msk[P];
#pragma unroll
                for (int p = 0; p < P; ++p) msk[p] = rows[lane * ROW + p * 4 + warp];
                transpose32<P>(msk, lane);
                const uint32_t at = a_tmem + slot * 8 * T;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    uint32_t x = 0u;
#pragma unroll
                    for (int p = 0; p < P; ++p)
                        if ((odd_mask(t) >> p) & 1) x ^= msk[p];
                    uint32_t r[8];
                    tc::expand_word(x, r);
                    tc::tmem_st8(at + 8 * t, r);
                }
                asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
            }
            asm volatile("tcgen05.fence::before_thread_sync;");
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&S.ready[slot]);
        }
        asm volatile("cp.async.wait_all;");
        wait_or_abort(S, &S.done, 0);
        asm volatile("tcgen05.fence::after_thread_sync;");
        // sums per head: threads with the same head hq (tid % 4)
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
            wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
        }
        workers_sync();   // every worker has read S.red (the maxima) before it is reused
        if (lane < 4) {
            S.red[lane][warp] = lsum;
            S.red[lane][4 + warp] = wsum;
        }
        // D of this lane's coordinate: term t, column 4 h + pc
        float dv[4][16];
        const uint32_t d_tmem = tmem + ((uint32_t)(32 * warp) << 16);
#pragma unroll
        for (int t = 0; t < T; ++t) tc::tmem_ld16(d_tmem + 16 * t, dv[t]);
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        workers_sync();
        if (!*(volatile int*)&S.abort) {
            const float unscale = 1.f / nscale;
            const int jc = 32 * warp + lane;
            const size_t stride = (size_t)a.d + 2;
            const size_t hstride = (size_t)a.nchunk * stride;
            float* pbase = a.partials + (((size_t)b * a.Hq + hbase) * a.nchunk + blockIdx.x) * stride;
            for (int h = 0; h < nh; ++h) {
                const float W = (S.red[h][4] + S.red[h][5]) + (S.red[h][6] + S.red[h][7]);
                float acc = a.c0 * W;
#pragma unroll
                for (int t = 0; t < T; ++t) {
                    const float sv = fmaf(dv[t][4 * h + 3], 1.f / 4096.f,
                                          fmaf(dv[t][4 * h + 2], 1.f / 256.f, fmaf(dv[t][4 * h + 1], 1.f / 16.f, dv[t][4 * h])));
                    acc = fmaf(a.kappa[t], sv * unscale, acc);
                }
                if (jc < a.d) pbase[h * hstride + 2 + jc] = acc;
                if (tid == 0) {
                    pbase[h * hstride] = M[h];
                    pbase[h * hstride + 1] = (S.red[h][0] + S.red[h][1]) + (S.red[h][2] + S.red[h][3]);
                }
            }
        }
    }
    tc::fence_before();
    __syncthreads();
    bool drained = true;
    if (*(volatile int*)&S.abort) {   // a wait ran out: flag it, and let the issued MMAs finish (bounded)
        if (tid == 0) set_error(a.err, TQ_DEVERR_TIMEOUT);
        drained = __syncthreads_and(tid != 0 || tc::mbar_wait(&S.done, 0u));
    }
    tc::fence_after();
    // an MMA that outlived the bounded drain still writes this memory: it is then left allocated
    if (warp == 0 && drained) tc::tmem_dealloc<kVTmemCols>(tmem);
}

}  // namespace

bool values_tc_supported(const tq_ctx* vc, int d) {
    if (!vc) return false;
    const Params& p = vc->prm;
    return d > 96 && d <= 128 && p.W == 4 && p.P >= 1 && p.P <= 3 && p.odd_walsh && p.d_hi == 0;
}

// Keys per CTA: the largest power of two in [512, kVChunkMax] that still gives every SM two rounds
// of 4 CTAs over all (batch, KV head, head quad) groups.
int values_tc_chunk(int B, int Hq, int Hkv, int64_t cap) {
    const int64_t groups = (int64_t)B * Hkv * ((Hq / Hkv + 3) / 4);
    int c = kVChunkMax;
    while (c > 512 && groups * ((cap + c - 1) / c) < 148 * 4 * 2) c >>= 1;
    return c;
}

cudaError_t launch_values_tc(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                             const int32_t* len, const void* values, const uint16_t* vnorm, int* err, float* partials,
                             int chunk, int nchunk, cudaStream_t s) {
    VtcArgs a{};
    a.logits = logits;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.d = d;
    a.cap = cap;
    a.len = len;
    a.chunk = chunk;
    a.nchunk = nchunk;
    a.err = err;
    a.vplanes = static_cast<const uint32_t*>(values);
    a.vnorm = vnorm;
    const Params& p = vc->prm;
    a.c0 = p.c0;
    for (int t = 0; t < 4; ++t) a.kappa[t] = t < p.nterms ? p.kappa[t] : 0.f;
    a.partials = partials;
    dim3 grid(nchunk, B * Hkv, (a.G + 3) / 4);
    cudaError_t e;
    switch (p.P) {
        case 1:
            e = cudaFuncSetAttribute(values_tc_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVSmem);
            if (e != cudaSuccess) return e;
            values_tc_kernel<1><<<grid, kVThreads + 32, kVSmem, s>>>(a);
            break;
        case 2:
            e = cudaFuncSetAttribute(values_tc_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVSmem);
            if (e != cudaSuccess) return e;
            values_tc_kernel<2><<<grid, kVThreads + 32, kVSmem, s>>>(a);
            break;
        default:
            e = cudaFuncSetAttribute(values_tc_kernel<3>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVSmem);
            if (e != cudaSuccess) return e;
            values_tc_kernel<3><<<grid, kVThreads + 32, kVSmem, s>>>(a);
            break;
    }
    return cudaGetLastError();
}

}  // namespace tq
