// tcgen05 / mbarrier primitives (inline PTX for sm_103a) shared by the tensor-core kernels:
// bounded mbarrier waits, tensor-memory allocation, loads and stores, MMA issue and commit for
// kind::f8f6f4 with A in tensor memory, K-major no-swizzle shared-memory descriptors, and the
// expansion of a 32-bit bit vector into e4m3 bytes.
#pragma once

#include <cstdint>

namespace tq {
namespace tc {
namespace {

constexpr int kSuspendNs = 20000;              // suspend-time hint of one try_wait
constexpr uint64_t kWaitNs = 1000000000ull;    // a wait gives up after one second

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase with the given parity to complete.  Each try_wait may suspend the thread
// for up to kSuspendNs (it resumes as soon as the phase completes); false once kWaitNs of
// wall-clock time (the GPU's global timer) have passed.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
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
__device__ __forceinline__ void mbar_init(uint64_t* bar, int count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
// Arrives on bar once every tcgen05 operation this thread issued before has completed.
__device__ __forceinline__ void commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar)));
}
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// Generic-proxy writes to shared memory made visible to the tensor cores' (async proxy) reads.
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Whole-warp tensor-memory allocation of COLS columns (a power of two >= 32); the address is
// written to *dst in shared memory.
template <int COLS>
__device__ __forceinline__ void tmem_alloc(uint32_t* dst) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)), "n"(COLS));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
template <int COLS>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "n"(COLS));
}

// 32 lanes x N consecutive 32-bit columns, one lane per thread of the warp.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
#pragma unroll
    for (int j = 0; j < 8; ++j) v[j] = __uint_as_float(r[j]);
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
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    float a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        v[j] = a[j];
        v[16 + j] = b[j];
    }
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
                 "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]));
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
            taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]));
}

__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(smem_u32(smem)), "l"(gmem));
}

// Instruction descriptor of kind::f8f6f4 with e4m3 A and B, fp32 D, both K-major, M = 128.
__host__ __device__ constexpr uint32_t idesc_e4m3(int n) { return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((128u >> 4) << 24); }

// D[128 x N] (+)= A[128 x 32] B[32 x N]: A from tensor memory, B from shared memory.
template <uint32_t IDESC>
__device__ __forceinline__ void mma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(IDESC), "r"(accumulate));
}

// K-major no-swizzle operand: core matrices of 8 rows x 16 bytes, LBO = 128 B along K,
// SBO = sbo bytes between 8-row groups; descriptor version 1.  Adding 16 to the descriptor moves
// its start 256 bytes on, i.e. one K step of 32 e4m3 values.
__device__ __forceinline__ uint64_t kmajor_desc(uint32_t saddr, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFF) | ((uint64_t)(128 >> 4) << 16) | ((uint64_t)((sbo >> 4) & 0x3FFF) << 32) |
           ((uint64_t)1 << 46);
}
// Byte offset of element (row r, k) in a [rows x ktot] 8-bit K-major no-swizzle operand.
__host__ __device__ __forceinline__ uint32_t kmajor8(int r, int k, int ktot) {
    return (uint32_t)(((r >> 3) * (ktot >> 4) + (k >> 4)) * 128 + (r & 7) * 16 + (k & 15));
}

// A bit vector as e4m3 bytes.  Bits 2 and 3 of a byte are, as e4m3, exactly 2^-7 (subnormal
// 4 x 2^-9) and 2^-6 (the smallest normal), so masking shifted copies of a 32-bit word gives four
// coordinates per register: register c holds in byte i bit 8 i + ((c + 2) & 7) of x, with value
// 2^-7 (c even) or 2^-6 (c odd).  The matching B operand scales its values by 2^7 or 2^6.
__device__ __forceinline__ void expand_word(uint32_t x, uint32_t* r) {
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
// Position k (within a word's 32 e4m3 bytes, as expand_word lays them out) of coordinate jj of
// the word, and the B scale that undoes the A value there.
__host__ __device__ __forceinline__ int expanded_k(int jj) { return 4 * (((jj & 7) - 2) & 7) + (jj >> 3); }
__host__ __device__ __forceinline__ float expanded_scale(int jj) { return (((jj & 7) - 2) & 1) ? 64.f : 128.f; }

// The W words of one bit vector into tensor-memory columns col .. col + 8 W - 1 of this warp's
// 32 lanes (8 columns per word), in stores of 32, 16 and 8 columns.
template <int W>
__device__ __forceinline__ void store_bits(uint32_t col, const uint32_t (&w)[W]) {
    int wd = 0;
#pragma unroll
    for (; wd + 4 <= W; wd += 4) {
        uint32_t r[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) expand_word(w[wd + i], r + 8 * i);
        tmem_st32(col + 8 * wd, r);
    }
    if (W - wd >= 2) {
        uint32_t r[16];
        expand_word(w[wd], r);
        expand_word(w[wd + 1], r + 8);
        tmem_st16(col + 8 * wd, r);
        wd += 2;
    }
    if (W - wd >= 1) {
        uint32_t r[8];
        expand_word(w[wd], r);
        tmem_st8(col + 8 * wd, r);
    }
}

}  // namespace
}  // namespace tc
}  // namespace tq
