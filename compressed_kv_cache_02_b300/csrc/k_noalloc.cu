// tq_attn_values_noalloc: the softmax + value step with its scratch in a fixed device array.
//
// Who needs this: callers that may not allocate device memory while they run.  Examples are
// a serving process that reserves all of its device memory in its own pool at start-up and
// forbids further cudaMalloc calls (an allocation can synchronise the device and can fail in
// the middle of a request), or a plugin host that hands kernels buffers but no allocator.
// Those callers can still pass the inputs and the output, but not a workspace.
//
// The scratch (the per-chunk partial softmax states) lives in the static array below.  Every
// GPU that loads this library holds the array until the process exits.  All calls on a device
// share it and it keeps what the last call wrote; the kernels write every partial they later
// read, so nothing has to start at zero.  Calls whose work overlaps on the GPU (different
// streams without ordering, or several host threads) race on the array.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "tq_internal.h"
#include "tq_kernels.h"

namespace tq {
namespace {

constexpr size_t kNoAllocScratchBytes = TQ_NOALLOC_SCRATCH_BYTES;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device with that device current.
constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

int scratch_for_current_device(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return fail(TQ_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return fail(TQ_ERR_UNSUPPORTED, "device ordinal above 63");
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(TQ_ERR_CUDA, std::string("cudaGetSymbolAddress of the static scratch: ") + cudaGetErrorString(e));
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TQ_OK;
}

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" int tq_attn_values_noalloc(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv,
                                      int64_t cap, const int32_t* len, const void* values, const uint16_t* v_norm,
                                      float* out, void* stream) {
    if (vc) {
        int dev = -1;
        if (cudaGetDevice(&dev) != cudaSuccess || dev != vc->device)
            return fail(TQ_ERR_ARG, "the value context belongs to another device than the current one");
        if (vc->mode != TQ_MODE_MSE) return fail(TQ_ERR_ARG, "vctx must be an MSE-mode context");
        if (vc->d_hi) return fail(TQ_ERR_UNSUPPORTED, "split (fractional bit width) value contexts are not supported");
        if (vc->d != d) return fail(TQ_ERR_ARG, "d must equal vctx's d");
        if (!v_norm || !aligned_to(v_norm, 2)) return fail(TQ_ERR_ARG, "coded values need v_norm");
    }
    if (d < 1 || d > 512) return fail(TQ_ERR_UNSUPPORTED, "tq_attn_values_noalloc supports d <= 512");
    if (B < 1 || Hkv < 1 || Hq < Hkv || Hq % Hkv != 0)
        return fail(TQ_ERR_ARG, "need B >= 1 and Hq a positive multiple of Hkv");
    if (cap < 1 || cap >= ((int64_t)1 << 31)) return fail(TQ_ERR_ARG, "cap must be in [1, 2^31)");
    if (!logits || !len || !values || !out) return fail(TQ_ERR_ARG, "a required pointer is NULL");
    if (!aligned_to(logits, 4) || !aligned_to(len, 4) || !aligned_to(values, 16) || !aligned_to(out, 4))
        return fail(TQ_ERR_ARG, "misaligned pointer");
    int chunk, nchunk;
    attn_chunking(nullptr, B, Hq, Hkv, cap, &chunk, &nchunk);
    const size_t need = (size_t)B * Hq * nchunk * (d + 2) * sizeof(float);
    if (need > kNoAllocScratchBytes)
        return fail(TQ_ERR_UNSUPPORTED, "tq_attn_values_noalloc needs " + std::to_string(need) +
                                            " bytes of scratch for these shapes; its static array holds " +
                                            std::to_string(kNoAllocScratchBytes) + " (use tq_attn_values)");
    void* scratch = nullptr;
    int rc = scratch_for_current_device(&scratch);
    if (rc != TQ_OK) return rc;
    cudaError_t e = launch_attn_values(vc, d, logits, B, Hq, Hkv, cap, len, values, v_norm, vc ? vc->derr : nullptr,
                                       static_cast<float*>(scratch), out, static_cast<cudaStream_t>(stream), nullptr,
                                       false);
    if (e != cudaSuccess)
        return fail(TQ_ERR_CUDA, std::string("tq_attn_values_noalloc launch: ") + cudaGetErrorString(e));
    return TQ_OK;
}
