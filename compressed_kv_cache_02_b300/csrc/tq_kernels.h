// Launchers of the libtq kernels (host side).  Each returns cudaGetLastError() of its
// launches; arguments are already validated by tq_api.cu.
#pragma once

#include <cuda_runtime.h>

#include <vector>

#include "tq_internal.h"

namespace tq {

// rows v < nv: out[v*ldo + i] = sum_j MT[j*dout + i] * in[v*ldi + j],  i < dout, j < din.
cudaError_t launch_apply_rows(const float* MT, int din, int dout, const float* in, size_t ldi,
                              int64_t nv, float* out, size_t ldo, cudaStream_t s);

// Quantize rows.  Row v of the input is x + v*ld_x; its output row is v (cap == 0) or
// v*cap + len[v / H] (decode append, cap > 0).
cudaError_t launch_quantize(const tq_ctx* c, const void* x, int dtype, int64_t n, int64_t ld_x,
                            int H, int64_t cap, const int32_t* len, uint32_t* planes,
                            uint32_t* signs, uint16_t* norm, uint16_t* rnorm, cudaStream_t s);

// tcgen05 bulk quantize (bf16 rows, d = 128).
bool quantize_tc_supported(const tq_ctx* c, int dtype, const void* x, int64_t n, int64_t ld_x);
void build_tc_operands(const float* Pi, const float* St, std::vector<uint16_t>& out);
cudaError_t launch_quantize_tc(const tq_ctx* c, const void* x, int64_t n, int64_t ld_x, uint32_t* planes,
                               uint32_t* signs, uint16_t* norm, uint16_t* rnorm, cudaStream_t s);

// tcgen05 polar-angle encoder (bf16 rows, d = 128, 7 levels of angles), k_quantize_tc.cu.
// bops: build_tc_operands(Pi, S Pi^T or NULL) on the device; cs: [7][32] floats, level l - 1 at
// 32 (l - 1): the cosines of its 2^bits centroids, then at + 16 their sines; tau: levels 2..7 (at
// l - 2), tan^2 of the level's 2^bits - 1 ascending thresholds (level 1 is the uniform sectors).
// Needs x 16-byte aligned and ld_x a multiple of 8.
struct PolarTcLaunch {
    int device;
    const void* x;
    int64_t n, ld_x;
    const void* bops;
    const float* cs;
    int bits, qjl, cw;
    float tau[6][15];
    uint32_t* codes;
    uint16_t* r16;
    uint32_t* signs;
    uint16_t* rnorm;
    int* err;
};
cudaError_t launch_polar_tc(const PolarTcLaunch& L, cudaStream_t s);

cudaError_t launch_advance_len(int32_t* len, int B, int64_t cap, int step, int* err, cudaStream_t s);

struct KeyCache {
    const uint32_t* planes;
    const uint32_t* signs;
    const uint16_t* norm;
    const uint16_t* rnorm;
    int64_t cap;
    const int32_t* len;
};

// Keys per CTA and the number of sequence chunks for an attention launch.
void attn_chunking(const tq_ctx* kc, int B, int Hq, int Hkv, int64_t cap, int* chunk, int* nchunk);

// logits[b][h][i] for i < len[b]; qrot/qproj prepared rows [B*Hq][d] / [B*Hq][m].
// image: scratch of logits_tc_image_bytes(B, Hq, Hkv) bytes for the tensor-core path.
cudaError_t launch_logits(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq,
                          int Hkv, const KeyCache& k, float scale, float* logits, void* image, cudaStream_t s);

// Tensor-core logits (tcgen05.mma kind::f8f6f4, A in TMEM) for 96 < d <= 128, m <= 128 and
// 1..3 MSE bits; usable when the cache also meets the bulk-copy alignment (16-byte fields,
// capacity a multiple of 8).  image: logits_tc_image_bytes(B, Hq, Hkv) bytes, 128-byte aligned.
bool logits_tc_supported(const tq_ctx* kc);
bool logits_tc_ok(const tq_ctx* kc, const KeyCache& k);
size_t logits_tc_image_bytes(int B, int Hq, int Hkv);
cudaError_t launch_logits_tc(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                             const KeyCache& k, float scale, float* logits, void* image, cudaStream_t s);

// Logits for split (fractional bit width) key contexts (prm.d_hi > 0), any d <= TQ_MAX_D.
cudaError_t launch_logits_split(const tq_ctx* kc, const float* qrot, const float* qproj, int B, int Hq, int Hkv,
                                const KeyCache& k, float scale, float* logits, cudaStream_t s);

// Split-sequence attention output: per-chunk partials (max, sum, acc[d]) then the combine.
cudaError_t launch_attn_output(const tq_ctx* kc, const tq_ctx* vc, const float* qrot,
                               const float* qproj, int B, int Hq, int Hkv, const KeyCache& k,
                               float scale, const void* values, const uint16_t* vnorm,
                               float* partials, float* out, cudaStream_t s);

// Softmax + value sum from precomputed logits, then the combine (vc NULL: bf16 values of dim d).
// part_out non-NULL: instead of the combine, one unnormalised partial state per (batch, head),
// [B*Hq][d + 2] = (max, sum of weights, weighted sum in the rotated basis), for a shard merge.
// allow_tc: the tensor-core kernel may be chosen (its chunking needs the workspace of
// values_ws_bytes in tq_api.cu; callers with a fixed smaller scratch pass false).
cudaError_t launch_attn_values(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                               const int32_t* len, const void* values, const uint16_t* vnorm, int* err,
                               float* partials, float* out, cudaStream_t s, float* part_out = nullptr,
                               bool allow_tc = true);

// Tensor-core value sum (tcgen05, k_values_tc.cu): MSE value contexts with 96 < d <= 128, 1..3 bits,
// symmetric tables, not split.  Writes the chunk partials of launch_attn_values' layout for chunks
// of values_tc_chunk() keys.
bool values_tc_supported(const tq_ctx* vc, int d);
int values_tc_chunk(int B, int Hq, int Hkv, int64_t cap);
cudaError_t launch_values_tc(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                             const int32_t* len, const void* values, const uint16_t* vnorm, int* err, float* partials,
                             int chunk, int nchunk, cudaStream_t s);

// out[bh] from R shards' partial states parts [R][BH][d + 2] (log-sum-exp merge, then Pi_v^T).
cudaError_t launch_merge_partials(const tq_ctx* vc, int d, const float* parts, int R, int64_t BH, float* out,
                                  cudaStream_t s);

// Global top-k from R shards' lists cand [R][nq][k] (row numbers local to each shard, shifted by
// offsets[r]; an entry with index INT_MAX is padding).
constexpr int kMaxShards = 64;
struct ShardOffsets {
    long long off[kMaxShards];
};
cudaError_t launch_topk_merge(const float* cand_s, const int32_t* cand_i, int R, int64_t nq, int k,
                              const ShardOffsets& offs, float* top_s, int32_t* top_i, cudaStream_t s);

// Search: per-chunk top-k candidates into cand (score, index pairs), then the merge.
void search_chunking(int64_t n, int k, int* chunk, int* nchunk);
cudaError_t launch_search(const tq_ctx* c, const float* qrot, const float* qproj, int64_t nq,
                          const uint32_t* planes, const uint32_t* signs, const uint16_t* norm,
                          const uint16_t* rnorm, int64_t n, int k, float* cand_s, int* cand_i,
                          float* top_s, int32_t* top_i, cudaStream_t s);

}  // namespace tq
