/*
 * tq.h -- C-ABI of libtq: the TurboQuant hot path on B300 (sm_103a).
 *
 * Method (source pages, by title and section):
 *   - juejin.cn post 7621817220135075850, section 二 "TurboQuant 的两段式": a random
 *     rotation then scalar quantization that spends most of the bits (PolarQuant), and
 *     ~1 bit of QJL on the residual; an asymmetric estimator pairs a high-precision query
 *     with the low-precision codes.
 *   - gitcode.csdn.net TurboQuant tutorial, sections "TurboQuant原理剖析" (r at 16 bits,
 *     2- or 3-bit codes plus 1 QJL bit = 3 or 4 bits in total), "PolarQuant" (rotate
 *     first), "将笛卡尔积坐标转为极坐标" (r = ||x|| kept as FP16) and "QJL" steps 1-3
 *     (residual = original minus reconstruction, Gaussian JL projection, keep the signs:
 *     > 0 -> 1, < 0 -> 0; the query against the signs gives an unbiased correction).
 *   - freelamp.com article 0328, sections "技术突破：极坐标量化" (random orthogonal
 *     rotation, no per-block scaling constants) and "误差补偿：QJL 变换与 1-bit 残差修正"
 *     (zero-bias estimate from 1-bit residual signs and the high-precision query).
 *   - juejin.cn post, section 三 (attention logits over the compressed KV cache; GloVe
 *     d=200 Recall@1@k search) and section 四 (data-oblivious, online, near-optimal).
 *
 * What a context computes, for a vector x in R^d (the readings the pages leave open are
 * stated with each step):
 *   n      = ||x||_2, stored as IEEE binary16 (round to nearest even)
 *   u      = Pi x / n            (u = 0 when n = 0); Pi a d x d random orthogonal matrix
 *   idx_j  = number of thresholds t_k with t_k < u_j  (nearest centroid; a value exactly on
 *            a threshold takes the lower index); centroids/thresholds are the Lloyd-Max
 *            quantizer of one coordinate of a uniform unit vector in R^d (reading: the
 *            rotated direction is exactly uniform on the sphere, so this table is
 *            data-oblivious and the same for every token and layer)
 *   PROD mode (bits = MSE bits + 1 QJL bit):
 *   r      = x - n16 Pi^T c[idx]  (the residual of the PolarQuant reconstruction)
 *   rnorm  = ||r||_2 as binary16 (reading: needed by the unbiased estimator)
 *   sign_j = [(S r)_j > 0] for j < m, S an m x d matrix of i.i.d. N(0,1) (exact 0 -> bit 0)
 *   MSE mode: only n and idx (bits = MSE bits).
 * Estimator for a full-precision query q (PROD keys):
 *   est(q, x) = n16 <Pi q, c[idx]> + rnorm16 sqrt(pi/2)/m <S q, 2 sign - 1>
 *   (the constant makes the correction unbiased: E_S[...] = <q, r>; the pages do not print it).
 *   MSE keys: est = n16 <Pi q, c[idx]>.
 *
 * Packed layout (the library's contract; the CPU oracle produces the same bytes):
 *   planes  uint32 [rows][P][W]   P = MSE bits, W = ceil(d/32); bit (j mod 32) of word
 *                                 j/32 of plane p holds bit p of idx_j; pad bits are 0
 *   signs   uint32 [rows][Ws]     Ws = ceil(m/32); bit (j mod 32) of word j/32 = sign_j
 *   norm    uint16 [rows]         binary16 bit pattern of n
 *   rnorm   uint16 [rows]         binary16 bit pattern of ||r||
 *   A KV cache is [B][Hkv][cap] rows; query head h reads KV head h / (Hq/Hkv).
 *
 * Conventions for every call:
 *   - Return value: TQ_OK or a TQ_ERR_* code; tq_last_error() gives a thread-local message.
 *     No call aborts the process.
 *   - Host arguments are checked before any launch (TQ_ERR_ARG / TQ_ERR_UNSUPPORTED).
 *   - Device pointers are caller-owned device memory (e.g. allocated by PyTorch); the
 *     library never allocates or frees them.  uint32 and float arrays must be 16-byte
 *     aligned; uint16 arrays 2-byte aligned.  bf16 inputs are raw bfloat16 bit patterns.
 *   - Compute calls are asynchronous on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).  The return status covers validation and launch errors;
 *     checks that can only run on the device (an fp16 norm overflow, len > cap) set bits of
 *     the context's device error word, which tq_sync_status() returns and clears.
 *   - The context must be used on the device that was current at tq_init*; calls on one
 *     context are not thread-safe against each other.
 *   - The library does not allocate in compute calls: scratch is the caller's `workspace`,
 *     sized by the *_workspace_size() calls.  tq_init* allocates the context's tables.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum tq_status {
    TQ_OK = 0,
    TQ_ERR_ARG = 1,          /* an argument is out of range, NULL or misaligned      */
    TQ_ERR_CUDA = 2,         /* a CUDA runtime call or kernel launch failed          */
    TQ_ERR_OOM = 3,          /* tq_init* could not allocate the context's tables     */
    TQ_ERR_UNSUPPORTED = 4,  /* a valid request this build does not implement        */
    TQ_ERR_DEVICE = 5        /* tq_sync_status: a device-side check failed           */
};

enum tq_dtype { TQ_F32 = 0, TQ_BF16 = 1 };
enum tq_mode { TQ_MODE_PROD = 0, TQ_MODE_MSE = 1 };

/* Bits of the device error word (returned through tq_sync_status' *flags). */
enum tq_device_error {
    TQ_DEVERR_NORM_OVERFLOW = 1,   /* a norm or residual norm rounded to binary16 infinity */
    TQ_DEVERR_LEN_RANGE = 2,       /* a len[b] was negative or above cap (clamped)         */
    TQ_DEVERR_TIMEOUT = 4          /* a bounded wait for the tensor cores gave up          */
};

#define TQ_MAX_D 1024
#define TQ_MAX_MSE_BITS 8   /* MSE mode; PROD mode takes 1..4 MSE bits (bits 2..5) */
#define TQ_MAX_TOPK 128

typedef struct tq_ctx tq_ctx;

/* ---------------------------------------------------------------- host-only helpers
 * These run on the CPU and need no GPU.                                              */

/* The Lloyd-Max codebook of one coordinate of a uniform unit vector in R^d: 2^mse_bits
 * centroids (ascending, index 0 the most negative) and 2^mse_bits - 1 thresholds, in
 * float64, computed by the Lloyd iteration with Gauss-Legendre quadrature of the density
 * Gamma(d/2)/(sqrt(pi)Gamma((d-1)/2)) (1-t^2)^((d-3)/2).  Pages: nonndazone.ru essay,
 * sections 3.2 (centroids where probability is higher) and 3.4 (precomputed once);
 * freelamp article, section 技术突破 (predictable law after rotation).  The table is the fixed
 * point of the Lloyd-Max conditions (midpoint thresholds, centroids at the cell means): up to 4
 * bits reached by the Lloyd iteration, from 5 bits by Newton's method on the same conditions.
 * 3 <= d <= TQ_MAX_D, 1 <= mse_bits <= TQ_MAX_MSE_BITS.  Arrays are caller-owned.     */
int tq_host_codebook(int d, int mse_bits, double* centroids, double* thresholds);

/* The seeded matrices of tq_init: Pi (d x d, row-major, Haar-random orthogonal) and S
 * (m x d, row-major, i.i.d. N(0,1)), rounded to float32.  Generator: splitmix64(seed) ->
 * uniforms ((z >> 11) + 1) * 2^-53 -> Box-Muller pairs (cos, sin); S takes normals
 * 0..m*d-1, the Gaussian G for Pi the next d*d; Pi = Q diag(sign(diag R)), G = QR
 * (Householder, float64).  Pages: freelamp article, section 技术突破 (random orthogonal
 * rotation); csdn tutorial, section QJL step 1 (Gaussian projection).  S may be NULL.  */
int tq_host_matrices(uint64_t seed, int d, int m, float* Pi, float* S);

/* ---------------------------------------------------------------- contexts */

/* PROD-mode context: bits = MSE bits + 1 QJL bit (2..5), m = d, matrices
 * from tq_host_matrices(seed, d, d).  Allocates the context's device tables on the
 * current device.  Pages: csdn tutorial, section TurboQuant原理剖析 (2+1 and 3+1 bits).   */
int tq_init(tq_ctx** out, uint64_t seed, int d, int bits);

/* General context.  mode TQ_MODE_PROD: bits = MSE bits + 1 (2..5), m = JL rows (1..TQ_MAX_D);
 * mode TQ_MODE_MSE: bits = MSE bits (1..TQ_MAX_MSE_BITS), m ignored (no QJL stage).
 * Contexts of 1..4 MSE bits take the table and tensor-core kernels; MSE contexts of 5..8 bits
 * take the generic CUDA-core kernels of every call (tq_quantize, tq_append, tq_attn_logits,
 * tq_attn_output, tq_attn_values, tq_search_topk) with the same results' contract;
 * tq_paged_decode_step takes 1..4-bit value contexts only (TQ_ERR_UNSUPPORTED otherwise).
 * Pi_host (d x d) and S_host (m x d, PROD only) are float32 row-major host arrays used as
 * given (copied); NULL means "generate from seed" as tq_host_matrices does.  Pi_host must
 * be orthogonal to float32 precision (not checked beyond finiteness).                  */
int tq_init_ex(tq_ctx** out, uint64_t seed, int d, int bits, int mode, int m,
               const float* Pi_host, const float* S_host);

/* Split (fractional bit width) context.  Pages: juejin.cn post, section 四 (KV quality at 3.5
 * and 2.5 bits per channel).  Reading: the first d_hi rotated coordinates are coded with the
 * (b+1)-bit Lloyd-Max table and the other d - d_hi with the b-bit one (b = MSE bits given by
 * bits and mode as in tq_init_ex; the QJL stage is unchanged), i.e. b + d_hi / d MSE bits per
 * coordinate on average: bits = 3, d_hi = d/2, PROD gives 3.5 bits per channel.
 * d_hi must be a multiple of 32 in [0, d] and b + 1 <= 4; d_hi = 0 is tq_init_ex.
 * Code rows: the b full planes (W words each, as tq_layout) followed by the top plane of the
 * first d_hi coordinates (ceil(d_hi / 32) words: bit j % 32 of word j / 32 holds bit b of
 * idx_j); tq_code_words gives the row length.  tq_quantize, tq_append and tq_attn_logits
 * accept split contexts (CUDA-core kernels), and tq_attn_values split MSE value contexts at
 * 96 < d <= 128; tq_attn_output and tq_search_topk return TQ_ERR_UNSUPPORTED for them.  */
int tq_init_split(tq_ctx** out, uint64_t seed, int d, int bits, int d_hi, int mode, int m,
                  const float* Pi_host, const float* S_host);

/* Words per code row (planes) of a context: MSE bits * W, plus ceil(d_hi / 32) for a split
 * context; and its d_hi (0 when not split).  Any output may be NULL.                      */
int tq_code_words(const tq_ctx* ctx, int* words, int* d_hi);

void tq_destroy(tq_ctx* ctx);   /* frees the context's tables; NULL is a no-op */

/* Fault injection for tests: after n more successful table allocations of tq_init* (process-
 * wide), the next one fails as if the device were out of memory — the init call returns
 * TQ_ERR_OOM, frees what it had allocated and leaves *out NULL — and the hook disarms.  n = -1
 * disarms it.  Off by default.                                                             */
int tq_debug_fail_alloc_after(int n);

/* d, m (0 in MSE mode), MSE bits and mode of a context.  Any output may be NULL.       */
int tq_info(const tq_ctx* ctx, int* d, int* m, int* mse_bits, int* mode);

/* Packed sizes per vector in 32-bit words: planes = MSE bits, words_per_plane = W,
 * sign_words = Ws (0 in MSE mode).  Any output may be NULL.                            */
int tq_layout(const tq_ctx* ctx, int* planes, int* words_per_plane, int* sign_words);

/* Kernel family on this context.  TQ_PATH_AUTO (the default) picks the fastest measured
 * family: tcgen05 tensor cores for bulk tq_quantize of bf16 rows at d = 128 (n >= 4096,
 * ld_x a multiple of 8, 16-byte aligned x; Pi, S Pi^T and r' as two bf16 pieces each, fp32
 * accumulation: codes and signs agree with exact arithmetic except within ~1e-5 of |x| of a
 * decision boundary), tcgen05 for tq_search_topk at d in (96,128] or
 * (192,256] with 1-3 MSE bits, the tcgen05 logits kernel (below) for tq_attn_logits on
 * keys of 2 MSE bits + QJL when batch x KV heads x head quads x cap >= 2^18, and the table
 * kernels for the other logits.  TQ_PATH_CUDA_CORE forces CUDA-core kernels everywhere;
 * TQ_PATH_TENSOR takes the tcgen05 kernels wherever they apply: tq_attn_logits (kind::f8f6f4,
 * key bits as e4m3 in tensor memory, fp32 accumulation; 96 < d <= 128, m <= 128, 1-3 MSE
 * bits, a cache capacity that is a multiple of 8 and 16-byte aligned code arrays, else the
 * table kernels) and the value sum of tq_attn_values / tq_attn_values_partial (coded values
 * of 1-3 MSE bits at 96 < d <= 128, even capacity, 4-byte aligned norms; the softmax weights
 * as e4m3 pieces, the value bits transposed per 32-key block).  Their waits are bounded: one
 * that runs out sets TQ_DEVERR_TIMEOUT.  All families compute the same estimator within the
 * documented tolerance.                                                                  */
enum tq_kernel_path { TQ_PATH_AUTO = 0, TQ_PATH_CUDA_CORE = 1, TQ_PATH_TENSOR = 2 };
int tq_set_kernel_path(tq_ctx* ctx, int path);

/* Copies the context's float32 Pi (d*d), S (m*d; PROD only) and float64 centroids
 * (2^P) and thresholds (2^P - 1) to host arrays.  Any output may be NULL.              */
int tq_export_matrices(const tq_ctx* ctx, float* Pi, float* S, double* centroids,
                       double* thresholds);

/* ---------------------------------------------------------------- quantization */

/* Quantize n rows of x (dtype TQ_F32 or TQ_BF16; row i at x + i*ld_x elements,
 * ld_x >= d) into row i of planes/signs/norm/rnorm (layout above).  signs and rnorm must
 * be NULL in MSE mode and non-NULL in PROD mode.  n may be 0.  Pages: csdn tutorial,
 * sections PolarQuant, 将笛卡尔积坐标转为极坐标 and QJL steps 1-2; juejin post §二.   */
int tq_quantize(tq_ctx* ctx, const void* x, int dtype, int64_t n, int64_t ld_x,
                uint32_t* planes, uint32_t* signs, uint16_t* norm, uint16_t* rnorm,
                void* stream);

/* Decode-step append: x is [B][H][d] contiguous (one new vector per (batch, KV head));
 * vector (b, h) is quantized into cache row (b*H + h)*cap + len[b].  len is a device
 * int32 [B], read only; a len[b] outside [0, cap) skips that batch's rows and sets
 * TQ_DEVERR_LEN_RANGE.  Pages: csdn tutorial, 背景 (every new token's vector enters the
 * KV cache); juejin post §四 (online quantization, no re-fit).                          */
int tq_append(tq_ctx* ctx, const void* x, int dtype, int B, int H, int64_t cap,
              const int32_t* len, uint32_t* planes, uint32_t* signs, uint16_t* norm,
              uint16_t* rnorm, void* stream);

/* len[b] += step for b < B on the device (clamped to [0, cap], TQ_DEVERR_LEN_RANGE when
 * clamped), so a captured decode step can advance the cache without a host round trip. */
int tq_advance_len(tq_ctx* ctx, int32_t* len, int B, int64_t cap, int step, void* stream);

/* Query preparation: qrot = Pi q ([nq][d]) and, in PROD mode, qproj = S q ([nq][m]) for
 * nq float32 rows q ([nq][d], contiguous).  qproj may be NULL in MSE mode.  Pages:
 * juejin post §二 (the query stays in high precision).                                  */
int tq_prep_queries(tq_ctx* ctx, const float* q, int64_t nq, float* qrot, float* qproj,
                    void* stream);

/* ---------------------------------------------------------------- attention */

/* Workspace bytes for tq_attn_logits / tq_attn_output with these shapes (the same size
 * serves both calls).                                                                  */
int tq_attn_workspace_size(const tq_ctx* kctx, int B, int Hq, int Hkv, int64_t cap,
                           size_t* bytes);

/* Attention logits over compressed keys: logits[b][h][i] = scale * est(q[b][h], key(b,
 * h / (Hq/Hkv), i)) for i < len[b]; entries i >= len[b] are not written.  q float32
 * [B][Hq][d]; keys in a [B][Hkv][cap] cache (k_signs, k_rnorm NULL for an MSE-mode kctx);
 * len device int32 [B]; logits float32 [B][Hq][cap].  Hq must be a multiple of Hkv.
 * Pages: juejin post §三 (attention logits from the compressed KV cache, the operation the
 * blog times on H100); csdn tutorial, QJL step 3 (estimator).                           */
int tq_attn_logits(tq_ctx* kctx, const float* q, int B, int Hq, int Hkv,
                   const uint32_t* k_planes, const uint32_t* k_signs, const uint16_t* k_norm,
                   const uint16_t* k_rnorm, int64_t cap, const int32_t* len, float scale,
                   float* logits, void* workspace, size_t ws_bytes, void* stream);

/* Attention output: out[b][h] = sum_{i < len[b]} softmax_i(logits) v_hat(b, h/(Hq/Hkv), i),
 * the logits as in tq_attn_logits.  vctx NULL: values are bfloat16 [B][Hkv][cap][d] in
 * `values` and v_norm is ignored.  vctx an MSE-mode context of the same d: `values` holds
 * its planes [B][Hkv][cap][P][W] and v_norm its norms, and v_hat = n16 Pi_v^T c_v[idx].
 * out float32 [B][Hq][d]; a batch with len[b] == 0 gets zeros.  Pages: nonndazone.ru
 * essay §2 (keys and values are both cached and compressed); juejin post §三.          */
int tq_attn_output(tq_ctx* kctx, const tq_ctx* vctx, const float* q, int B, int Hq,
                   int Hkv, const uint32_t* k_planes, const uint32_t* k_signs,
                   const uint16_t* k_norm, const uint16_t* k_rnorm, int64_t cap,
                   const int32_t* len, float scale, const void* values,
                   const uint16_t* v_norm, float* out, void* workspace, size_t ws_bytes,
                   void* stream);

/* Workspace bytes for tq_attn_values with these shapes.                               */
int tq_attn_values_workspace_size(int d, int B, int Hq, int Hkv, int64_t cap, size_t* bytes);

/* Softmax + value sum from logits already computed (e.g. by tq_attn_logits):
 * out[b][h] = sum_{i < len[b]} softmax_i(logits[b][h][0..len[b])) v_hat(b, h/(Hq/Hkv), i).
 * logits float32 [B][Hq][cap] (already scaled); values and v_norm as in tq_attn_output
 * (vctx NULL: bfloat16 values of dimension d; else vctx's MSE codes and d == vctx's d).
 * d <= 512.  With vctx NULL there is no device error word: a len[b] outside [0, cap] is
 * clamped without a flag.  Pages: nonndazone.ru essay §2 (compressed values); the softmax-weighted sum
 * of the values is the attention step that follows the logits of juejin.cn post §三.    */
int tq_attn_values(const tq_ctx* vctx, int d, const float* logits, int B, int Hq, int Hkv,
                   int64_t cap, const int32_t* len, const void* values, const uint16_t* v_norm,
                   float* out, void* workspace, size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- sharded attention and search
 * A sequence (or a database) cut into R contiguous blocks held by R processes, one GPU each.  The
 * pages time both operations on one GPU (juejin.cn post, section 三); the reading for R blocks is
 * the exact split of the softmax: each block contributes its partial state, and the states are
 * merged by their maxima (log-sum-exp).  The exchange between processes (an all-gather of the
 * partial states, or of the per-block top-k lists) is the caller's: these calls compute on one
 * device and take device buffers.                                                            */

/* As tq_attn_values over this call's block of the sequence (len[b] = the number of positions the
 * block holds for batch b), but instead of the output it writes one partial state per (batch,
 * query head): part float32 [B][Hq][d + 2] = (m, l, a[0..d)) with m the largest logit, l = sum_i
 * exp(logit_i - m) and a = sum_i exp(logit_i - m) v_i; for coded values a is in the value
 * context's rotated basis (v_i = n16 c_v[idx_i], before Pi_v^T).  A sequence with no positions in
 * the block gets m = -inf, l = 0, a = 0.  Workspace: tq_attn_values_workspace_size.          */
int tq_attn_values_partial(const tq_ctx* vctx, int d, const float* logits, int B, int Hq, int Hkv,
                           int64_t cap, const int32_t* len, const void* values, const uint16_t* v_norm,
                           float* part, void* workspace, size_t ws_bytes, void* stream);

/* out[b][h] (float32 [B][Hq][d]) from the partial states of R blocks, parts float32
 * [R][B][Hq][d + 2] as tq_attn_values_partial writes them:  with M = max_r m_r,
 *   out = Pi_v^T (sum_r exp(m_r - M) a_r) / sum_r exp(m_r - M) l_r
 * (no rotation for bf16 values: vctx NULL); zeros where every block is empty.                */
int tq_attn_merge_partials(const tq_ctx* vctx, int d, const float* parts, int R, int B, int Hq,
                           float* out, void* stream);

/* Global top-k from R blocks' lists: cand_s float32 [R][nq][k] and cand_i int32 [R][nq][k] (row
 * numbers within block r, as tq_search_topk returns them; an entry whose index is INT32_MAX is
 * padding, for a block with fewer than k rows); row_offsets host int64 [R] (block r's first global
 * row, each in [0, 2^31)).  top_s / top_i [nq][k]: the k best of all blocks' candidates by score
 * descending, equal scores by global row ascending.  1 <= R <= 64, 1 <= k <= TQ_MAX_TOPK.     */
int tq_topk_merge(const float* cand_s, const int32_t* cand_i, int R, int64_t nq, int k,
                  const int64_t* row_offsets, float* top_s, int32_t* top_i, void* stream);

/* Size of the static scratch array behind tq_attn_values_noalloc (8 MiB per device).     */
#define TQ_NOALLOC_SCRATCH_BYTES (8u << 20)

/* tq_attn_values without a workspace argument, for callers that may not allocate device
 * memory while they run (a server that reserves all device memory in its own pool at
 * start-up and forbids cudaMalloc afterwards, since an allocation can synchronise the device
 * and can fail mid-request; a plugin host that passes buffers but no allocator).  The pages
 * have no counterpart: this is an interface variant, the arithmetic is tq_attn_values'.
 * Scratch: a file-scope device array of TQ_NOALLOC_SCRATCH_BYTES that every GPU loading the
 * library keeps until exit.  Shapes needing more than that (B*Hq*nchunk*(d+2)*4 bytes, as
 * tq_attn_values_workspace_size reports) are rejected with TQ_ERR_UNSUPPORTED, and so are
 * split (fractional bit width) value contexts, which tq_attn_values takes.  The first call on a
 * device looks up the array's device address (cudaGetSymbolAddress) with that device current
 * and keeps it for the life of the process; make that first call before any stream capture.
 * A cudaDeviceReset (or any teardown of the device's primary context) invalidates the kept
 * address: do not call this entry point on that device afterwards.  No call allocates or frees
 * memory.  All calls on a device share the array: calls that overlap on the GPU race.       */
int tq_attn_values_noalloc(const tq_ctx* vctx, int d, const float* logits, int B, int Hq, int Hkv,
                           int64_t cap, const int32_t* len, const void* values, const uint16_t* v_norm,
                           float* out, void* stream);

/* ---------------------------------------------------------------- search */

/* Workspace bytes for tq_search_topk.                                                  */
int tq_search_workspace_size(const tq_ctx* ctx, int64_t nq, int64_t n, int k, size_t* bytes);

/* Top-k search: for each of nq float32 queries ([nq][d]) the k database rows (coded by
 * ctx, rows 0..n-1) with the largest est(q, x), ordered by score descending and equal
 * scores by row ascending.  top_score float32 [nq][k], top_idx int32 [nq][k].
 * 1 <= k <= min(n, TQ_MAX_TOPK); n < 2^31.  Pages: juejin post §三 (GloVe Recall@1@k
 * against PQ and RabitQ) and §四 (near-zero indexing time).                            */
int tq_search_topk(tq_ctx* ctx, const float* q, int64_t nq, const uint32_t* planes,
                   const uint32_t* signs, const uint16_t* norm, const uint16_t* rnorm,
                   int64_t n, int k, float* top_score, int32_t* top_idx, void* workspace,
                   size_t ws_bytes, void* stream);

/* ---------------------------------------------------------------- polar-angle encoder
 * The recursive polar representation of the pages: csdn tutorial, section 将笛卡尔积坐标转为
 * 极坐标 (the length r kept at FP16 and d - 1 low-bit angles for the direction) and section
 * TurboQuant原理剖析 (2 or 3 bits per angle, then 1 QJL bit per dimension); freelamp article,
 * section 技术突破：极坐标量化 (rotation first; a recursive polar transform into one radius and
 * a series of angles whose law is known in closed form).
 * Readings: y = Pi x is transformed by pairing neighbours: level 1 maps (y_2i, y_2i+1) to a
 * radius and an angle atan2(y_2i+1, y_2i) in [0, 2 pi); level l pairs the level-(l-1) radii into
 * an angle atan2(right, left) in [0, pi/2]; d/2 + d/4 + ... + 1 = d - 1 angles.  Level 1 angles
 * are uniform (table: cells of width 2 pi / 2^b, centroids at their centres); a level-l angle has
 * density proportional to (sin psi cos psi)^(2^(l-1) - 1) and its own Lloyd-Max table.  Every
 * angle takes b bits.  The QJL stage and the estimator are those of the PROD mode, on the
 * residual x - Pi^T y_hat, y_hat rebuilt from the fp16 radius and the angle centroids.
 * Code rows: the d - 1 codes (level 1 left to right, then level 2, ...) as consecutive b-bit
 * fields of one little-endian bit stream (code a in stream bits a*b .. a*b + b - 1; stream bit
 * t = bit t % 32 of word t / 32), tq_polar_layout words per vector.                        */
#define TQ_POLAR_MAX_BITS 4
typedef struct tq_polar tq_polar;

/* The level-`level` angle table (1 <= level <= 8, 1 <= bits <= 4): 2^bits centroids ascending
 * and 2^bits - 1 thresholds, float64, caller-owned arrays.  Host only.                     */
int tq_host_polar_codebook(int level, int bits, double* centroids, double* thresholds);

/* d in {16, 32, 64, 128, 256}; bits per angle 1..4; qjl 1 adds the QJL stage with m = d rows.
 * Pi_host (d x d) and S_host (d x d) float32 row-major as in tq_init_ex (NULL: seeded).     */
int tq_polar_init(tq_polar** out, uint64_t seed, int d, int bits, int qjl, const float* Pi_host,
                  const float* S_host);
void tq_polar_destroy(tq_polar* ctx);

/* Words per vector of the code rows and of the sign rows (0 without QJL).                  */
int tq_polar_layout(const tq_polar* ctx, int* code_words, int* sign_words);

/* Encodes n rows of x (device, TQ_F32 or TQ_BF16, row stride ld_x >= d elements) into codes
 * [n][code_words], r16 [n] (binary16 bits of |x|) and, with QJL, signs [n][sign_words] and
 * rnorm16 [n] (binary16 bits of |x - x_hat|).  Device buffers, caller-owned; asynchronous on
 * `stream`.  A radius rounding to binary16 infinity sets TQ_DEVERR_NORM_OVERFLOW.           */
int tq_polar_quantize(tq_polar* ctx, const void* x, int dtype, int64_t n, int64_t ld_x,
                      uint32_t* codes, uint16_t* r16, uint32_t* signs, uint16_t* rnorm16,
                      void* stream);

/* Kernel family of tq_polar_quantize (enum tq_kernel_path).  TQ_PATH_AUTO (the default)
 * encodes bf16 rows at d = 128 with n >= 4096 (ld_x a multiple of 8, x 16-byte aligned) on
 * the tcgen05 tensor cores (y = Pi x and the QJL projection (S Pi^T) r' as bf16 MMAs with the
 * matrices and r' split into two bf16 pieces each, fp32 accumulation, the product of the two
 * small pieces left out; r' = y - y_hat in the rotated basis)
 * and everything else on CUDA cores; TQ_PATH_TENSOR takes the tensor-core encoder for every n
 * where the dtype, d and alignment allow it; TQ_PATH_CUDA_CORE never.  Both families give the
 * same codes up to angles within float rounding of a threshold.  TQ_ERR_ARG for another path.  */
int tq_polar_set_kernel_path(tq_polar* ctx, int path);

/* out[i][k] = scale * est(q_i, x_k) for nq fp32 queries q [nq][d] against n coded rows
 * (device buffers, out [nq][n] fp32 row-major).  Asynchronous on `stream`.                 */
int tq_polar_scores(tq_polar* ctx, const float* q, int64_t nq, const uint32_t* codes,
                    const uint16_t* r16, const uint32_t* signs, const uint16_t* rnorm16,
                    int64_t n, float scale, float* out, void* stream);

/* As tq_sync_status, for the polar context's device error word.                            */
int tq_polar_sync_status(tq_polar* ctx, void* stream, int* flags);

/* ---------------------------------------------------------------- fused paged decode step
 * One decode step over a paged compressed KV cache in a single persistent (cooperative) launch.
 * Pages: juejin.cn post, section 三 (attention logits over the compressed KV cache); csdn
 * tutorial, section 背景 (every generated token joins the cache).  Readings: a page holds
 * page_size consecutive token slots of one sequence for every KV head; the pools are
 *   kplanes [num_pages][Hkv][page_size][P_k][4] u32, ksigns [..][4] u32, knorm, krnorm [..] fp16,
 *   vplanes [num_pages][Hkv][page_size][P_v][4] u32, vnorm [..] fp16
 * (rows in the layouts of tq_layout); block_table [B][max_pages] int32 gives the page of
 * sequence b's tokens i*page_size .. (i+1)*page_size - 1.  The step quantizes k_new and v_new
 * [B][Hkv][128] (TQ_F32 or TQ_BF16) into position len[b], then for every query head computes
 *   out[b][h] = sum_{i <= len[b]} softmax_i(scale * est(q[b][h], key_i)) * v_hat_i
 * (q [B][Hq][128] fp32, GQA groups of Hq / Hkv heads; out [B][Hq][128] fp32), and sets
 * len[b] += 1.  Keys: a PROD context with d = m = 128 and 1..3 MSE bits; values: an MSE context
 * with d = 128.  page_size is a positive multiple of 32; the page of position len[b] must be in
 * the table (an entry outside 0..num_pages-1 or len[b] >= max_pages * page_size sets
 * TQ_DEVERR_LEN_RANGE in kctx's error word and skips that append).  Device buffers are
 * caller-owned; planes, signs and the workspace 16-byte aligned; asynchronous on `stream`.
 * The launch's grid barriers are bounded: one that gives up sets TQ_DEVERR_TIMEOUT.        */
int tq_paged_workspace_size(int B, int Hq, int Hkv, int max_pages, int page_size, size_t* bytes);
int tq_paged_decode_step(tq_ctx* kctx, const tq_ctx* vctx, const float* q, const void* k_new,
                         const void* v_new, int dtype, int B, int Hq, int Hkv,
                         const int32_t* block_table, int max_pages, int page_size, int num_pages,
                         int32_t* len, uint32_t* kplanes, uint32_t* ksigns, uint16_t* knorm,
                         uint16_t* krnorm, uint32_t* vplanes, uint16_t* vnorm, float scale,
                         float* out, void* workspace, size_t workspace_bytes, void* stream);

/* Self-test of the bounded device waits (the grid barriers of tq_paged_decode_step use the same
 * code): launches one thread that arrives at a two-party counter nobody else joins, so its wait
 * gives up after its poll limit (about a second) and sets TQ_DEVERR_TIMEOUT in ctx's error word;
 * the kernel then returns and the context stays usable.  Synchronous on `stream`.  Returns
 * TQ_OK when the launch ran (read the flag with tq_sync_status).                           */
int tq_selftest_wait_timeout(tq_ctx* ctx, void* stream);

/* ---------------------------------------------------------------- status */

/* Synchronises `stream`, then reads and clears the context's device error word.  Returns
 * TQ_OK when it was 0, TQ_ERR_DEVICE (flags in *flags, which may be NULL) otherwise, or
 * TQ_ERR_CUDA when the synchronisation itself failed.                                   */
int tq_sync_status(tq_ctx* ctx, void* stream, int* flags);

/* Message for the last failing call on this thread ("" if none).  Valid until the next
 * call on this thread.                                                                  */
const char* tq_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* TQ_H */
