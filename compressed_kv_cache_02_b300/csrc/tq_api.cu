// The C-ABI of libtq (include/tq.h): argument checks, context set-up and the launches.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "tq_internal.h"
#include "tq_kernels.h"

namespace tq {

static thread_local std::string g_err;

int fail(int code, const std::string& msg) {
    g_err = msg;
    return code;
}

namespace {

int cuda_fail(cudaError_t e, const char* what) {
    return fail(TQ_ERR_CUDA, std::string(what) + ": " + cudaGetErrorName(e) + " (" + cudaGetErrorString(e) + ")");
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define TQ_REQUIRE(cond, code, msg) \
    do {                            \
        if (!(cond)) return fail(code, msg); \
    } while (0)

int check_ctx(const tq_ctx* c) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    TQ_REQUIRE(dev == c->device, TQ_ERR_ARG, "context was created on device " + std::to_string(c->device) +
                                                 " but device " + std::to_string(dev) + " is current");
    return TQ_OK;
}

// Fault injection for the allocation-failure tests: when >= 0, the table allocation after that
// many more successful ones fails as if the device were out of memory (then the hook disarms).
std::atomic<int> g_fail_alloc_after{-1};

template <typename T>
int upload(T** dst, const std::vector<T>& src) {
    int armed = g_fail_alloc_after.load();
    while (armed >= 0 && !g_fail_alloc_after.compare_exchange_weak(armed, armed - 1)) {
    }
    if (armed == 0) {
        *dst = nullptr;
        return fail(TQ_ERR_OOM, "cudaMalloc of context tables failed: simulated by tq_debug_fail_alloc_after");
    }
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(dst), src.size() * sizeof(T));
    if (e != cudaSuccess) {
        *dst = nullptr;
        cudaGetLastError();
        return fail(TQ_ERR_OOM, std::string("cudaMalloc of context tables failed: ") + cudaGetErrorString(e));
    }
    e = cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy of context tables");
    return TQ_OK;
}

void free_ctx(tq_ctx* c) {
    if (!c) return;
    cudaFree(c->dPiT);
    cudaFree(c->dPi);
    cudaFree(c->dST);
    cudaFree(c->dStT);
    cudaFree(c->derr);
    cudaFree(c->bops);
    cudaFree(c->dtab);
    delete c;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

const char* tq_last_error(void) { return g_err.c_str(); }

int tq_host_codebook(int d, int mse_bits, double* centroids, double* thresholds) {
    TQ_REQUIRE(d >= 3 && d <= TQ_MAX_D, TQ_ERR_ARG, "d must be in [3, 1024]");
    TQ_REQUIRE(mse_bits >= 1 && mse_bits <= TQ_MAX_MSE_BITS, TQ_ERR_ARG, "mse_bits must be in [1, 8]");
    std::vector<double> c, t;
    lloyd_max_codebook(d, mse_bits, c, t);
    if (centroids) std::memcpy(centroids, c.data(), c.size() * sizeof(double));
    if (thresholds) std::memcpy(thresholds, t.data(), t.size() * sizeof(double));
    return TQ_OK;
}

int tq_host_matrices(uint64_t seed, int d, int m, float* Pi, float* S) {
    TQ_REQUIRE(d >= 3 && d <= TQ_MAX_D, TQ_ERR_ARG, "d must be in [3, 1024]");
    TQ_REQUIRE(m >= 1 && m <= TQ_MAX_D, TQ_ERR_ARG, "m must be in [1, 1024]");
    std::vector<double> P, Sd;
    seeded_matrices(seed, d, m, P, Sd);
    if (Pi) for (size_t i = 0; i < P.size(); ++i) Pi[i] = static_cast<float>(P[i]);
    if (S) for (size_t i = 0; i < Sd.size(); ++i) S[i] = static_cast<float>(Sd[i]);
    return TQ_OK;
}

static int init_ctx(tq_ctx** out, uint64_t seed, int d, int bits, int d_hi, int mode, int m, const float* Pi_host,
                    const float* S_host) {
    TQ_REQUIRE(out != nullptr, TQ_ERR_ARG, "out is NULL");
    *out = nullptr;
    TQ_REQUIRE(d >= 3 && d <= TQ_MAX_D, TQ_ERR_ARG, "d must be in [3, 1024]");
    TQ_REQUIRE(mode == TQ_MODE_PROD || mode == TQ_MODE_MSE, TQ_ERR_ARG, "mode must be TQ_MODE_PROD or TQ_MODE_MSE");
    const int P = (mode == TQ_MODE_PROD) ? bits - 1 : bits;
    if (mode == TQ_MODE_PROD)
        TQ_REQUIRE(P >= 1 && P <= kFastBits, TQ_ERR_ARG, "PROD mode needs bits in [2, 5]");
    else
        TQ_REQUIRE(P >= 1 && P <= TQ_MAX_MSE_BITS, TQ_ERR_ARG, "MSE mode needs bits in [1, 8]");
    TQ_REQUIRE(d_hi >= 0 && d_hi <= d && d_hi % 32 == 0, TQ_ERR_ARG, "d_hi must be a multiple of 32 in [0, d]");
    if (d_hi) TQ_REQUIRE(P + 1 <= kFastBits, TQ_ERR_ARG, "the split table needs MSE bits + 1 <= 4");
    if (mode == TQ_MODE_PROD) TQ_REQUIRE(m >= 1 && m <= TQ_MAX_D, TQ_ERR_ARG, "m must be in [1, 1024]");
    else m = 0;

    tq_ctx* c = new (std::nothrow) tq_ctx();
    TQ_REQUIRE(c != nullptr, TQ_ERR_OOM, "host allocation failed");
    cudaError_t e = cudaGetDevice(&c->device);
    if (e != cudaSuccess) { delete c; return cuda_fail(e, "cudaGetDevice"); }
    c->d = d; c->m = m; c->bits = bits; c->mode = mode; c->P = P; c->L = 1 << P;
    c->W = (d + 31) / 32;
    c->Ws = m ? (m + 31) / 32 : 0;

    // Matrices as data, or generated from the seed (float64, then rounded to float32).
    std::vector<double> Pd, Sd;
    if (!Pi_host || (m && !S_host)) seeded_matrices(seed, d, m ? m : 1, Pd, Sd);
    c->Pi.resize((size_t)d * d);
    for (size_t i = 0; i < c->Pi.size(); ++i) c->Pi[i] = Pi_host ? Pi_host[i] : static_cast<float>(Pd[i]);
    if (m) {
        c->S.resize((size_t)m * d);
        for (size_t i = 0; i < c->S.size(); ++i) c->S[i] = S_host ? S_host[i] : static_cast<float>(Sd[i]);
    }
    for (float v : c->Pi) if (!std::isfinite(v)) { delete c; return fail(TQ_ERR_ARG, "Pi has a non-finite entry"); }
    for (float v : c->S) if (!std::isfinite(v)) { delete c; return fail(TQ_ERR_ARG, "S has a non-finite entry"); }

    lloyd_max_codebook(d, P, c->centroids, c->thresholds);
    c->d_hi = d_hi;
    if (d_hi) lloyd_max_codebook(d, P + 1, c->centroids_hi, c->thresholds_hi);

    Params& p = c->prm;
    p.d = d; p.m = m; p.P = P; p.L = c->L; p.W = c->W; p.Ws = c->Ws;
    p.d_hi = d_hi;
    p.W_hi = (d_hi + 31) / 32;
    p.row_words = P * c->W + p.W_hi;
    for (int k = 0; k < kMaxLevels; ++k) {
        const int Lh = 2 * c->L;
        p.centroids_hi[k] = (d_hi && k < Lh) ? static_cast<float>(c->centroids_hi[k]) : 0.f;
        p.thresholds_hi[k] = (d_hi && k < Lh - 1) ? static_cast<float>(c->thresholds_hi[k]) : INFINITY;
    }
    p.qjl = m ? 1 : 0;
    p.qjl_scale = m ? static_cast<float>(std::sqrt(M_PI / 2.0) / m) : 0.f;
    for (int k = 0; k < kMaxLevels; ++k) {
        p.centroids[k] = k < c->L ? static_cast<float>(c->centroids[k]) : 0.f;
        p.thresholds[k] = k < c->L - 1 ? static_cast<float>(c->thresholds[k]) : INFINITY;
    }
    double c0 = c->centroids[0];
    std::vector<int> masks;
    std::vector<double> kappa;
    if (P <= kFastBits) walsh_form(c->centroids, P, c0, masks, kappa);
    p.c0 = static_cast<float>(c0);
    p.nterms = static_cast<int>(masks.size());
    {
        std::vector<int> odd;
        for (int S = 1; S < c->L; ++S)
            if (__builtin_popcount(S) & 1) odd.push_back(S);
        p.odd_walsh = (masks == odd) ? 1 : 0;
    }
    for (int t = 0; t < kMaxTerms; ++t) {
        p.mask[t] = t < p.nterms ? masks[t] : 0;
        p.kappa[t] = t < p.nterms ? static_cast<float>(kappa[t]) : 0.f;
    }

    if (d_hi) {
        double c0h;
        std::vector<int> mh;
        std::vector<double> kh;
        walsh_form(c->centroids_hi, P + 1, c0h, mh, kh);
        std::vector<int> odd;
        for (int S = 1; S < 2 * c->L; ++S)
            if (__builtin_popcount(S) & 1) odd.push_back(S);
        p.c0_hi = static_cast<float>(c0h);
        p.split_walsh = (mh == odd && p.odd_walsh) ? 1 : 0;
        for (int t = 0; t < kMaxTerms; ++t) {
            p.kappa_hi[t] = t < (int)kh.size() ? static_cast<float>(kh[t]) : 0.f;
            p.kappa_lo_x[t] = 0.f;
            if (t < (int)odd.size() && !(odd[t] >> P & 1))
                for (int u = 0; u < p.nterms; ++u)
                    if (masks[u] == odd[t]) p.kappa_lo_x[t] = static_cast<float>(kappa[u]);
        }
    }

    // Device tables: Pi^T and Pi for the rotations, S^T for queries, (S Pi^T)^T for residuals.
    std::vector<float> PiT((size_t)d * d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) PiT[(size_t)j * d + i] = c->Pi[(size_t)i * d + j];
    int rc;
    if ((rc = upload(&c->dPiT, PiT)) != TQ_OK || (rc = upload(&c->dPi, c->Pi)) != TQ_OK) { free_ctx(c); return rc; }
    if (m) {
        std::vector<float> ST((size_t)d * m), StT((size_t)d * m);
        for (int i = 0; i < m; ++i)
            for (int j = 0; j < d; ++j) ST[(size_t)j * m + i] = c->S[(size_t)i * d + j];
        // (S Pi^T)[i][j] = sum_k S[i][k] Pi[j][k], in float64 from the float32 matrices.
        for (int i = 0; i < m; ++i)
            for (int j = 0; j < d; ++j) {
                double s = 0.0;
                for (int k = 0; k < d; ++k) s += (double)c->S[(size_t)i * d + k] * (double)c->Pi[(size_t)j * d + k];
                StT[(size_t)j * m + i] = static_cast<float>(s);
            }
        if ((rc = upload(&c->dST, ST)) != TQ_OK || (rc = upload(&c->dStT, StT)) != TQ_OK) { free_ctx(c); return rc; }
    }
    if (d == 128 && (m == 0 || m == 128)) {   // tcgen05 operands for bulk quantization
        std::vector<float> St;
        if (m) {
            St.resize((size_t)128 * 128);
            for (int i = 0; i < 128; ++i)
                for (int j = 0; j < 128; ++j) {
                    double acc = 0.0;
                    for (int k = 0; k < 128; ++k) acc += (double)c->S[(size_t)i * 128 + k] * (double)c->Pi[(size_t)j * 128 + k];
                    St[(size_t)i * 128 + j] = static_cast<float>(acc);
                }
        }
        std::vector<uint16_t> ops;
        build_tc_operands(c->Pi.data(), m ? St.data() : nullptr, ops);
        if ((rc = upload(&c->bops, ops)) != TQ_OK) { free_ctx(c); return rc; }
    }
    std::vector<float> tab(2 * c->L - 1);
    for (int k = 0; k < c->L; ++k) tab[k] = static_cast<float>(c->centroids[k]);
    for (int k = 0; k + 1 < c->L; ++k) tab[c->L + k] = static_cast<float>(c->thresholds[k]);
    if ((rc = upload(&c->dtab, tab)) != TQ_OK) { free_ctx(c); return rc; }
    p.tab = c->dtab;
    std::vector<int> zero(1, 0);
    if ((rc = upload(&c->derr, zero)) != TQ_OK) { free_ctx(c); return rc; }
    *out = c;
    return TQ_OK;
}

int tq_init_ex(tq_ctx** out, uint64_t seed, int d, int bits, int mode, int m, const float* Pi_host,
               const float* S_host) {
    return init_ctx(out, seed, d, bits, 0, mode, m, Pi_host, S_host);
}

int tq_init_split(tq_ctx** out, uint64_t seed, int d, int bits, int d_hi, int mode, int m, const float* Pi_host,
                  const float* S_host) {
    return init_ctx(out, seed, d, bits, d_hi, mode, m, Pi_host, S_host);
}

int tq_code_words(const tq_ctx* c, int* words, int* d_hi) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    if (words) *words = c->prm.row_words;
    if (d_hi) *d_hi = c->d_hi;
    return TQ_OK;
}

int tq_init(tq_ctx** out, uint64_t seed, int d, int bits) {
    return tq_init_ex(out, seed, d, bits, TQ_MODE_PROD, d, nullptr, nullptr);
}

void tq_destroy(tq_ctx* ctx) { free_ctx(ctx); }

int tq_debug_fail_alloc_after(int n) {
    if (n < -1) return fail(TQ_ERR_ARG, "tq_debug_fail_alloc_after: n >= -1");
    g_fail_alloc_after.store(n);
    return TQ_OK;
}

int tq_info(const tq_ctx* c, int* d, int* m, int* mse_bits, int* mode) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    if (d) *d = c->d;
    if (m) *m = c->m;
    if (mse_bits) *mse_bits = c->P;
    if (mode) *mode = c->mode;
    return TQ_OK;
}

int tq_layout(const tq_ctx* c, int* planes, int* words_per_plane, int* sign_words) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    if (planes) *planes = c->P;
    if (words_per_plane) *words_per_plane = c->W;
    if (sign_words) *sign_words = c->Ws;
    return TQ_OK;
}

int tq_set_kernel_path(tq_ctx* c, int path) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    TQ_REQUIRE(path == TQ_PATH_AUTO || path == TQ_PATH_CUDA_CORE || path == TQ_PATH_TENSOR, TQ_ERR_ARG,
               "path must be TQ_PATH_AUTO, TQ_PATH_CUDA_CORE or TQ_PATH_TENSOR");
    c->kernel_path = path;
    return TQ_OK;
}

int tq_export_matrices(const tq_ctx* c, float* Pi, float* S, double* centroids, double* thresholds) {
    TQ_REQUIRE(c != nullptr, TQ_ERR_ARG, "context is NULL");
    if (Pi) std::memcpy(Pi, c->Pi.data(), c->Pi.size() * sizeof(float));
    if (S && c->m) std::memcpy(S, c->S.data(), c->S.size() * sizeof(float));
    if (centroids) std::memcpy(centroids, c->centroids.data(), c->centroids.size() * sizeof(double));
    if (thresholds) std::memcpy(thresholds, c->thresholds.data(), c->thresholds.size() * sizeof(double));
    return TQ_OK;
}

static int check_codes_out(const tq_ctx* c, uint32_t* planes, uint32_t* signs, uint16_t* norm, uint16_t* rnorm) {
    TQ_REQUIRE(planes && norm, TQ_ERR_ARG, "planes and norm must be non-NULL");
    TQ_REQUIRE(aligned(planes, 4) && aligned(norm, 2), TQ_ERR_ARG, "planes must be 4-byte and norm 2-byte aligned");
    if (c->m) {
        TQ_REQUIRE(signs && rnorm, TQ_ERR_ARG, "PROD mode needs signs and rnorm");
        TQ_REQUIRE(aligned(signs, 4) && aligned(rnorm, 2), TQ_ERR_ARG, "signs must be 4-byte and rnorm 2-byte aligned");
    } else {
        TQ_REQUIRE(!signs && !rnorm, TQ_ERR_ARG, "MSE mode takes no signs or rnorm");
    }
    return TQ_OK;
}

int tq_quantize(tq_ctx* c, const void* x, int dtype, int64_t n, int64_t ld_x, uint32_t* planes, uint32_t* signs,
                uint16_t* norm, uint16_t* rnorm, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(n >= 0, TQ_ERR_ARG, "n must be >= 0");
    if (n == 0) return TQ_OK;
    TQ_REQUIRE(dtype == TQ_F32 || dtype == TQ_BF16, TQ_ERR_ARG, "dtype must be TQ_F32 or TQ_BF16");
    TQ_REQUIRE(x != nullptr, TQ_ERR_ARG, "x is NULL");
    TQ_REQUIRE(aligned(x, dtype == TQ_F32 ? 4 : 2), TQ_ERR_ARG, "x is misaligned for its dtype");
    TQ_REQUIRE(ld_x >= c->d, TQ_ERR_ARG, "ld_x must be >= d");
    if ((rc = check_codes_out(c, planes, signs, norm, rnorm))) return rc;
    cudaError_t e = quantize_tc_supported(c, dtype, x, n, ld_x)
                        ? launch_quantize_tc(c, x, n, ld_x, planes, signs, norm, rnorm, static_cast<cudaStream_t>(stream))
                        : launch_quantize(c, x, dtype, n, ld_x, 1, 0, nullptr, planes, signs, norm, rnorm,
                                          static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_quantize launch");
}

int tq_append(tq_ctx* c, const void* x, int dtype, int B, int H, int64_t cap, const int32_t* len, uint32_t* planes,
              uint32_t* signs, uint16_t* norm, uint16_t* rnorm, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(B >= 0 && H >= 1 && cap >= 1, TQ_ERR_ARG, "need B >= 0, H >= 1, cap >= 1");
    if (B == 0) return TQ_OK;
    TQ_REQUIRE(dtype == TQ_F32 || dtype == TQ_BF16, TQ_ERR_ARG, "dtype must be TQ_F32 or TQ_BF16");
    TQ_REQUIRE(x && len, TQ_ERR_ARG, "x and len must be non-NULL");
    TQ_REQUIRE(aligned(x, dtype == TQ_F32 ? 4 : 2) && aligned(len, 4), TQ_ERR_ARG, "x or len misaligned");
    if ((rc = check_codes_out(c, planes, signs, norm, rnorm))) return rc;
    cudaError_t e = launch_quantize(c, x, dtype, (int64_t)B * H, c->d, H, cap, len, planes, signs, norm, rnorm,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_append launch");
}

int tq_advance_len(tq_ctx* c, int32_t* len, int B, int64_t cap, int step, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(len && aligned(len, 4), TQ_ERR_ARG, "len must be non-NULL and 4-byte aligned");
    TQ_REQUIRE(B >= 0 && cap >= 1, TQ_ERR_ARG, "need B >= 0, cap >= 1");
    cudaError_t e = launch_advance_len(len, B, cap, step, c->derr, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_advance_len launch");
}

int tq_prep_queries(tq_ctx* c, const float* q, int64_t nq, float* qrot, float* qproj, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(nq >= 0, TQ_ERR_ARG, "nq must be >= 0");
    if (nq == 0) return TQ_OK;
    TQ_REQUIRE(q && qrot && aligned(q, 4) && aligned(qrot, 4), TQ_ERR_ARG, "q and qrot must be non-NULL, 4-byte aligned");
    if (c->m) TQ_REQUIRE(qproj && aligned(qproj, 4), TQ_ERR_ARG, "PROD mode needs qproj");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_apply_rows(c->dPiT, c->d, c->d, q, c->d, nq, qrot, c->d, s);
    if (e == cudaSuccess && c->m) e = launch_apply_rows(c->dST, c->d, c->m, q, c->d, nq, qproj, c->m, s);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_prep_queries launch");
}

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

struct AttnWs {
    size_t qrot, qproj, partials, image, total;
};

static AttnWs attn_ws_layout(const tq_ctx* c, int B, int Hq, int Hkv, int64_t cap) {
    int chunk, nchunk;
    attn_chunking(c, B, Hq, Hkv, cap, &chunk, &nchunk);
    AttnWs w;
    w.qrot = 0;
    w.qproj = round_up((size_t)B * Hq * c->d * sizeof(float), 256);
    w.partials = w.qproj + round_up((size_t)B * Hq * c->m * sizeof(float), 256);
    w.image = w.partials + round_up((size_t)B * Hq * nchunk * (c->d + 2) * sizeof(float), 256);
    w.total = w.image + (logits_tc_supported(c) ? round_up(logits_tc_image_bytes(B, Hq, Hkv), 256) : 0);
    return w;
}

int tq_attn_workspace_size(const tq_ctx* c, int B, int Hq, int Hkv, int64_t cap, size_t* bytes) {
    TQ_REQUIRE(c && bytes, TQ_ERR_ARG, "context and bytes must be non-NULL");
    TQ_REQUIRE(B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && cap >= 1, TQ_ERR_ARG,
               "need B >= 1, cap >= 1 and Hq a positive multiple of Hkv");
    *bytes = attn_ws_layout(c, B, Hq, Hkv, cap).total;
    return TQ_OK;
}

static int check_attn(const tq_ctx* c, const float* q, int B, int Hq, int Hkv, const uint32_t* kp, const uint32_t* ks,
                      const uint16_t* kn, const uint16_t* kr, int64_t cap, const int32_t* len, void* ws, size_t ws_bytes) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0, TQ_ERR_ARG, "need B >= 1 and Hq a positive multiple of Hkv");
    TQ_REQUIRE(cap >= 1 && cap < (int64_t)1 << 31, TQ_ERR_ARG, "cap must be in [1, 2^31)");
    TQ_REQUIRE(q && kp && kn && len && ws, TQ_ERR_ARG, "q, keys, len and workspace must be non-NULL");
    TQ_REQUIRE(aligned(q, 16) && aligned(kp, 16) && aligned(kn, 2) && aligned(len, 4) && aligned(ws, 256), TQ_ERR_ARG,
               "q and planes must be 16-byte, workspace 256-byte aligned");
    if (c->m) TQ_REQUIRE(ks && kr && aligned(ks, 16) && aligned(kr, 2), TQ_ERR_ARG, "PROD keys need signs and rnorm");
    TQ_REQUIRE(ws_bytes >= attn_ws_layout(c, B, Hq, Hkv, cap).total, TQ_ERR_ARG,
               "workspace too small (see tq_attn_workspace_size)");
    return TQ_OK;
}

int tq_attn_logits(tq_ctx* c, const float* q, int B, int Hq, int Hkv, const uint32_t* kp, const uint32_t* ks,
                   const uint16_t* kn, const uint16_t* kr, int64_t cap, const int32_t* len, float scale, float* logits,
                   void* ws, size_t ws_bytes, void* stream) {
    int rc = check_attn(c, q, B, Hq, Hkv, kp, ks, kn, kr, cap, len, ws, ws_bytes);
    if (rc) return rc;
    TQ_REQUIRE(logits && aligned(logits, 4), TQ_ERR_ARG, "logits must be non-NULL");
    AttnWs w = attn_ws_layout(c, B, Hq, Hkv, cap);
    char* base = static_cast<char*>(ws);
    float* qrot = reinterpret_cast<float*>(base + w.qrot);
    float* qproj = c->m ? reinterpret_cast<float*>(base + w.qproj) : nullptr;
    if ((rc = tq_prep_queries(c, q, (int64_t)B * Hq, qrot, qproj, stream))) return rc;
    KeyCache k{kp, ks, kn, kr, cap, len};
    cudaError_t e = c->d_hi ? launch_logits_split(c, qrot, qproj, B, Hq, Hkv, k, scale, logits,
                                                  static_cast<cudaStream_t>(stream))
                            : launch_logits(c, qrot, qproj, B, Hq, Hkv, k, scale, logits, base + w.image,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_attn_logits launch");
}

int tq_attn_output(tq_ctx* c, const tq_ctx* vc, const float* q, int B, int Hq, int Hkv, const uint32_t* kp,
                   const uint32_t* ks, const uint16_t* kn, const uint16_t* kr, int64_t cap, const int32_t* len,
                   float scale, const void* values, const uint16_t* v_norm, float* out, void* ws, size_t ws_bytes,
                   void* stream) {
    int rc = check_attn(c, q, B, Hq, Hkv, kp, ks, kn, kr, cap, len, ws, ws_bytes);
    if (rc) return rc;
    TQ_REQUIRE(c->d <= 512, TQ_ERR_UNSUPPORTED, "tq_attn_output supports d <= 512");
    TQ_REQUIRE(c->d_hi == 0 && (!vc || vc->d_hi == 0), TQ_ERR_UNSUPPORTED,
               "tq_attn_output does not take split (fractional bit width) contexts");
    TQ_REQUIRE(values && out && aligned(values, 16) && aligned(out, 4), TQ_ERR_ARG, "values and out must be non-NULL");
    if (vc) {
        if ((rc = check_ctx(vc))) return rc;
        TQ_REQUIRE(vc->mode == TQ_MODE_MSE && vc->d == c->d, TQ_ERR_ARG, "vctx must be an MSE-mode context of the same d");
        TQ_REQUIRE(v_norm && aligned(v_norm, 2), TQ_ERR_ARG, "coded values need v_norm");
    }
    AttnWs w = attn_ws_layout(c, B, Hq, Hkv, cap);
    char* base = static_cast<char*>(ws);
    float* qrot = reinterpret_cast<float*>(base + w.qrot);
    float* qproj = c->m ? reinterpret_cast<float*>(base + w.qproj) : nullptr;
    float* partials = reinterpret_cast<float*>(base + w.partials);
    if ((rc = tq_prep_queries(c, q, (int64_t)B * Hq, qrot, qproj, stream))) return rc;
    KeyCache k{kp, ks, kn, kr, cap, len};
    cudaError_t e = launch_attn_output(c, vc, qrot, qproj, B, Hq, Hkv, k, scale, values, v_norm, partials, out,
                                       static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_attn_output launch");
}

static size_t values_ws_bytes(int d, int B, int Hq, int Hkv, int64_t cap) {
    int chunk, nchunk;
    attn_chunking(nullptr, B, Hq, Hkv, cap, &chunk, &nchunk);
    // the tensor-core value kernel's chunks (values_tc_chunk) may be shorter: room for either
    const int tchunk = values_tc_chunk(B, Hq, Hkv, cap);
    const int64_t tn = (cap + tchunk - 1) / tchunk;
    if (tn > nchunk) nchunk = (int)tn;
    return round_up((size_t)B * Hq * nchunk * (d + 2) * sizeof(float), 256);
}

int tq_attn_values_workspace_size(int d, int B, int Hq, int Hkv, int64_t cap, size_t* bytes) {
    TQ_REQUIRE(bytes != nullptr, TQ_ERR_ARG, "bytes is NULL");
    TQ_REQUIRE(d >= 1 && d <= 512, TQ_ERR_ARG, "d must be in [1, 512]");
    TQ_REQUIRE(B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0 && cap >= 1, TQ_ERR_ARG,
               "need B >= 1, cap >= 1 and Hq a positive multiple of Hkv");
    *bytes = values_ws_bytes(d, B, Hq, Hkv, cap);
    return TQ_OK;
}

static int values_call(const char* name, const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv,
                       int64_t cap, const int32_t* len, const void* values, const uint16_t* v_norm, float* out,
                       void* ws, size_t ws_bytes, void* stream, float* part_out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (vc) {
        int rc = check_ctx(vc);
        if (rc) return rc;
        TQ_REQUIRE(vc->mode == TQ_MODE_MSE, TQ_ERR_ARG, "vctx must be an MSE-mode context");
        TQ_REQUIRE(vc->d == d, TQ_ERR_ARG, "d must equal vctx's d");
        TQ_REQUIRE(vc->d_hi == 0 || (d > 96 && d <= 128), TQ_ERR_UNSUPPORTED,
                   std::string(name) + " takes split (fractional bit width) value contexts at 96 < d <= 128 only");
        TQ_REQUIRE(v_norm && aligned(v_norm, 2), TQ_ERR_ARG, "coded values need v_norm");
    }
    TQ_REQUIRE(d >= 1 && d <= 512, TQ_ERR_UNSUPPORTED, std::string(name) + " supports d <= 512");
    TQ_REQUIRE(B >= 1 && Hkv >= 1 && Hq >= Hkv && Hq % Hkv == 0, TQ_ERR_ARG, "need B >= 1 and Hq a positive multiple of Hkv");
    TQ_REQUIRE(cap >= 1 && cap < (int64_t)1 << 31, TQ_ERR_ARG, "cap must be in [1, 2^31)");
    TQ_REQUIRE(logits && len && values && out && ws, TQ_ERR_ARG, "a required pointer is NULL");
    TQ_REQUIRE(aligned(logits, 4) && aligned(len, 4) && aligned(values, 16) && aligned(out, 4) && aligned(ws, 256),
               TQ_ERR_ARG, "misaligned pointer");
    TQ_REQUIRE(ws_bytes >= values_ws_bytes(d, B, Hq, Hkv, cap), TQ_ERR_ARG,
               "workspace too small (see tq_attn_values_workspace_size)");
    // without a context (bf16 values) there is no error word: out-of-range lengths are clamped
    int* err = vc ? vc->derr : nullptr;
    e = launch_attn_values(vc, d, logits, B, Hq, Hkv, cap, len, values, v_norm, err, static_cast<float*>(ws),
                           part_out ? nullptr : out, static_cast<cudaStream_t>(stream), part_out);
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, (std::string(name) + " launch").c_str());
}

int tq_attn_values(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                   const int32_t* len, const void* values, const uint16_t* v_norm, float* out, void* ws,
                   size_t ws_bytes, void* stream) {
    return values_call("tq_attn_values", vc, d, logits, B, Hq, Hkv, cap, len, values, v_norm, out, ws, ws_bytes,
                       stream, nullptr);
}

int tq_attn_values_partial(const tq_ctx* vc, int d, const float* logits, int B, int Hq, int Hkv, int64_t cap,
                           const int32_t* len, const void* values, const uint16_t* v_norm, float* part, void* ws,
                           size_t ws_bytes, void* stream) {
    return values_call("tq_attn_values_partial", vc, d, logits, B, Hq, Hkv, cap, len, values, v_norm, part, ws,
                       ws_bytes, stream, part);
}

int tq_attn_merge_partials(const tq_ctx* vc, int d, const float* parts, int R, int B, int Hq, float* out,
                           void* stream) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (vc) {
        int rc = check_ctx(vc);
        if (rc) return rc;
        TQ_REQUIRE(vc->mode == TQ_MODE_MSE && vc->d == d, TQ_ERR_ARG, "vctx must be an MSE-mode context of dimension d");
    }
    TQ_REQUIRE(d >= 1 && d <= 512, TQ_ERR_UNSUPPORTED, "tq_attn_merge_partials supports d <= 512");
    TQ_REQUIRE(R >= 1 && B >= 1 && Hq >= 1, TQ_ERR_ARG, "need R >= 1, B >= 1, Hq >= 1");
    TQ_REQUIRE(parts && out && aligned(parts, 4) && aligned(out, 4), TQ_ERR_ARG, "parts and out must be non-NULL, 4-byte aligned");
    e = launch_merge_partials(vc, d, parts, R, (int64_t)B * Hq, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_attn_merge_partials launch");
}

int tq_topk_merge(const float* cand_s, const int32_t* cand_i, int R, int64_t nq, int k, const int64_t* row_offsets,
                  float* top_s, int32_t* top_i, void* stream) {
    TQ_REQUIRE(R >= 1 && R <= kMaxShards, TQ_ERR_ARG, "R must be in [1, 64]");
    TQ_REQUIRE(k >= 1 && k <= TQ_MAX_TOPK && nq >= 0 && nq < ((int64_t)1 << 31), TQ_ERR_ARG,
               "need 1 <= k <= 128 and 0 <= nq < 2^31");
    if (nq == 0) return TQ_OK;
    TQ_REQUIRE(cand_s && cand_i && row_offsets && top_s && top_i, TQ_ERR_ARG, "a required pointer is NULL");
    TQ_REQUIRE(aligned(cand_s, 4) && aligned(cand_i, 4) && aligned(top_s, 4) && aligned(top_i, 4), TQ_ERR_ARG,
               "misaligned pointer");
    ShardOffsets offs{};
    for (int r = 0; r < R; ++r) {
        TQ_REQUIRE(row_offsets[r] >= 0 && row_offsets[r] < ((int64_t)1 << 31), TQ_ERR_ARG,
                   "row offsets must be in [0, 2^31)");
        offs.off[r] = row_offsets[r];
    }
    cudaError_t e = launch_topk_merge(cand_s, cand_i, R, nq, k, offs, top_s, top_i, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_topk_merge launch");
}

struct SearchWs {
    size_t qrot, qproj, cs, ci, total;
};

static SearchWs search_ws_layout(const tq_ctx* c, int64_t nq, int64_t n, int k) {
    int chunk, nchunk;
    search_chunking(n, k, &chunk, &nchunk);
    SearchWs w;
    w.qrot = 0;
    w.qproj = round_up((size_t)nq * c->d * sizeof(float), 256);
    w.cs = w.qproj + round_up((size_t)nq * c->m * sizeof(float), 256);
    w.ci = w.cs + round_up((size_t)nq * nchunk * k * sizeof(float), 256);
    w.total = w.ci + round_up((size_t)nq * nchunk * k * sizeof(int), 256);
    return w;
}

int tq_search_workspace_size(const tq_ctx* c, int64_t nq, int64_t n, int k, size_t* bytes) {
    TQ_REQUIRE(c && bytes, TQ_ERR_ARG, "context and bytes must be non-NULL");
    TQ_REQUIRE(nq >= 0 && n >= 1 && n < ((int64_t)1 << 31) && k >= 1 && k <= TQ_MAX_TOPK && k <= n, TQ_ERR_ARG,
               "need nq >= 0, 1 <= k <= min(n, 128), n < 2^31");
    *bytes = search_ws_layout(c, nq, n, k).total;
    return TQ_OK;
}

int tq_search_topk(tq_ctx* c, const float* q, int64_t nq, const uint32_t* planes, const uint32_t* signs,
                   const uint16_t* norm, const uint16_t* rnorm, int64_t n, int k, float* top_score, int32_t* top_idx,
                   void* ws, size_t ws_bytes, void* stream) {
    int rc = check_ctx(c);
    if (rc) return rc;
    TQ_REQUIRE(nq >= 0 && n >= 1 && n < ((int64_t)1 << 31) && k >= 1 && k <= TQ_MAX_TOPK && k <= n, TQ_ERR_ARG,
               "need nq >= 0, 1 <= k <= min(n, 128), n < 2^31");
    if (nq == 0) return TQ_OK;
    TQ_REQUIRE(c->d_hi == 0, TQ_ERR_UNSUPPORTED, "tq_search_topk does not take split (fractional bit width) contexts");
    TQ_REQUIRE(q && planes && norm && top_score && top_idx && ws, TQ_ERR_ARG, "a required pointer is NULL");
    TQ_REQUIRE(aligned(q, 16) && aligned(planes, 16) && aligned(norm, 2) && aligned(ws, 256) &&
                   aligned(top_score, 4) && aligned(top_idx, 4),
               TQ_ERR_ARG, "misaligned pointer");
    if (c->m) TQ_REQUIRE(signs && rnorm && aligned(signs, 16) && aligned(rnorm, 2), TQ_ERR_ARG, "PROD codes need signs and rnorm");
    SearchWs w = search_ws_layout(c, nq, n, k);
    TQ_REQUIRE(ws_bytes >= w.total, TQ_ERR_ARG, "workspace too small (see tq_search_workspace_size)");
    char* base = static_cast<char*>(ws);
    float* qrot = reinterpret_cast<float*>(base + w.qrot);
    float* qproj = c->m ? reinterpret_cast<float*>(base + w.qproj) : nullptr;
    if ((rc = tq_prep_queries(c, q, nq, qrot, qproj, stream))) return rc;
    cudaError_t e = launch_search(c, qrot, qproj, nq, planes, signs, norm, rnorm, n, k,
                                  reinterpret_cast<float*>(base + w.cs), reinterpret_cast<int*>(base + w.ci),
                                  top_score, top_idx, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? TQ_OK : cuda_fail(e, "tq_search_topk launch");
}

int tq_sync_status(tq_ctx* c, void* stream, int* flags) {
    int rc = check_ctx(c);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronisation");
    int v = 0;
    e = cudaMemcpy(&v, c->derr, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device error word");
    if (flags) *flags = v;
    if (v) {
        e = cudaMemset(c->derr, 0, sizeof(int));
        if (e != cudaSuccess) return cuda_fail(e, "clearing the device error word");
        return fail(TQ_ERR_DEVICE, "device-side check failed, flags " + std::to_string(v));
    }
    return TQ_OK;
}

}  // extern "C"
