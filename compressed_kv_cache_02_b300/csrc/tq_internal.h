// Internal types shared by the host set-up code and the CUDA translation units of libtq.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "tq.h"

namespace tq {

// The table kernels (byte tables, Walsh form, tensor-core logits, the tcgen05 quantizer) and the
// tables carried in the kernel parameters cover up to kFastBits MSE bits; wider MSE-mode tables
// (up to TQ_MAX_MSE_BITS) live in device memory (Params::tab) and take the generic kernels.
constexpr int kFastBits = 4;
constexpr int kMaxLevels = 1 << kFastBits;           // 16 centroids in the parameter tables
constexpr int kMaxTerms = kMaxLevels - 1;            // nonzero subsets of the bit planes
constexpr int kMaxCodeLevels = 1 << TQ_MAX_MSE_BITS; // 256: the widest table

// Everything a kernel needs about a context, passed by value as a kernel parameter.
struct Params {
    int d, m, P, L, W, Ws;   // dimension, JL rows (0 in MSE mode), planes, levels, words
    const float* tab;        // device: the L centroids then the L - 1 thresholds (float32), any P
    int qjl;                 // 1 in PROD mode
    float qjl_scale;         // sqrt(pi/2) / m
    float centroids[kMaxLevels];    // the first min(L, 16) entries of tab (P <= kFastBits: all)
    float thresholds[kMaxLevels];
    // Walsh form (P <= kFastBits only; nterms = 0 and odd_walsh = 0 above) of the table (see host_setup.cpp): c(idx) = c0 + sum_t kappa[t] * x_t(idx),
    // where x_t(idx) = parity of the idx bits selected by mask[t].
    float c0;
    int nterms;
    int odd_walsh;   // 1 when the terms are exactly the odd-size subsets in increasing order
    int mask[kMaxTerms];
    float kappa[kMaxTerms];
    // Split (fractional bit width) contexts: coordinates j < d_hi use the (P+1)-bit table below
    // and store bit P of idx in a partial top plane of W_hi words after the P full planes.
    int d_hi;        // 0: every coordinate uses the P-bit table
    int W_hi;        // words of the top plane, ceil(d_hi / 32)
    int row_words;   // words per code row: P * W + W_hi
    float centroids_hi[kMaxLevels];
    float thresholds_hi[kMaxLevels];
    // Walsh forms over the P + 1 planes of a split row (the top plane read as 0 for coordinates
    // >= d_hi): term t is the t-th odd subset of P + 1 bits; kappa_lo_x is the P-bit table's
    // coefficient of that subset (0 when it contains bit P), kappa_hi the (P+1)-bit table's.
    float c0_hi;
    int split_walsh;   // 1 when both tables are odd (symmetric) in these terms
    float kappa_hi[kMaxTerms];
    float kappa_lo_x[kMaxTerms];
};

// Host-side set-up (host_setup.cpp).
void lloyd_max_codebook(int d, int bits, std::vector<double>& centroids,
                        std::vector<double>& thresholds);
void seeded_matrices(uint64_t seed, int d, int m, std::vector<double>& Pi,
                     std::vector<double>& S);
void walsh_form(const std::vector<double>& centroids, int bits, double& c0,
                std::vector<int>& masks, std::vector<double>& kappa);
void polar_angle_codebook(int level, int bits, std::vector<double>& centroids,
                          std::vector<double>& thresholds);

// Thread-local error message (tq_api.cu).
int fail(int code, const std::string& msg);

}  // namespace tq

struct tq_ctx {
    int device = 0;
    int d = 0, m = 0, bits = 0, mode = 0, P = 0, L = 0, W = 0, Ws = 0;
    std::vector<float> Pi, S;                 // float32 host copies, row-major
    std::vector<double> centroids, thresholds;
    int d_hi = 0;                                   // split contexts: see Params
    std::vector<double> centroids_hi, thresholds_hi;
    tq::Params prm{};
    float* dPiT = nullptr;    // [d][d]  PiT[j*d+i] = Pi[i][j]      (y = Pi x)
    float* dPi = nullptr;     // [d][d]  row-major Pi                (o = Pi^T a)
    float* dST = nullptr;     // [d][m]  ST[j*m+i] = S[i][j]        (u = S q)
    float* dStT = nullptr;    // [d][m]  StT[j*m+i] = (S Pi^T)[i][j] (S r = (S Pi^T)(Pi x - n c))
    uint16_t* bops = nullptr; // d = 128: tcgen05 B operands (2 bf16 pieces of Pi, of S Pi^T)
    float* dtab = nullptr;    // [L centroids | L - 1 thresholds] float32 (Params::tab)
    int* derr = nullptr;      // device error word
    int kernel_path = TQ_PATH_AUTO;   // logits kernel family (tq_set_kernel_path)
};
