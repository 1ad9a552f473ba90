// Host-side set-up of a TurboQuant context: seeded matrices, the Lloyd-Max table and its
// Walsh form.  Runs once per context, in float64, on the CPU.
//
// Pages: freelamp.com article 0328, section 技术突破 (a random orthogonal rotation first,
// after which the coordinates follow a predictable law); gitcode.csdn.net tutorial,
// section QJL step 1 (Gaussian JL projection of the residual); nonndazone.ru essay,
// sections 3.2 and 3.4 (centroids placed where probability is high, precomputed once
// for all tokens and layers).
#include <algorithm>
#include <cmath>
#include <stdexcept>
#include <vector>

#include "tq_internal.h"

namespace tq {
namespace {

// ---------------------------------------------------------------- random numbers
// splitmix64 (Steele, Lea, Flood, OOPSLA 2014), output k uses state seed + (k+1)*gamma.
struct SplitMix64 {
    uint64_t state;
    explicit SplitMix64(uint64_t s) : state(s) {}
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ULL;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        return z ^ (z >> 31);
    }
    // uniform in (0, 1]
    double uniform() { return (static_cast<double>(next() >> 11) + 1.0) * 0x1.0p-53; }
};

// Box-Muller: each pair of uniforms (u1, u2) yields r cos(2 pi u2), r sin(2 pi u2).
std::vector<double> normals(uint64_t seed, size_t count) {
    SplitMix64 g(seed);
    std::vector<double> out(count + 1);
    for (size_t k = 0; k < count; k += 2) {
        double u1 = g.uniform(), u2 = g.uniform();
        double r = std::sqrt(-2.0 * std::log(u1));
        double th = 2.0 * M_PI * u2;
        out[k] = r * std::cos(th);
        out[k + 1] = r * std::sin(th);
    }
    out.resize(count);
    return out;
}

// Householder QR of the row-major n x n matrix A; returns Q with the columns' signs fixed
// so that diag(R) > 0 (Q diag(sign(diag R)) is Haar-distributed when A is Gaussian).
std::vector<double> haar_from_gaussian(std::vector<double> A, int n) {
    std::vector<std::vector<double>> vs(n);
    std::vector<double> rdiag(n);
    for (int k = 0; k < n; ++k) {
        double norm2 = 0.0;
        for (int i = k; i < n; ++i) norm2 += A[(size_t)i * n + k] * A[(size_t)i * n + k];
        double nx = std::sqrt(norm2);
        double x0 = A[(size_t)k * n + k];
        double alpha = (x0 >= 0.0) ? -nx : nx;   // reflect onto -sign(x0) ||x|| e1
        std::vector<double> v(n - k);
        for (int i = k; i < n; ++i) v[i - k] = A[(size_t)i * n + k];
        v[0] -= alpha;
        double vn2 = 0.0;
        for (double e : v) vn2 += e * e;
        if (vn2 > 0.0) {
            double inv = 1.0 / std::sqrt(vn2);
            for (double& e : v) e *= inv;
            for (int j = k; j < n; ++j) {
                double dot = 0.0;
                for (int i = k; i < n; ++i) dot += v[i - k] * A[(size_t)i * n + j];
                for (int i = k; i < n; ++i) A[(size_t)i * n + j] -= 2.0 * v[i - k] * dot;
            }
        } else {
            alpha = x0;
        }
        rdiag[k] = alpha;
        vs[k] = std::move(v);
    }
    // Q = H_0 H_1 ... H_{n-1}: apply the reflectors in reverse order to the identity.
    std::vector<double> Q((size_t)n * n, 0.0);
    for (int i = 0; i < n; ++i) Q[(size_t)i * n + i] = 1.0;
    for (int k = n - 1; k >= 0; --k) {
        const std::vector<double>& v = vs[k];
        if (v.empty()) continue;
        for (int j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int i = k; i < n; ++i) dot += v[i - k] * Q[(size_t)i * n + j];
            for (int i = k; i < n; ++i) Q[(size_t)i * n + j] -= 2.0 * v[i - k] * dot;
        }
    }
    for (int j = 0; j < n; ++j) {
        if (rdiag[j] < 0.0)
            for (int i = 0; i < n; ++i) Q[(size_t)i * n + j] = -Q[(size_t)i * n + j];
    }
    return Q;
}

// ---------------------------------------------------------------- quadrature
struct GaussLegendre {
    std::vector<double> x, w;   // nodes and weights on [-1, 1]
    explicit GaussLegendre(int n) : x(n), w(n) {
        for (int i = 0; i < n; ++i) {
            double z = std::cos(M_PI * (i + 0.75) / (n + 0.5));
            double dp = 0.0;
            for (int it = 0; it < 100; ++it) {
                double p0 = 1.0, p1 = z;
                for (int k = 2; k <= n; ++k) {
                    double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                    p0 = p1;
                    p1 = p2;
                }
                dp = n * (z * p1 - p0) / (z * z - 1.0);
                double dz = p1 / dp;
                z -= dz;
                if (std::fabs(dz) < 1e-16) break;
            }
            x[i] = z;
            w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
        }
    }
};

struct SphereMarginal {
    int d;
    double log_c;
    double reach;   // beyond |t| > reach the density is below 1e-40 of its peak
    GaussLegendre gl{32};
    explicit SphereMarginal(int d_) : d(d_) {
        log_c = std::lgamma(d / 2.0) - 0.5 * std::log(M_PI) - std::lgamma((d - 1) / 2.0);
        reach = std::min(1.0, 14.0 / std::sqrt((double)d));
    }
    double pdf(double t) const {
        if (std::fabs(t) >= 1.0) return 0.0;
        return std::exp(log_c + 0.5 * (d - 3) * std::log1p(-t * t));
    }
    // (integral of f, integral of t f) over (a, b), composite 32-point Gauss-Legendre.
    void moments(double a, double b, double& m0, double& m1) const {
        a = std::max(a, -reach);
        b = std::min(b, reach);
        m0 = m1 = 0.0;
        if (b <= a) return;
        double h = 0.25 / std::sqrt((double)d);
        int panels = std::max(1, (int)std::ceil((b - a) / h));
        double step = (b - a) / panels;
        for (int p = 0; p < panels; ++p) {
            double lo = a + p * step, mid = lo + 0.5 * step, half = 0.5 * step;
            for (size_t i = 0; i < gl.x.size(); ++i) {
                double t = mid + half * gl.x[i];
                double f = pdf(t) * gl.w[i] * half;
                m0 += f;
                m1 += t * f;
            }
        }
    }
};

}  // namespace

void seeded_matrices(uint64_t seed, int d, int m, std::vector<double>& Pi, std::vector<double>& S) {
    std::vector<double> g = normals(seed, (size_t)m * d + (size_t)d * d);
    S.assign(g.begin(), g.begin() + (size_t)m * d);
    std::vector<double> G(g.begin() + (size_t)m * d, g.end());
    Pi = haar_from_gaussian(std::move(G), d);
}

// One Lloyd step from centroids c: thresholds t at the midpoints, and per cell its probability
// m0, first moment m1 and mean g = m1 / m0 (the new centroid).
static void lloyd_cells(const SphereMarginal& f, const std::vector<double>& c, std::vector<double>& t,
                        std::vector<double>& m0, std::vector<double>& g) {
    const int L = (int)c.size();
    t.resize(L - 1);
    m0.resize(L);
    g.resize(L);
    for (int k = 0; k + 1 < L; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
    for (int k = 0; k < L; ++k) {
        const double a = (k == 0) ? -1.0 : t[k - 1];
        const double b = (k == L - 1) ? 1.0 : t[k];
        double p0, p1;
        f.moments(a, b, p0, p1);
        m0[k] = p0;
        g[k] = p0 > 0.0 ? p1 / p0 : c[k];
    }
}

// Start for many levels: the high-resolution optimum, whose centroid density is proportional to
// f^(1/3) = (1 - t^2)^((d-3)/6) (up to a constant): its quantiles at (k + 1/2) / L, from the
// cumulative integral of f^(1/3) on a fine grid (composite Gauss-Legendre), linearly interpolated.
static std::vector<double> high_rate_start(int d, int L) {
    const double reach = std::min(1.0, 40.0 / std::sqrt((double)d));
    const int panels = 8192;
    const double step = 2.0 * reach / panels;
    GaussLegendre gl(16);
    std::vector<double> edge(panels + 1), cum(panels + 1, 0.0);
    for (int i = 0; i <= panels; ++i) edge[i] = -reach + i * step;
    for (int i = 0; i < panels; ++i) {
        const double mid = edge[i] + 0.5 * step, half = 0.5 * step;
        double acc = 0.0;
        for (size_t n = 0; n < gl.x.size(); ++n) {
            const double x = mid + half * gl.x[n];
            acc += gl.w[n] * half * std::exp((d - 3) / 6.0 * std::log1p(-x * x));
        }
        cum[i + 1] = cum[i] + acc;
    }
    std::vector<double> c(L);
    int i = 0;
    for (int k = 0; k < L; ++k) {
        const double target = (k + 0.5) / L * cum[panels];
        while (i + 1 < panels && cum[i + 1] < target) ++i;
        const double w = cum[i + 1] - cum[i];
        c[k] = edge[i] + (w > 0.0 ? (target - cum[i]) / w : 0.5) * step;
    }
    return c;
}

// Lloyd-Max: thresholds at midpoints of adjacent centroids, centroids at the conditional
// means of their cells; the fixed point is unique (f_d is log-concave for d >= 3).
// Up to 4 bits it is reached by repeating the Lloyd step.  From 5 bits on one step contracts the
// error by only ~1 - O(1/L^2), so the same conditions are solved by Newton's method on
// F(c) = g(c) - c from the high-rate start: with A_k = f(lo_k)(g_k - lo_k)/m0_k and
// B_k = f(hi_k)(hi_k - g_k)/m0_k (the cell mean's derivatives in its edges, each edge moving by
// 1/2 with its two centroids) the Jacobian of c - g is tridiagonal, row k being
// (-A_k/2, 1 - (A_k + B_k)/2, -B_k/2); it is solved by the Thomas algorithm, a step that would
// break the ordering is halved, and the solve stops once a further Lloyd step would move no
// centroid by more than 5e-14 (the rounding level of the step's quadrature).
void lloyd_max_codebook(int d, int bits, std::vector<double>& c, std::vector<double>& t) {
    const int L = 1 << bits;
    SphereMarginal f(d);
    c.resize(L);
    t.resize(L - 1);
    std::vector<double> m0, g;
    if (bits <= 4) {
        const double spread = std::min(1.0, 2.0 / std::sqrt((double)d));   // start inside (-1, 1)
        for (int k = 0; k < L; ++k) c[k] = (2.0 * k + 1.0 - L) / L * spread;
        for (int it = 0; it < 200000; ++it) {
            lloyd_cells(f, c, t, m0, g);
            double moved = 0.0;
            for (int k = 0; k < L; ++k) moved = std::max(moved, std::fabs(g[k] - c[k]));
            c = g;
            if (moved < 4e-16) break;   // at the fixed point up to rounding
        }
    } else {
        c = high_rate_start(d, L);
        std::vector<double> lo(L), di(L), up(L), rhs(L), step(L), cn(L);
        for (int it = 0; it < 200; ++it) {
            lloyd_cells(f, c, t, m0, g);
            double res = 0.0;
            for (int k = 0; k < L; ++k) res = std::max(res, std::fabs(g[k] - c[k]));
            if (res <= 5e-14) break;
            for (int k = 0; k < L; ++k) {
                const double a = (k == 0) ? -1.0 : t[k - 1];
                const double b = (k == L - 1) ? 1.0 : t[k];
                const double A = (k == 0) ? 0.0 : f.pdf(a) * (g[k] - a) / m0[k];
                const double B = (k == L - 1) ? 0.0 : f.pdf(b) * (b - g[k]) / m0[k];
                lo[k] = -0.5 * A;
                di[k] = 1.0 - 0.5 * (A + B);
                up[k] = -0.5 * B;
                rhs[k] = g[k] - c[k];
            }
            // Thomas algorithm: forward elimination, back substitution
            for (int k = 1; k < L; ++k) {
                const double w = lo[k] / di[k - 1];
                di[k] -= w * up[k - 1];
                rhs[k] -= w * rhs[k - 1];
            }
            step[L - 1] = rhs[L - 1] / di[L - 1];
            for (int k = L - 2; k >= 0; --k) step[k] = (rhs[k] - up[k] * step[k + 1]) / di[k];
            for (int halvings = 0; halvings < 60; ++halvings) {
                bool ok = true;
                for (int k = 0; k < L; ++k) cn[k] = c[k] + step[k];
                if (!(cn[0] > -1.0 && cn[L - 1] < 1.0)) ok = false;
                for (int k = 0; ok && k + 1 < L; ++k) ok = cn[k] < cn[k + 1];
                if (ok) break;
                for (double& v : step) v *= 0.5;
            }
            c = cn;
        }
    }
    for (int k = 0; k < L / 2; ++k) {   // the density is even: symmetrise
        double s = 0.5 * (c[L - 1 - k] - c[k]);
        c[k] = -s;
        c[L - 1 - k] = s;
    }
    for (int k = 0; k + 1 < L; ++k) t[k] = 0.5 * (c[k] + c[k + 1]);
    if (L % 2 == 0) t[L / 2 - 1] = 0.0;
}

// Walsh form of a table indexed by bits b_0..b_{P-1} (b_0 the least significant): with
// s_i = 2 b_i - 1, c(idx) = sum_S chat_S prod_{i in S} s_i, chat_S = mean_idx c(idx)
// prod_{i in S} s_i(idx).  Since prod_{i in S} s_i = (-1)^|S| (1 - 2 x_S), x_S the parity
// of the bits in S, a dot product with a query q becomes
//     sum_j q_j c(idx_j) = c(0) sum_j q_j + sum_{S != 0} kappa_S sum_j q_j x_{S,j},
// kappa_S = -2 (-1)^|S| chat_S: masked sums of q over whole bit-plane words (XORs of planes).
// For the symmetric Lloyd-Max table only the odd-|S| terms are nonzero.
void walsh_form(const std::vector<double>& c, int bits, double& c0, std::vector<int>& masks,
                std::vector<double>& kappa) {
    const int L = 1 << bits;
    double cmax = 0.0;
    for (double v : c) cmax = std::max(cmax, std::fabs(v));
    masks.clear();
    kappa.clear();
    c0 = c[0];
    for (int S = 1; S < L; ++S) {
        double acc = 0.0;
        for (int idx = 0; idx < L; ++idx) {
            double p = 1.0;
            for (int i = 0; i < bits; ++i)
                if (S >> i & 1) p *= ((idx >> i) & 1) ? 1.0 : -1.0;
            acc += c[idx] * p;
        }
        double chat = acc / L;
        if (std::fabs(chat) <= 1e-14 * cmax) continue;
        int pc = __builtin_popcount(S);
        masks.push_back(S);
        kappa.push_back(-2.0 * ((pc & 1) ? -1.0 : 1.0) * chat);
    }
}

}  // namespace tq

namespace tq {

// Lloyd-Max table of the level-`level` angles of the recursive polar transform.  Level 1 angles
// are uniform on [0, 2 pi): the uniform table (cells [j D, (j+1) D), centroids (j + 1/2) D).
// A level-l angle (l >= 2) is atan2 of two independent chi radii with k = 2^(l-1) degrees of
// freedom, density proportional to (sin psi cos psi)^(k-1) on [0, pi/2], which is log-concave:
// the Lloyd iteration (midpoint thresholds, cell means by composite Gauss-Legendre) has one fixed
// point, symmetric about pi/4.
void polar_angle_codebook(int level, int bits, std::vector<double>& c, std::vector<double>& t) {
    const int L = 1 << bits;
    c.resize(L);
    t.resize(L - 1);
    if (level == 1) {
        const double D = 2.0 * M_PI / L;
        for (int j = 0; j < L; ++j) c[j] = (j + 0.5) * D;
        for (int j = 0; j + 1 < L; ++j) t[j] = (j + 1) * D;
        return;
    }
    const double k = std::ldexp(1.0, level - 1);
    const double q = M_PI / 4.0;
    const double reach = std::min(q, 12.0 / std::sqrt(k));   // the density is negligible beyond
    const double h = std::min(q / 4.0, 0.25 / std::sqrt(k));
    GaussLegendre gl(32);
    auto logf = [&](double psi) { return (k - 1.0) * std::log(std::sin(2.0 * psi)); };
    const double logpeak = logf(q);
    auto moments = [&](double a, double b, double& m0, double& m1) {
        a = std::max(a, q - reach);
        b = std::min(b, q + reach);
        m0 = m1 = 0.0;
        if (b <= a) return;
        const int panels = std::max(1, (int)std::ceil((b - a) / h));
        const double step = (b - a) / panels;
        for (int p = 0; p < panels; ++p) {
            const double mid = a + (p + 0.5) * step, half = 0.5 * step;
            for (size_t i = 0; i < gl.x.size(); ++i) {
                const double psi = mid + half * gl.x[i];
                const double f = std::exp(logf(psi) - logpeak) * gl.w[i] * half;
                m0 += f;
                m1 += psi * f;
            }
        }
    };
    const double spread = std::min(q, 1.5 / std::sqrt(k));
    for (int j = 0; j < L; ++j) c[j] = q + (2.0 * j + 1.0 - L) / L * spread;
    std::vector<double> cn(L);
    for (int it = 0; it < 200000; ++it) {
        for (int j = 0; j + 1 < L; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
        double moved = 0.0;
        for (int j = 0; j < L; ++j) {
            const double a = (j == 0) ? 0.0 : t[j - 1];
            const double b = (j == L - 1) ? 2.0 * q : t[j];
            double m0, m1;
            moments(a, b, m0, m1);
            cn[j] = m0 > 0.0 ? m1 / m0 : c[j];
            moved = std::max(moved, std::fabs(cn[j] - c[j]));
        }
        c = cn;
        if (moved < 1e-15) break;
    }
    for (int j = 0; j < L / 2; ++j) {   // symmetric about pi/4
        const double s = 0.5 * ((c[L - 1 - j] - q) - (c[j] - q));
        c[j] = q - s;
        c[L - 1 - j] = q + s;
    }
    for (int j = 0; j + 1 < L; ++j) t[j] = 0.5 * (c[j] + c[j + 1]);
    if (L % 2 == 0) t[L / 2 - 1] = q;
}

}  // namespace tq
