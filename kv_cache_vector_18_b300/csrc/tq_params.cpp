// Host-side construction of a TurboQuant quantizer's parameters in float64.
//
// «Шаг 1» (random rotation): Π is the orthogonal factor of a Gaussian matrix,
//   made unique by requiring a positive diagonal in R.
// «QJL»: S is a Gaussian matrix, drawn from a stream independent of Π's
//   (community finding #3: a shared matrix correlates the two stages).
// «Шаг 2» (Lloyd–Max): 1-D continuous k-means for the coordinate law
//   f_X(x) = Γ(d/2)/(√π Γ((d−1)/2))·(1−x²)^((d−3)/2) on [−1, 1] (the Lemma),
//   alternating "boundaries = midpoints" and "centroids = conditional means".
//
// Walsh–Hadamard option (community finding #3 of the page: WHT for the MSE stage,
//   an independent transform for QJL): Π = H_d·diag(σ)/√d with H_d the natural-
//   order Hadamard matrix, (H_d)_ji = (−1)^popcount(j & i), and σ_i = +1 iff the
//   i-th uniform of its own stream is below ½.  S is unchanged.
//
// Numerics here are this library's own: Householder QR, and cell integrals by
// composite Gauss–Legendre quadrature of f_X and x·f_X.
#include <math.h>

#include <map>
#include <mutex>
#include <utility>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kPiStreamTag = 0x5049524F54415445ull;  // "PIROTATE"
constexpr uint64_t kSStreamTag = 0x514A4C534B455443ull;   // "QJLSKETC"
constexpr uint64_t kWhtStreamTag = 0x5748545349474E53ull; // "WHTSIGNS"

// SplitMix64 (Steele, Lea & Flood 2014), counter form: output i mixes seed + (i+1)·φ.
inline uint64_t splitmix64_at(uint64_t seed, uint64_t i) {
    uint64_t z = seed + (i + 1) * kGolden;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

inline double uniform_at(uint64_t seed, uint64_t i) {
    return (double)(splitmix64_at(seed, i) >> 11) * 0x1.0p-53;
}

// Row-major n = rows·cols i.i.d. N(0,1) values: Box–Muller on uniform pairs (2k, 2k+1).
void gaussian_fill(uint64_t seed, size_t n, double* out) {
    for (size_t k = 0; 2 * k < n; ++k) {
        double u1 = uniform_at(seed, 2 * k);
        double u2 = uniform_at(seed, 2 * k + 1);
        if (u1 == 0.0) u1 = 0x1.0p-53;
        double r = sqrt(-2.0 * log(u1));
        double a = 2.0 * M_PI * u2;
        out[2 * k] = r * cos(a);
        if (2 * k + 1 < n) out[2 * k + 1] = r * sin(a);
    }
}

// Π_ji = (−1)^popcount(j & i)·σ_i/√d.
void hadamard_rotation(int d, uint64_t seed, std::vector<double>* Pi) {
    Pi->assign((size_t)d * d, 0.0);
    const double s = 1.0 / sqrt((double)d);
    for (int i = 0; i < d; ++i) {
        const double sig = uniform_at(seed ^ kWhtStreamTag, (uint64_t)i) < 0.5 ? s : -s;
        for (int j = 0; j < d; ++j) (*Pi)[(size_t)j * d + i] = (__builtin_popcount((unsigned)(j & i)) & 1) ? -sig : sig;
    }
}

// Π = Q·diag(sign(R_ii)) for G = QR, by Householder reflections.
void rotation_from_gaussian(int d, const std::vector<double>& G, std::vector<double>* Pi) {
    std::vector<double> A(G);
    std::vector<std::vector<double>> vs(d);
    std::vector<double> rdiag(d);
    for (int k = 0; k < d; ++k) {
        double nrm = 0.0;
        for (int i = k; i < d; ++i) nrm += A[i * d + k] * A[i * d + k];
        nrm = sqrt(nrm);
        double alpha = A[k * d + k] > 0 ? -nrm : nrm;
        std::vector<double> v(d - k);
        for (int i = k; i < d; ++i) v[i - k] = A[i * d + k];
        v[0] -= alpha;
        double vn = 0.0;
        for (double e : v) vn += e * e;
        vn = sqrt(vn);
        if (vn > 0) {
            for (double& e : v) e /= vn;
            for (int j = k; j < d; ++j) {
                double dot = 0.0;
                for (int i = k; i < d; ++i) dot += v[i - k] * A[i * d + j];
                for (int i = k; i < d; ++i) A[i * d + j] -= 2.0 * dot * v[i - k];
            }
        }
        rdiag[k] = A[k * d + k];
        vs[k] = std::move(v);
    }
    // Q = H_0 H_1 … H_{d−1}: apply the reflections to I from the last one.
    std::vector<double> Q((size_t)d * d, 0.0);
    for (int i = 0; i < d; ++i) Q[i * d + i] = 1.0;
    for (int k = d - 1; k >= 0; --k) {
        const std::vector<double>& v = vs[k];
        for (int j = 0; j < d; ++j) {
            double dot = 0.0;
            for (int i = k; i < d; ++i) dot += v[i - k] * Q[i * d + j];
            for (int i = k; i < d; ++i) Q[i * d + j] -= 2.0 * dot * v[i - k];
        }
    }
    Pi->assign((size_t)d * d, 0.0);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) (*Pi)[i * d + j] = Q[i * d + j] * (rdiag[j] < 0 ? -1.0 : 1.0);
}

// 20-point Gauss–Legendre nodes/weights on [−1, 1] (Newton on P_n).
struct GaussLegendre {
    static constexpr int n = 20;
    double x[n], w[n];
    GaussLegendre() {
        for (int i = 0; i < n; ++i) {
            double z = cos(M_PI * (i + 0.75) / (n + 0.5));
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
                if (fabs(dz) < 1e-17) break;
            }
            x[i] = z;
            w[i] = 2.0 / ((1.0 - z * z) * dp * dp);
        }
    }
};

// ∫_lo^hi f_X and ∫_lo^hi x f_X by composite Gauss–Legendre (kPanels panels).
void cell_integrals(int d, double lo, double hi, double* mass, double* moment) {
    static const GaussLegendre gl;
    constexpr int kPanels = 48;
    const double cd = exp(lgamma(d / 2.0) - lgamma((d - 1) / 2.0)) / sqrt(M_PI);
    const double p = (d - 3) / 2.0;
    double m0 = 0.0, m1 = 0.0;
    const double h = (hi - lo) / kPanels;
    for (int k = 0; k < kPanels; ++k) {
        double a = lo + k * h, mid = a + 0.5 * h;
        for (int i = 0; i < GaussLegendre::n; ++i) {
            double x = mid + 0.5 * h * gl.x[i];
            double f = exp(p * log1p(-x * x));
            m0 += gl.w[i] * f;
            m1 += gl.w[i] * x * f;
        }
    }
    *mass = cd * 0.5 * h * m0;
    *moment = cd * 0.5 * h * m1;
}

void lloyd_max(int d, int levels, std::vector<double>* c_out, std::vector<double>* t_out) {
    std::vector<double> c(levels), t(levels > 1 ? levels - 1 : 0);
    if (levels == 1) {
        c[0] = 0.0;
        *c_out = c;
        *t_out = t;
        return;
    }
    const double sigma = 1.0 / sqrt((double)d);
    for (int i = 0; i < levels; ++i) c[i] = sigma * 2.5 * (2.0 * (i + 0.5) / levels - 1.0);
    double best = 1e300;
    int last_improve = 0;
    for (int it = 0; it < 100000; ++it) {
        for (int i = 0; i + 1 < levels; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
        double delta = 0.0, cmax = 0.0;
        for (int i = 0; i < levels; ++i) {
            double lo = i == 0 ? -1.0 : t[i - 1];
            double hi = i == levels - 1 ? 1.0 : t[i];
            double m0, m1;
            cell_integrals(d, lo, hi, &m0, &m1);
            double cn = m1 / m0;
            delta = fmax(delta, fabs(cn - c[i]));
            cmax = fmax(cmax, fabs(cn));
            c[i] = cn;
        }
        if (delta < best) {
            best = delta;
            last_improve = it;
        }
        if (delta <= 2e-16 * cmax || it - last_improve > 64) break;
    }
    for (int i = 0; i + 1 < levels; ++i) t[i] = 0.5 * (c[i] + c[i + 1]);
    *c_out = c;
    *t_out = t;
}

// Codebooks depend only on (d, levels); cache them process-wide.
void cached_codebook(int d, int levels, std::vector<double>* c, std::vector<double>* t) {
    static std::mutex mu;
    static std::map<std::pair<int, int>, std::pair<std::vector<double>, std::vector<double>>> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_pair(d, levels);
    auto it = cache.find(key);
    if (it == cache.end()) {
        std::vector<double> cc, tt;
        lloyd_max(d, levels, &cc, &tt);
        it = cache.emplace(key, std::make_pair(cc, tt)).first;
    }
    *c = it->second.first;
    *t = it->second.second;
}

}  // namespace

int build_host_params(int d, int bits, int variant, int rotation, uint64_t seed, HostParams* out) {
    if (d < kMinD || d > kMaxD || d % 32 != 0)
        return fail(TQ_EUNSUPPORTED, "d=%d unsupported (need a multiple of 32 in [32, 256])", d);
    if (variant != TQ_MSE && variant != TQ_PROD) return fail(TQ_EINVAL, "variant=%d invalid", variant);
    if (rotation != TQ_ROT_QR && rotation != TQ_ROT_HADAMARD) return fail(TQ_EINVAL, "rotation=%d invalid", rotation);
    if (rotation == TQ_ROT_HADAMARD && (d & (d - 1)) != 0)
        return fail(TQ_EUNSUPPORTED, "the Hadamard rotation needs d a power of two (d=%d)", d);
    if (bits < 1 || bits > 4) return fail(TQ_EUNSUPPORTED, "bits=%d unsupported (1..4)", bits);
    HostParams hp;
    hp.d = d;
    hp.bits = bits;
    hp.variant = variant;
    hp.seed = seed;
    hp.rotation = rotation;
    hp.b_mse = variant == TQ_MSE ? bits : bits - 1;
    hp.levels = 1 << hp.b_mse;
    if (rotation == TQ_ROT_QR) {
        std::vector<double> G((size_t)d * d);
        gaussian_fill(seed ^ kPiStreamTag, G.size(), G.data());
        rotation_from_gaussian(d, G, &hp.Pi);
    } else {
        hadamard_rotation(d, seed, &hp.Pi);
    }
    if (variant == TQ_PROD) {
        hp.S.resize((size_t)d * d);
        gaussian_fill(seed ^ kSStreamTag, hp.S.size(), hp.S.data());
    }
    cached_codebook(d, hp.levels, &hp.centroids, &hp.bounds);
    *out = std::move(hp);
    return TQ_OK;
}

}  // namespace tq
