// tq_codebook.cpp -- host-side Lloyd-Max solver for the turbo3 / turbo2 codebooks.
//
// "llama.cpp に TurboQuant を実装", section "What TurboQuant does differently": after the
// Walsh-Hadamard rotation every coordinate of a normalised block follows the same,
// outlier-free law, and a fixed Lloyd-Max scalar quantiser per coordinate is near
// optimal -- no calibration data.  The law is that of one coordinate Y of a uniformly
// random unit vector in R^d (d = 128): Y^2 ~ Beta(1/2, (d-1)/2), density
// f(y) = K (1 - y^2)^((d-3)/2) on [-1, 1].
//
// Lloyd's fixed point: thresholds are midpoints of neighbouring centroids, and every
// centroid is the conditional mean of its cell.  Here the cell mass comes from the
// regularised incomplete beta function (Lentz continued fraction) and the first moment
// from its closed form  int y f = K/(2(a+1)) [(1-y^2)^(a+1)]  with a = (d-3)/2.
#include <cmath>
#include <cstring>

#include "tq_internal.cuh"

namespace tq {
namespace {

constexpr int kDim = kBlock;

// Continued fraction of the incomplete beta function, modified Lentz method.
double beta_cf(double p, double q, double x) {
    const double tiny = 1e-300;
    double c = 1.0, d = 1.0 - (p + q) * x / (p + 1.0);
    if (std::fabs(d) < tiny) d = tiny;
    d = 1.0 / d;
    double h = d;
    for (int m = 1; m <= 10000; ++m) {
        double m2 = 2.0 * m;
        double aa = m * (q - m) * x / ((p + m2 - 1.0) * (p + m2));
        d = 1.0 + aa * d;
        if (std::fabs(d) < tiny) d = tiny;
        c = 1.0 + aa / c;
        if (std::fabs(c) < tiny) c = tiny;
        d = 1.0 / d;
        h *= d * c;
        aa = -(p + m) * (p + q + m) * x / ((p + m2) * (p + m2 + 1.0));
        d = 1.0 + aa * d;
        if (std::fabs(d) < tiny) d = tiny;
        c = 1.0 + aa / c;
        if (std::fabs(c) < tiny) c = tiny;
        d = 1.0 / d;
        double del = d * c;
        h *= del;
        if (std::fabs(del - 1.0) < 1e-17) break;
    }
    return h;
}

// Regularised incomplete beta I_x(p, q).
double inc_beta(double p, double q, double x) {
    if (x <= 0.0) return 0.0;
    if (x >= 1.0) return 1.0;
    double lbeta = std::lgamma(p) + std::lgamma(q) - std::lgamma(p + q);
    double front = std::exp(p * std::log(x) + q * std::log1p(-x) - lbeta);
    if (x < (p + 1.0) / (p + q + 2.0)) return front * beta_cf(p, q, x) / p;
    return 1.0 - front * beta_cf(q, p, 1.0 - x) / q;
}

// G(y) = P(0 < Y <= y) for y >= 0 and -P(y < Y < 0) for y < 0, so that the mass of
// (a, b] is G(b) - G(a) without cancellation around 1/2.
double half_cdf(double y) {
    const double p = 0.5, q = 0.5 * (kDim - 1);
    double g = 0.5 * inc_beta(p, q, y * y);
    return y < 0.0 ? -g : g;
}

// Unnormalised first moment primitive: int y (1-y^2)^a dy = -(1-y^2)^(a+1) / (2(a+1)).
double moment_prim(double y) {
    const double a = 0.5 * (kDim - 3);
    double u = 1.0 - y * y;
    if (u <= 0.0) return 0.0;
    return -std::pow(u, a + 1.0) / (2.0 * (a + 1.0));
}

}  // namespace

void solve_codebook(int levels, double *centroids) {
    const double a = 0.5 * (kDim - 3);
    // normalising constant K = Gamma(d/2) / (sqrt(pi) Gamma((d-1)/2))
    const double K = std::exp(std::lgamma(0.5 * kDim) - std::lgamma(0.5 * (kDim - 1)) -
                              0.5 * std::log(M_PI));
    (void)a;
    double c[8], edge[9];
    // start from equally likely cells: evenly spaced over +-2 standard deviations
    const double sd = 1.0 / std::sqrt((double)kDim);
    for (int j = 0; j < levels; ++j) c[j] = sd * (-2.0 + 4.0 * (j + 0.5) / levels);
    for (int it = 0; it < 20000; ++it) {
        edge[0] = -1.0;
        edge[levels] = 1.0;
        for (int j = 1; j < levels; ++j) edge[j] = 0.5 * (c[j - 1] + c[j]);
        double move = 0.0;
        for (int j = 0; j < levels; ++j) {
            double mass = half_cdf(edge[j + 1]) - half_cdf(edge[j]);
            double mom = K * (moment_prim(edge[j + 1]) - moment_prim(edge[j]));
            double cn = mom / mass;
            move = std::fmax(move, std::fabs(cn - c[j]));
            c[j] = cn;
        }
        if (move < 1e-16) break;
    }
    std::memcpy(centroids, c, sizeof(double) * (size_t)levels);
}

}  // namespace tq
