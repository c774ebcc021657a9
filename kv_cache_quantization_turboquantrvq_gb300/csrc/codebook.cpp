// codebook.cpp - host-side TurboQuantRVQ codebooks (binary64, rounded to fp32).
//
// VeloxQuant-MLX blog, tag "rvq", "The pipeline, as it actually runs": stage 1
// quantizes the rotated row against a Gaussian codebook and stage 2 quantizes
// the residual against a Laplacian-fit codebook; "What 'quantize' means here,
// precisely": boundaries are midpoints of sorted centroids.  The pages do not
// spell out how the codebooks are built; this library uses the Lloyd-Max
// (minimum mean-squared-error) quantizers of
//   stage 1: N(0, 1/D), the distribution of a coordinate of a rotated unit row;
//   stage 2: Laplace(0, beta), beta = E|r| (Laplace maximum-likelihood scale)
//            of the stage-1 residual r under N(0, 1/D).
// Both densities are symmetric, so each quantizer is iterated on its positive
// half and mirrored, which makes the codebooks exactly antisymmetric.
#include <cmath>
#include <cstring>

namespace vq {
namespace {

double phi(double z) { return std::exp(-0.5 * z * z) * 0.39894228040143267794; }

// P(a < Z <= b), Z standard normal, with complementary error functions in the tails.
double norm_mass(double a, double b)
{
    const double r2 = 0.70710678118654752440;
    if (a >= 0.0) return 0.5 * (std::erfc(a * r2) - std::erfc(b * r2));
    if (b <= 0.0) return 0.5 * (std::erfc(-b * r2) - std::erfc(-a * r2));
    return 1.0 - 0.5 * std::erfc(-a * r2) - 0.5 * std::erfc(b * r2);
}

// Conditional mean of N(0, s^2) on (a, b].
double gauss_mean(double a, double b, double s)
{
    const double za = a / s, zb = b / s;
    const double pa = std::isinf(za) ? 0.0 : phi(za);
    const double pb = std::isinf(zb) ? 0.0 : phi(zb);
    return s * (pa - pb) / norm_mass(za, zb);
}

// Conditional mean of Laplace(0, beta) on (a, b], 0 <= a < b: the positive
// half is an exponential law with mean beta.
double laplace_mean(double a, double b, double beta)
{
    if (std::isinf(b)) return a + beta;
    const double ea = std::exp(-a / beta), eb = std::exp(-b / beta);
    return beta + (a * ea - b * eb) / (ea - eb);
}

// Lloyd-Max on the positive half: m = levels/2 centroids, cells
// [0, t1], (t1, t2], ..., (t_{m-1}, inf) with t_k the midpoints.
bool lloyd_half(int levels, bool gaussian, double scale, double *half)
{
    const int m = levels / 2;
    for (int k = 0; k < m; ++k) half[k] = scale * (3.0 * k + 1.5) / m;
    for (int it = 0; it < 2000000; ++it) {
        double moved = 0.0;
        for (int k = 0; k < m; ++k) {
            const double lo = k == 0 ? 0.0 : 0.5 * (half[k - 1] + half[k]);
            const double hi = k == m - 1 ? INFINITY : 0.5 * (half[k] + half[k + 1]);
            const double c = gaussian ? gauss_mean(lo, hi, scale) : laplace_mean(lo, hi, scale);
            moved = std::fmax(moved, std::fabs(c - half[k]));
            half[k] = c;
        }
        if (moved <= 1e-15 * scale) return true;
    }
    return false;
}

void mirror(int levels, const double *half, double *c)
{
    const int m = levels / 2;
    for (int k = 0; k < m; ++k) {
        c[m + k] = half[k];
        c[m - 1 - k] = -half[k];
    }
}

// E|Y - c[i(Y)]| for Y ~ N(0, s^2): per cell, split at the centroid and use
// int_u^v (y - c) phi_s(y) dy = s^2 (phi_s(u) - phi_s(v)) - c P(u < Y <= v).
double residual_mean_abs(int levels, const double *c, double s)
{
    double tot = 0.0;
    for (int k = 0; k < levels; ++k) {
        const double lo = k == 0 ? -INFINITY : 0.5 * (c[k - 1] + c[k]);
        const double hi = k == levels - 1 ? INFINITY : 0.5 * (c[k] + c[k + 1]);
        const double zl = lo / s, zc = c[k] / s, zh = hi / s;
        const double pl = std::isinf(zl) ? 0.0 : phi(zl);
        const double ph = std::isinf(zh) ? 0.0 : phi(zh);
        const double pc = phi(zc);
        tot += s * (pc - ph) - c[k] * norm_mass(zc, zh);  // above the centroid
        tot += c[k] * norm_mass(zl, zc) - s * (pl - pc);  // below the centroid
    }
    return tot;
}

}  // namespace

bool rvq_codebook_f64(int D, int bits, double *g, double *l, double *beta_out)
{
    const int L = 1 << bits;
    double half[32];
    const double sigma = 1.0 / std::sqrt((double)D);
    if (!lloyd_half(L, true, sigma, half)) return false;
    mirror(L, half, g);
    const double beta = residual_mean_abs(L, g, sigma);
    if (!lloyd_half(L, false, beta, half)) return false;
    mirror(L, half, l);
    if (beta_out) *beta_out = beta;
    return true;
}

}  // namespace vq
