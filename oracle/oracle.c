/*
 * Reference oracle for the KV-cache flush codecs (TurboQuantRVQ and KIVI).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, single-threaded
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or constant with the CUDA library, and the product path never
 * loads it.  Everything is computed in IEEE binary64 unless a step states a
 * narrower precision on purpose (the stored fp32 norm, the fp32/fp16 KIVI
 * scale, the fp16 outputs).
 *
 * Sources (web pages, cited by title and section):
 *   [RVQ]  VeloxQuant-MLX blog, tag "rvq": the post on fusing the TurboQuantRVQ
 *          quantize -> pack chain into one kernel.
 *   [TQ]   VeloxQuant-MLX blog, tag "turboquant": "five hand-tuned Metal
 *          compute kernels" post.
 *   [KIVI] VeloxQuant-MLX blog, tag "kivi", first post (two bit-exact KIVI
 *          kernels) and second post (KIVI 0.8.0 release, "What KIVI is").
 *
 * Parity pins: every exported function is pinned by a test under tests/
 * (test_oracle_*.py) against closed forms, textbook values, brute force or
 * invariants; none is pinned only against itself.
 */
#define _DEFAULT_SOURCE
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* IEEE binary16 <-> binary64, written out from the format definition.       */
/* ------------------------------------------------------------------------ */

/* Exact value of an IEEE binary16 bit pattern. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)man, -24); /* subnormal: man * 2^-24 */
    } else if (exp == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp((double)(man | 0x400), exp - 25); /* (1024+man) * 2^(exp-15-10) */
    }
    return sign ? -v : v;
}

/* Round a binary64 value to the nearest binary16 (ties to even). */
uint16_t oracle_f64_to_f16_rn(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00; /* rounds to infinity */
    /* Find the quantum (spacing) of binary16 numbers around a. */
    int e;
    double quantum;
    if (a < ldexp(1.0, -14)) {
        quantum = ldexp(1.0, -24); /* subnormal range */
    } else {
        frexp(a, &e);               /* a = f * 2^e, f in [0.5, 1) */
        quantum = ldexp(1.0, e - 11); /* 11 significant bits */
    }
    double q = a / quantum;           /* exact: quantum is a power of two */
    double fl = floor(q);
    double frac = q - fl;             /* exact */
    double n;
    if (frac > 0.5) n = fl + 1.0;
    else if (frac < 0.5) n = fl;
    else n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double r = n * quantum;           /* exact */
    /* Re-encode r, which is a binary16 value (or 65536 -> inf, handled above). */
    if (r == 0.0) return sign;
    if (r < ldexp(1.0, -14)) {
        return sign | (uint16_t)(r / ldexp(1.0, -24));
    }
    frexp(r, &e);
    int biased = e - 1 + 15;
    double man = r / ldexp(1.0, e - 11) - 1024.0;
    return sign | (uint16_t)(biased << 10) | (uint16_t)man;
}

/* Round a binary64 value to the nearest binary32 (ties to even), via the C
 * cast, which IEEE hosts implement as round-to-nearest-even. */
static float f64_to_f32(double x) { return (float)x; }

/* ------------------------------------------------------------------------ */
/* Walsh-Hadamard matrix, Sylvester order.                                   */
/* [TQ] "Kernel 3: Fused Hadamard + Quantize": y = H x / sqrt(D), computed   */
/* there by a range-based butterfly whose lower output is a+b and upper      */
/* output is b-a at each stride; that butterfly is the Sylvester matrix      */
/* H[i][j] = (-1)^popcount(i & j).                                           */
/* ------------------------------------------------------------------------ */

static int popcount_u32(unsigned v)
{
    int c = 0;
    while (v) { c += v & 1u; v >>= 1; }
    return c;
}

void oracle_hadamard_matrix(int D, double *H)
{
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j)
            H[(long)i * D + j] = (popcount_u32((unsigned)(i & j)) & 1) ? -1.0 : 1.0;
}

/*
 * The rotation of the randomised-sign variant.  [TQ] "Kernel 3: Fused
 * Hadamard + Quantize" states TurboQuantMSE's rotation as diag * H * x /
 * sqrt(D); its kernel listing multiplies each loaded x by diag before the
 * butterfly, i.e. computes H diag(s) x / sqrt(D).  Reading: the listing's
 * order, R = H diag(s) (column j of H scaled by s_j), with s_j = -1 when bit
 * j of signs[j / 32] is set.  signs NULL gives R = H.  R / sqrt(D) is
 * orthogonal; its inverse is R^T / sqrt(D) = diag(s) H / sqrt(D).
 */
static void rotation_matrix(int D, const uint32_t *signs, double *R)
{
    oracle_hadamard_matrix(D, R);
    if (!signs) return;
    for (int j = 0; j < D; ++j) {
        if ((signs[j / 32] >> (j % 32)) & 1u)
            for (int i = 0; i < D; ++i) R[(long)i * D + j] = -R[(long)i * D + j];
    }
}

/* ------------------------------------------------------------------------ */
/* Codebooks.                                                                */
/* [RVQ] "The pipeline, as it actually runs": stage 1 quantizes against a     */
/* Gaussian codebook, stage 2 quantizes the residual against a               */
/* Laplacian-fit codebook.  Both are 2^b-level scalar codebooks.             */
/* Reading (the pages give no procedure): stage 1 is the Lloyd-Max quantizer */
/* for N(0, 1/D); stage 2 is the Lloyd-Max quantizer for Laplace(0, beta)    */
/* where beta = E|r| (the Laplace maximum-likelihood scale) of the stage-1   */
/* residual r under N(0, 1/D).  Both densities are symmetric, so both        */
/* quantizers are computed on the positive half and mirrored.                */
/* ------------------------------------------------------------------------ */

static double std_pdf(double z) { return exp(-0.5 * z * z) / sqrt(2.0 * M_PI); }

/* P(a < Z <= b) for a standard normal Z, accurate in the tails. */
static double std_prob(double a, double b)
{
    if (a >= 0.0) return 0.5 * (erfc(a / M_SQRT2) - erfc(b / M_SQRT2));
    if (b <= 0.0) return 0.5 * (erfc(-b / M_SQRT2) - erfc(-a / M_SQRT2));
    return 1.0 - 0.5 * erfc(-a / M_SQRT2) - 0.5 * erfc(b / M_SQRT2);
}

/* E[Y | a < Y <= b] for Y ~ N(0, sigma^2): sigma (pdf(a') - pdf(b')) / P. */
static double gauss_cond_mean(double a, double b, double sigma)
{
    double za = a / sigma, zb = b / sigma;
    double pa = isinf(za) ? 0.0 : std_pdf(za);
    double pb = isinf(zb) ? 0.0 : std_pdf(zb);
    return sigma * (pa - pb) / std_prob(za, zb);
}

/* E[X | a < X <= b] for X ~ Laplace(0, beta), 0 <= a < b <= inf.  On the
 * positive half the density is exponential with mean beta. */
static double laplace_cond_mean(double a, double b, double beta)
{
    if (isinf(b)) return a + beta;
    double ea = exp(-a / beta), eb = exp(-b / beta);
    return beta + (a * ea - b * eb) / (ea - eb);
}

/*
 * Lloyd-Max iteration for a symmetric density.  `levels` is even.  The
 * positive half holds m = levels/2 centroids c[0..m-1] (ascending) with
 * boundaries 0 = t_0 < t_1 < ... < t_{m-1} < t_m = inf, where t_k is the
 * midpoint of c[k-1] and c[k] (nearest-neighbour condition) and each c[k] is
 * the conditional mean of its cell (centroid condition).  Iterates until no
 * centroid moves by more than tol.  kind 0 = Gaussian(sigma), 1 = Laplace(beta).
 * Returns the number of iterations used, or -1 without convergence.
 */
static int lloyd_max_positive_half(int levels, int kind, double scale, double *c_half,
                                   int max_iter, double tol)
{
    int m = levels / 2;
    /* Start from equally spaced points on (0, 3*scale). */
    for (int k = 0; k < m; ++k) c_half[k] = scale * 3.0 * (k + 0.5) / m;
    for (int it = 1; it <= max_iter; ++it) {
        double moved = 0.0;
        for (int k = 0; k < m; ++k) {
            double lo = (k == 0) ? 0.0 : 0.5 * (c_half[k - 1] + c_half[k]);
            double hi = (k == m - 1) ? INFINITY : 0.5 * (c_half[k] + c_half[k + 1]);
            double cn = (kind == 0) ? gauss_cond_mean(lo, hi, scale)
                                    : laplace_cond_mean(lo, hi, scale);
            double d = fabs(cn - c_half[k]);
            if (d > moved) moved = d;
            c_half[k] = cn;
        }
        if (moved <= tol) return it;
    }
    return -1;
}

/* Full symmetric codebook, ascending: c[0..levels-1], c[levels-1-k] = -c[k]. */
static int lloyd_max_full(int levels, int kind, double scale, double *c)
{
    double half[64];
    int it = lloyd_max_positive_half(levels, kind, scale, half, 1000000, 1e-15 * scale);
    int m = levels / 2;
    for (int k = 0; k < m; ++k) {
        c[m + k] = half[k];
        c[m - 1 - k] = -half[k];
    }
    return it;
}

/* Exported for the pins: Lloyd-Max centroids (ascending) for N(0, sigma^2). */
int oracle_lloyd_max_gaussian(int levels, double sigma, double *c)
{
    return lloyd_max_full(levels, 0, sigma, c);
}

/* Exported for the pins: Lloyd-Max centroids (ascending) for Laplace(0, beta). */
int oracle_lloyd_max_laplace(int levels, double beta, double *c)
{
    return lloyd_max_full(levels, 1, beta, c);
}

/*
 * beta = E|Y - c[i(Y)]| for Y ~ N(0, sigma^2), where i(Y) is the cell of Y in
 * the quantizer with ascending centroids c[] and midpoint boundaries.  Each
 * cell (lo, hi] is split at its centroid; on each piece |y - c| has one sign
 * and the integral of (y - c) phi_sigma(y) over (u, v] is
 * sigma^2 (phi_sigma(u) - phi_sigma(v)) - c P(u < Y <= v).
 */
double oracle_stage1_residual_mean_abs(int levels, const double *c, double sigma)
{
    double total = 0.0;
    for (int k = 0; k < levels; ++k) {
        double lo = (k == 0) ? -INFINITY : 0.5 * (c[k - 1] + c[k]);
        double hi = (k == levels - 1) ? INFINITY : 0.5 * (c[k] + c[k + 1]);
        double ck = c[k];
        /* integral over (ck, hi] of (y - ck) phi */
        double zc = ck / sigma, zh = hi / sigma, zl = lo / sigma;
        double pc = std_pdf(zc);
        double ph = isinf(zh) ? 0.0 : std_pdf(zh);
        double pl = isinf(zl) ? 0.0 : std_pdf(zl);
        /* sigma^2 * phi_sigma(y) = sigma * std_pdf(y/sigma) */
        double upper = sigma * (pc - ph) - ck * std_prob(zc, zh);
        /* integral over (lo, ck] of (ck - y) phi */
        double lower = ck * std_prob(zl, zc) - sigma * (pl - pc);
        total += upper + lower;
    }
    return total;
}

/*
 * The two RVQ codebooks for head dimension D and b bits per stage:
 *   c1[2^b], b1[2^b - 1]: stage 1, Lloyd-Max for N(0, 1/D);
 *   c2[2^b], b2[2^b - 1]: stage 2, Lloyd-Max for Laplace(0, beta), beta = E|r|.
 * Boundaries are the midpoints of adjacent centroids ([RVQ] "What 'quantize'
 * means here, precisely"), formed in binary64 from the binary64 centroids and
 * then rounded to binary32; centroids are rounded to binary32.
 */
int oracle_rvq_codebooks(int D, int bits, float *c1, float *b1, float *c2, float *b2,
                         double *beta_out)
{
    int L = 1 << bits;
    double g[64], l[64];
    double sigma = 1.0 / sqrt((double)D);
    if (oracle_lloyd_max_gaussian(L, sigma, g) < 0) return -1;
    double beta = oracle_stage1_residual_mean_abs(L, g, sigma);
    if (oracle_lloyd_max_laplace(L, beta, l) < 0) return -2;
    for (int k = 0; k < L; ++k) {
        c1[k] = f64_to_f32(g[k]);
        c2[k] = f64_to_f32(l[k]);
    }
    for (int k = 0; k + 1 < L; ++k) {
        b1[k] = f64_to_f32(0.5 * (g[k] + g[k + 1]));
        b2[k] = f64_to_f32(0.5 * (l[k] + l[k + 1]));
    }
    if (beta_out) *beta_out = beta;
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Bit packing.                                                              */
/* [RVQ] "The kernel" and [TQ] "Kernel 1: Bit-Packing": b-bit codes, LSB     */
/* first: element i of a run goes to word i / E at shift (i mod E) * b with  */
/* E = floor(32/b) codes per word (b = 3: 10 codes, the top 2 bits zero).    */
/* ------------------------------------------------------------------------ */

void oracle_pack_lsb_first(const uint8_t *codes, long n, int bits, uint32_t *words)
{
    int per_word = 32 / bits;
    uint32_t mask = (1u << bits) - 1u;
    long n_words = (n + per_word - 1) / per_word;
    for (long w = 0; w < n_words; ++w) words[w] = 0;
    for (long i = 0; i < n; ++i)
        words[i / per_word] |= ((uint32_t)codes[i] & mask) << ((i % per_word) * bits);
}

void oracle_unpack_lsb_first(const uint32_t *words, long n, int bits, uint8_t *codes)
{
    int per_word = 32 / bits;
    uint32_t mask = (1u << bits) - 1u;
    for (long i = 0; i < n; ++i)
        codes[i] = (uint8_t)((words[i / per_word] >> ((i % per_word) * bits)) & mask);
}

/* ------------------------------------------------------------------------ */
/* TurboQuantRVQ encode.                                                     */
/* [RVQ] "The pipeline, as it actually runs" and "What 'quantize' means      */
/* here, precisely": for each key row x (D values):                          */
/*   n = ||x||_2 (kept as the row norm), u = x / n                           */
/*   y = R u / sqrt(D)                        (rotate; R = H, or H diag(s)    */
/*                                             for the randomised signs)     */
/*   i1 = #{k : y > b1_k}                     (stage-1 boundary count)       */
/*   r = y - c1[i1]                           (dequantize1, residual)        */
/*   i2 = #{k : r > b2_k}                     (stage-2 boundary count)       */
/* then both index streams are bit-packed separately.                        */
/* Reading: a zero row (n == 0) has u = 0.                                   */
/* Tie flags: a code is flagged when its pre-quantization value is within    */
/* 1e-5 of a boundary; a stage-1 flag also flags the stage-2 code, whose     */
/* input depends on i1.                                                      */
/* ------------------------------------------------------------------------ */

#define RVQ_TIE_BAND 1e-5

void oracle_rvq_encode(const uint16_t *x_f16, long N, int D, int bits,
                       const float *c1, const float *b1, const float *c2, const float *b2,
                       uint8_t *idx1, uint8_t *idx2, uint32_t *packed1, uint32_t *packed2,
                       float *norms, uint8_t *tie1, uint8_t *tie2, double *y_out, double *r_out,
                       const uint32_t *signs)
{
    int L = 1 << bits;
    int W = (D + 32 / bits - 1) / (32 / bits);  /* words per row: E = floor(32/b) codes each */
    double *H = (double *)malloc(sizeof(double) * D * D);
    double *x = (double *)malloc(sizeof(double) * D);
    double *u = (double *)malloc(sizeof(double) * D);
    uint8_t *q1 = (uint8_t *)malloc(D), *q2 = (uint8_t *)malloc(D);
    rotation_matrix(D, signs, H);
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (long row = 0; row < N; ++row) {
        const uint16_t *xr = x_f16 + row * D;
        double n2 = 0.0;
        for (int d = 0; d < D; ++d) {
            x[d] = oracle_f16_to_f64(xr[d]);
            n2 += x[d] * x[d];
        }
        double n = sqrt(n2);
        norms[row] = f64_to_f32(n);
        for (int d = 0; d < D; ++d) u[d] = (n == 0.0) ? 0.0 : x[d] / n;
        for (int i = 0; i < D; ++i) {
            double acc = 0.0;
            for (int j = 0; j < D; ++j) acc += H[(long)i * D + j] * u[j];
            double y = acc * inv_sqrt_d;
            int k1 = 0, t1 = 0;
            for (int k = 0; k < L - 1; ++k) {
                if (y > (double)b1[k]) k1++;
                if (fabs(y - (double)b1[k]) < RVQ_TIE_BAND) t1 = 1;
            }
            double r = y - (double)c1[k1];
            int k2 = 0, t2 = t1;
            for (int k = 0; k < L - 1; ++k) {
                if (r > (double)b2[k]) k2++;
                if (fabs(r - (double)b2[k]) < RVQ_TIE_BAND) t2 = 1;
            }
            q1[i] = (uint8_t)k1;
            q2[i] = (uint8_t)k2;
            if (idx1) idx1[row * D + i] = (uint8_t)k1;
            if (idx2) idx2[row * D + i] = (uint8_t)k2;
            if (tie1) tie1[row * D + i] = (uint8_t)t1;
            if (tie2) tie2[row * D + i] = (uint8_t)t2;
            if (y_out) y_out[row * D + i] = y;
            if (r_out) r_out[row * D + i] = r;
        }
        if (packed1) oracle_pack_lsb_first(q1, D, bits, packed1 + row * W);
        if (packed2) oracle_pack_lsb_first(q2, D, bits, packed2 + row * W);
    }
    free(H); free(x); free(u); free(q1); free(q2);
}

/*
 * TurboQuantRVQ unpack + dequant.  [TQ] "Kernel 5: Fused RVQ Decode + Attend"
 * decodes a key in the rotated domain as c1[i1] + c2[i2].  Reading: the flush
 * codec returns the original domain, so the rotation is undone (H / sqrt(D) is
 * symmetric and its own inverse) and the stored norm re-applied:
 *   x_hat = n * H (c1[i1] + c2[i2]) / sqrt(D), rounded to binary16,
 * and with the randomised signs the transpose of the encoder's rotation,
 *   x_hat = n * R^T (c1[i1] + c2[i2]) / sqrt(D),  R = H diag(s).
 */
void oracle_rvq_decode(const uint32_t *packed1, const uint32_t *packed2, const float *norms,
                       long N, int D, int bits, const float *c1, const float *c2,
                       uint16_t *out_f16, double *out_f64, const uint32_t *signs)
{
    int W = (D + 32 / bits - 1) / (32 / bits);
    double *H = (double *)malloc(sizeof(double) * D * D);
    double *yh = (double *)malloc(sizeof(double) * D);
    uint8_t *q1 = (uint8_t *)malloc(D), *q2 = (uint8_t *)malloc(D);
    rotation_matrix(D, signs, H);
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (long row = 0; row < N; ++row) {
        oracle_unpack_lsb_first(packed1 + row * W, D, bits, q1);
        oracle_unpack_lsb_first(packed2 + row * W, D, bits, q2);
        for (int i = 0; i < D; ++i) yh[i] = (double)c1[q1[i]] + (double)c2[q2[i]];
        double n = (double)norms[row];
        for (int j = 0; j < D; ++j) {
            double acc = 0.0;
            for (int i = 0; i < D; ++i) acc += H[(long)i * D + j] * yh[i];  /* R^T */
            double v = n * acc * inv_sqrt_d;
            if (out_f64) out_f64[row * D + j] = v;
            if (out_f16) out_f16[row * D + j] = oracle_f64_to_f16_rn(v);
        }
    }
    free(H); free(yh); free(q1); free(q2);
}

/*
 * Decode-time attention over a TurboQuantRVQ key cache.  [TQ] "Kernel 5:
 * Fused RVQ Decode + Attend": keys decoded on the fly from the two code
 * streams, online softmax, values accumulated, never materialising the keys.
 * Readings (the pages give the loop, not the interface): one query token per
 * (batch, query head); query head hq reads kv head hq / (Hq / Hkv)
 * (grouped-query attention); a key is the flush codec's decoded row
 *   k_s = n_s * R^T (c1[i1] + c2[i2]) / sqrt(D)      (original domain;
 *                                                     R = H or H diag(s))
 * values are fp16; only the first lens[b] tokens of a cache take part
 * (lens NULL: all S_cap); the weights are the exact softmax of
 * scale * (q . k_s); an empty cache gives zeros.  Binary64 throughout, the
 * output rounded once to binary16.
 *
 * q [B, Hq, D] fp16; packed1/2 [B, Hkv, S_cap, D*b/32]; norms [B, Hkv, S_cap];
 * v [B, Hkv, S_cap, D] fp16; out [B, Hq, D].
 */
void oracle_rvq_attend(const uint16_t *q_f16, const uint32_t *packed1, const uint32_t *packed2,
                       const float *norms, const uint16_t *v_f16, const int32_t *lens, int B,
                       int Hq, int Hkv, int S_cap, int D, int bits, const float *c1,
                       const float *c2, double scale, uint16_t *out_f16, double *out_f64,
                       const uint32_t *signs)
{
    int W = (D + 32 / bits - 1) / (32 / bits), G = Hq / Hkv;
    double *H = (double *)malloc(sizeof(double) * D * D);
    double *K = (double *)malloc(sizeof(double) * (size_t)S_cap * D);
    double *yh = (double *)malloc(sizeof(double) * D);
    double *sc = (double *)malloc(sizeof(double) * (S_cap > 0 ? S_cap : 1));
    double *acc = (double *)malloc(sizeof(double) * D);
    uint8_t *q1 = (uint8_t *)malloc(D), *q2 = (uint8_t *)malloc(D);
    rotation_matrix(D, signs, H);
    double inv_sqrt_d = 1.0 / sqrt((double)D);
    for (int b = 0; b < B; ++b) {
        int len = lens ? lens[b] : S_cap;
        if (len > S_cap) len = S_cap;
        if (len < 0) len = 0;
        for (int h = 0; h < Hkv; ++h) {
            long base = ((long)b * Hkv + h) * S_cap;
            for (int s = 0; s < len; ++s) {
                oracle_unpack_lsb_first(packed1 + (base + s) * W, D, bits, q1);
                oracle_unpack_lsb_first(packed2 + (base + s) * W, D, bits, q2);
                for (int i = 0; i < D; ++i) yh[i] = (double)c1[q1[i]] + (double)c2[q2[i]];
                double n = (double)norms[base + s];
                for (int j = 0; j < D; ++j) {
                    double a = 0.0;
                    for (int i = 0; i < D; ++i) a += H[(long)i * D + j] * yh[i];  /* R^T */
                    K[(long)s * D + j] = n * a * inv_sqrt_d;
                }
            }
            for (int g = 0; g < G; ++g) {
                long qo = ((long)b * Hq + (long)h * G + g) * D;
                double m = -INFINITY;
                for (int s = 0; s < len; ++s) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += oracle_f16_to_f64(q_f16[qo + d]) * K[(long)s * D + d];
                    sc[s] = scale * dot;
                    if (sc[s] > m) m = sc[s];
                }
                double l = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int s = 0; s < len; ++s) {
                    double w = exp(sc[s] - m);
                    l += w;
                    for (int d = 0; d < D; ++d) acc[d] += w * oracle_f16_to_f64(v_f16[(base + s) * D + d]);
                }
                for (int d = 0; d < D; ++d) {
                    double o = len > 0 ? acc[d] / l : 0.0;
                    if (out_f64) out_f64[qo + d] = o;
                    if (out_f16) out_f16[qo + d] = oracle_f64_to_f16_rn(o);
                }
            }
        }
    }
    free(H); free(K); free(yh); free(sc); free(acc); free(q1); free(q2);
}

/* ------------------------------------------------------------------------ */
/* KIVI asymmetric min/max group quantization.                               */
/* [KIVI] first post, "What we're actually optimizing" and second post,      */
/* "What KIVI is": per group, zero = min, scale = (max - min)/(2^b - 1),     */
/* q = round((x - zero)/scale), recon = q*scale + zero.                      */
/* Keys are grouped per channel (a group is G consecutive tokens of one      */
/* channel); values per token (a group is G consecutive channels of one      */
/* token).  Only tokens [0, S_q) are quantized; the most recent              */
/* residual_length tokens stay fp16 and are not touched.                     */
/* Rounding is half to even ([KIVI] "Rounding mode").  Ragged token groups   */
/* are padded with the edge value ([KIVI] "Padding semantics"), which is a   */
/* member of the group already, so min and max are those of the real         */
/* members.                                                                  */
/* Readings: t = (x - min)(2^b - 1)/(max - min) is formed exactly (the       */
/* numerator and denominator are exact in binary64, one rounding in the      */
/* division); a constant group has q = 0 and scale 0; the stored scale is    */
/* fp16(fp32((max - min)/(2^b - 1))) with both roundings to nearest even;    */
/* the stored zero is the group minimum (exact in fp16).                     */
/* Tie flag: |t - (k + 1/2)| < 1e-4 for some integer k.                      */
/* ------------------------------------------------------------------------ */

#define KIVI_TIE_BAND 1e-4

/* fp32 round-to-nearest-even of the exact quotient num/den, where num and den
 * are exact binary64 values and den is a small positive integer. */
static float rn32_of_quotient(double num, double den)
{
    double q = num / den;           /* correctly rounded binary64 quotient */
    float f = f64_to_f32(q);
    /* q can only differ in its fp32 rounding from the exact quotient when q is
     * exactly halfway between two binary32 numbers; decide that case with the
     * exact remainder num - q*den (exact via fma). */
    float other = (double)f > q ? nextafterf(f, -INFINITY) : nextafterf(f, INFINITY);
    double mid = 0.5 * ((double)f + (double)other);
    if (q == mid) {
        double rem = fma(-q, den, num); /* sign of exact quotient - q */
        if (rem > 0.0) return (double)f > (double)other ? f : other;
        if (rem < 0.0) return (double)f < (double)other ? f : other;
    }
    return f;
}

static void kivi_group(const double *vals, int n, int bits, uint8_t *q, uint8_t *tie,
                       uint16_t *scale_h, uint16_t *zero_h)
{
    double levels = (double)((1 << bits) - 1);
    double mn = vals[0], mx = vals[0];
    for (int i = 1; i < n; ++i) {
        if (vals[i] < mn) mn = vals[i];
        if (vals[i] > mx) mx = vals[i];
    }
    *zero_h = oracle_f64_to_f16_rn(mn);
    if (mx == mn) {
        *scale_h = 0;
        for (int i = 0; i < n; ++i) { q[i] = 0; tie[i] = 0; }
        return;
    }
    *scale_h = oracle_f64_to_f16_rn((double)rn32_of_quotient(mx - mn, levels));
    for (int i = 0; i < n; ++i) {
        double t = ((vals[i] - mn) * levels) / (mx - mn);
        double r = nearbyint(t); /* default rounding mode: to nearest, ties to even */
        if (r < 0.0) r = 0.0;
        if (r > levels) r = levels;
        q[i] = (uint8_t)r;
        double f = t - floor(t);
        tie[i] = fabs(f - 0.5) < KIVI_TIE_BAND ? 1 : 0;
    }
}

/*
 * x: [BH, S, D] fp16 bits.  Quantizes tokens [0, S_q).
 * per_channel = 1 (keys): groups of G tokens per channel; NG = ceil(S_q/G);
 *   codes[bh][s][d]; scale/zero[bh][g][d];
 *   packed[((bh*NG + g)*(G*b/32) + w)*D + d] holds tokens g*G + w*(32/b) + j
 *   at shift j*b (slots past S_q hold 0).
 * per_channel = 0 (values): groups of G channels per token;
 *   codes[bh][s][d]; scale/zero[bh][s][d/G];
 *   packed[(bh*S_q + s)*(D*b/32) + d/(32/b)] at shift (d mod 32/b)*b.
 */
void oracle_kivi_quant(const uint16_t *x_f16, long BH, int S, int D, int bits, int G, int S_q,
                       int per_channel, uint8_t *codes, uint16_t *scale_h, uint16_t *zero_h,
                       uint32_t *packed, uint8_t *tie)
{
    double vals[1024];
    uint8_t q[1024], t[1024];
    int per_word = 32 / bits;
    if (per_channel) {
        int NG = (S_q + G - 1) / G;
        int wpg = G * bits / 32;
        for (long bh = 0; bh < BH; ++bh)
            for (int g = 0; g < NG; ++g)
                for (int d = 0; d < D; ++d) {
                    int s0 = g * G, s1 = s0 + G < S_q ? s0 + G : S_q;
                    int n = s1 - s0;
                    for (int i = 0; i < n; ++i)
                        vals[i] = oracle_f16_to_f64(x_f16[(bh * S + s0 + i) * D + d]);
                    uint16_t sc, ze;
                    kivi_group(vals, n, bits, q, t, &sc, &ze);
                    long gi = bh * NG + g;
                    scale_h[gi * D + d] = sc;
                    zero_h[gi * D + d] = ze;
                    for (int w = 0; w < wpg; ++w) {
                        uint32_t word = 0;
                        for (int j = 0; j < per_word; ++j) {
                            int i = w * per_word + j;
                            if (i < n) word |= (uint32_t)q[i] << (j * bits);
                        }
                        packed[(gi * wpg + w) * D + d] = word;
                    }
                    for (int i = 0; i < n; ++i) {
                        codes[(bh * S_q + s0 + i) * D + d] = q[i];
                        if (tie) tie[(bh * S_q + s0 + i) * D + d] = t[i];
                    }
                }
    } else {
        int NGD = D / G;
        int wpr = D * bits / 32;
        for (long bh = 0; bh < BH; ++bh)
            for (int s = 0; s < S_q; ++s) {
                long row = bh * S_q + s;
                uint8_t rowq[1024];
                for (int j = 0; j < NGD; ++j) {
                    for (int i = 0; i < G; ++i)
                        vals[i] = oracle_f16_to_f64(x_f16[(bh * S + s) * D + j * G + i]);
                    uint16_t sc, ze;
                    kivi_group(vals, G, bits, q, t, &sc, &ze);
                    scale_h[row * NGD + j] = sc;
                    zero_h[row * NGD + j] = ze;
                    for (int i = 0; i < G; ++i) {
                        rowq[j * G + i] = q[i];
                        codes[row * D + j * G + i] = q[i];
                        if (tie) tie[row * D + j * G + i] = t[i];
                    }
                }
                oracle_pack_lsb_first(rowq, D, bits, packed + row * wpr);
            }
    }
}

/*
 * KIVI dequant: x_hat = q * scale + zero with the stored fp16 scale and zero,
 * evaluated exactly in binary64 and rounded once to binary16 ([KIVI] first
 * post, "FMA contraction": the product and the sum; here the product is exact,
 * so contraction cannot change the result).  Output [BH, S_q, D] fp16 bits.
 * Layouts as in oracle_kivi_quant.
 */
void oracle_kivi_dequant(const uint32_t *packed, const uint16_t *scale_h, const uint16_t *zero_h,
                         long BH, int S_q, int D, int bits, int G, int per_channel,
                         uint16_t *out_f16)
{
    int per_word = 32 / bits;
    uint32_t mask = (1u << bits) - 1u;
    if (per_channel) {
        int NG = (S_q + G - 1) / G;
        int wpg = G * bits / 32;
        for (long bh = 0; bh < BH; ++bh)
            for (int s = 0; s < S_q; ++s)
                for (int d = 0; d < D; ++d) {
                    int g = s / G, i = s % G;
                    long gi = bh * NG + g;
                    uint32_t word = packed[(gi * wpg + i / per_word) * D + d];
                    uint32_t q = (word >> ((i % per_word) * bits)) & mask;
                    double v = (double)q * oracle_f16_to_f64(scale_h[gi * D + d]) +
                               oracle_f16_to_f64(zero_h[gi * D + d]);
                    out_f16[(bh * S_q + s) * D + d] = oracle_f64_to_f16_rn(v);
                }
    } else {
        int NGD = D / G;
        int wpr = D * bits / 32;
        for (long bh = 0; bh < BH; ++bh)
            for (int s = 0; s < S_q; ++s) {
                long row = bh * S_q + s;
                for (int d = 0; d < D; ++d) {
                    uint32_t word = packed[row * wpr + d / per_word];
                    uint32_t q = (word >> ((d % per_word) * bits)) & mask;
                    double v = (double)q * oracle_f16_to_f64(scale_h[row * NGD + d / G]) +
                               oracle_f16_to_f64(zero_h[row * NGD + d / G]);
                    out_f16[row * D + d] = oracle_f64_to_f16_rn(v);
                }
            }
    }
}

/*
 * Decode-time attention over a KIVI cache with dequantization inside the
 * attention ([KIVI] first post, closing section: "Dequant-in-SDPA - teach
 * attention to read packed codes directly, so expansion happens in registers
 * and never in RAM"; the reconstruction is the quantizer's g_hat = q * scale
 * + zero, [KIVI] second post, "What KIVI is").  Readings: keys and values are
 * reconstructed exactly (binary64, no fp16 rounding of the expansion); the
 * cache of sequence b is its first lens[b] quantized tokens (lens NULL: all
 * S_cap) followed by the first res_lens[b] tokens of the fp16 residual window
 * (res_lens NULL: all R), the window holding the most recent tokens ([KIVI]
 * second post: "KIVI holds the last R tokens in fp16"); one query token per
 * (batch, query head), query head hq reads kv head hq / (Hq / Hkv); exact
 * softmax of scale * (q . k); an empty cache gives zeros.
 *
 * Layouts: the flush's (oracle_kivi_quant) with S_cap tokens per (b, h):
 *   k_packed [B*Hkv, NG, G*b/32, D] (NG = S_cap / G), k_scale/k_zero [B*Hkv, NG, D];
 *   v_packed [B*Hkv, S_cap, D*b/32], v_scale/v_zero [B*Hkv, S_cap, D/G];
 *   k_res, v_res [B*Hkv, R, D] fp16; q [B, Hq, D]; out [B, Hq, D].
 */
void oracle_kivi_attend(const uint16_t *q_f16, const uint32_t *k_packed, const uint16_t *k_scale,
                        const uint16_t *k_zero, const uint32_t *v_packed, const uint16_t *v_scale,
                        const uint16_t *v_zero, const uint16_t *k_res, const uint16_t *v_res,
                        const int32_t *lens, const int32_t *res_lens, int B, int Hq, int Hkv,
                        int S_cap, int R, int D, int bits, int G, double scale, uint16_t *out_f16,
                        double *out_f64)
{
    int per_word = 32 / bits, NG = S_cap / G, wpg = G * bits / 32, wpr = D * bits / 32;
    uint32_t mask = (1u << bits) - 1u;
    int GQ = Hq / Hkv, T = S_cap + R;
    double *K = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    double *V = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * D);
    double *sc = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    double *acc = (double *)malloc(sizeof(double) * D);
    for (int b = 0; b < B; ++b) {
        int L = lens ? lens[b] : S_cap;
        if (L > S_cap) L = S_cap;
        if (L < 0) L = 0;
        int Lr = res_lens ? res_lens[b] : R;
        if (Lr > R) Lr = R;
        if (Lr < 0) Lr = 0;
        for (int h = 0; h < Hkv; ++h) {
            long bh = (long)b * Hkv + h;
            for (int s = 0; s < L; ++s) {
                int g = s / G, i = s % G;
                long gi = bh * NG + g;
                long row = bh * S_cap + s;
                for (int d = 0; d < D; ++d) {
                    uint32_t kw = k_packed[(gi * wpg + i / per_word) * D + d];
                    uint32_t kq = (kw >> ((i % per_word) * bits)) & mask;
                    K[(long)s * D + d] = (double)kq * oracle_f16_to_f64(k_scale[gi * D + d]) +
                                         oracle_f16_to_f64(k_zero[gi * D + d]);
                    uint32_t vw = v_packed[row * wpr + d / per_word];
                    uint32_t vq = (vw >> ((d % per_word) * bits)) & mask;
                    V[(long)s * D + d] = (double)vq * oracle_f16_to_f64(v_scale[row * (D / G) + d / G]) +
                                         oracle_f16_to_f64(v_zero[row * (D / G) + d / G]);
                }
            }
            for (int r = 0; r < Lr; ++r)
                for (int d = 0; d < D; ++d) {
                    K[(long)(L + r) * D + d] = oracle_f16_to_f64(k_res[(bh * R + r) * D + d]);
                    V[(long)(L + r) * D + d] = oracle_f16_to_f64(v_res[(bh * R + r) * D + d]);
                }
            int n = L + Lr;
            for (int gq = 0; gq < GQ; ++gq) {
                long qo = ((long)b * Hq + (long)h * GQ + gq) * D;
                double m = -INFINITY;
                for (int s = 0; s < n; ++s) {
                    double dot = 0.0;
                    for (int d = 0; d < D; ++d) dot += oracle_f16_to_f64(q_f16[qo + d]) * K[(long)s * D + d];
                    sc[s] = scale * dot;
                    if (sc[s] > m) m = sc[s];
                }
                double l = 0.0;
                for (int d = 0; d < D; ++d) acc[d] = 0.0;
                for (int s = 0; s < n; ++s) {
                    double w = exp(sc[s] - m);
                    l += w;
                    for (int d = 0; d < D; ++d) acc[d] += w * V[(long)s * D + d];
                }
                for (int d = 0; d < D; ++d) {
                    double o = n > 0 ? acc[d] / l : 0.0;
                    if (out_f64) out_f64[qo + d] = o;
                    if (out_f16) out_f16[qo + d] = oracle_f64_to_f16_rn(o);
                }
            }
        }
    }
    free(K); free(V); free(sc); free(acc);
}

/* ------------------------------------------------------------------------ */
/* QJL encode.                                                               */
/* [TQ] "Kernel 4: QJL Encode - Simdgroup Sign Packing": for each key x the  */
/* m bits of sign(S x), a bit being 1 when the dot product with sketch row   */
/* j is >= 0, packed least-significant bit first (bit j of byte k is sketch  */
/* row 8k + j; on little-endian words, bit j of word w is row 32w + j), and  */
/* the key's Euclidean norm stored as fp16.                                  */
/* Readings: S is the caller's m x d sketch matrix in fp16 (the page reads   */
/* it as a buffer converted to float); m is a multiple of 32.                */
/* Every product of two fp16 values is a dyadic rational m1 m2 2^(e1+e2)     */
/* with |m1 m2| < 2^22 and e1 + e2 >= -48, so the dot product (and the sum  */
/* of squares) is accumulated exactly as a 128-bit integer in units of       */
/* 2^-48: the signs are exact.  tie flags a sketch bit whose |dot| is below  */
/* 1e-5 of sum |S_jd x_d|, norm_tie a norm within 1e-6 (relative) of an fp16 */
/* rounding boundary: the places where an fp32 evaluation may differ.       */
/* ------------------------------------------------------------------------ */

/* x (fp16 bits) as an integer multiple of 2^-24: x = mant * 2^-24 exactly. */
static __int128 f16_to_units24(uint16_t h)
{
    int sign = (h >> 15) & 1, e = (h >> 10) & 31;
    int64_t f = h & 1023;
    __int128 v;
    if (e == 0) v = f;                               /* subnormal: f * 2^-24 */
    else v = (__int128)(f | 1024) << (e - 1);        /* (1024 + f) 2^(e - 25) = ... * 2^-24 */
    return sign ? -v : v;
}

static double units48_to_f64(__int128 v)
{
    /* exact conversion of the high and low 64-bit halves, then one add */
    int neg = v < 0;
    unsigned __int128 u = neg ? (unsigned __int128)(-v) : (unsigned __int128)v;
    double hi = (double)(uint64_t)(u >> 64) * 18446744073709551616.0;
    double lo = (double)(uint64_t)u;
    double r = (hi + lo) * ldexp(1.0, -48);
    return neg ? -r : r;
}

void oracle_qjl_encode(const uint16_t *x_f16, long N, int d, const uint16_t *s_f16, int m,
                       uint32_t *packed, uint16_t *norms_f16, uint8_t *tie, uint8_t *norm_tie)
{
    int W = m / 32;
    for (long n = 0; n < N; ++n) {
        const uint16_t *x = x_f16 + n * d;
        for (int w = 0; w < W; ++w) packed[n * W + w] = 0;
        for (int j = 0; j < m; ++j) {
            const uint16_t *s = s_f16 + (long)j * d;
            __int128 dot = 0;
            double mag = 0.0;
            for (int k = 0; k < d; ++k) {
                dot += f16_to_units24(s[k]) * f16_to_units24(x[k]);
                mag += fabs(oracle_f16_to_f64(s[k]) * oracle_f16_to_f64(x[k]));
            }
            if (dot >= 0) packed[n * W + j / 32] |= 1u << (j % 32);
            if (tie) tie[n * m + j] = fabs(units48_to_f64(dot)) < 1e-5 * mag;
        }
        __int128 q = 0;
        for (int k = 0; k < d; ++k) {
            __int128 u = f16_to_units24(x[k]);
            q += u * u;
        }
        double nr = sqrt(units48_to_f64(q));
        norms_f16[n] = oracle_f64_to_f16_rn(nr);
        if (norm_tie)
            norm_tie[n] = oracle_f64_to_f16_rn(nr * (1.0 + 1e-6)) != oracle_f64_to_f16_rn(nr * (1.0 - 1e-6));
    }
}
