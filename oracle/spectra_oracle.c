/*
 * spectra_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow, fp64 CPU restatement of spectral transform coding of a
 * KV cache, written from the method's description so that the CUDA library
 * can be checked against it.  Only the tests, the smoke entry point and the
 * benchmark's CPU-baseline leg may load this file's shared object.  It shares
 * no code, header, table or constant with the CUDA library.
 *
 * Sources (page title, section):
 *   [SPECTRA]  "Sintesi Tecnica: SPECTRA" (gist.science 2608.07915),
 *              sections "Metodologia" and "La Pipeline di SPECTRA".
 *   [SPECTRA-abs] SPECTRA abstract (arxivdaily 2608.07915).
 *   [ABL]      "Technisch Overzicht: Ablatie, Statistische Inferentie en
 *              Validatie voor KV-Cache Compressie" (gist.science 2607.09683),
 *              section "Experimentele Opstelling".
 *
 * Every routine is a direct loop over its definition; nothing is blocked,
 * fused or reordered.  Where the pages leave a step open, the reading taken
 * is stated at the routine.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Gram matrix.  [SPECTRA] "Metodologia" item 3 weights the transform by the
 * activation second moment G = E[h^T h]; [ABL] calibrates a per-head basis
 * on representative tokens.  Reading: uncentred, averaged over the n
 * calibration vectors:  G[i][j] = (1/n) sum_t x[t][i] x[t][j].
 * x is row t at x + t*ldx, d contiguous components. */
void orc_gram(const double* x, long n, long ldx, int d, double* G)
{
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) {
            double s = 0.0;
            for (long t = 0; t < n; ++t)
                s += x[t * ldx + i] * x[t * ldx + j];
            G[i * d + j] = (n > 0) ? s / (double)n : 0.0;
        }
}

/* ------------------------------------------------------------------------ */
/* Eigenbasis of G.  [SPECTRA] "Metodologia" item 1 and pipeline phase 1: the
 * cache is rotated into a basis computed from its own statistics, where the
 * coordinates are uncorrelated and ordered by energy.  [ABL] "per-head
 * eigenbasis".  Computed here by the textbook serial cyclic Jacobi method
 * (row-by-row sweep over all pairs p<q), each rotation chosen to annihilate
 * a[p][q] with the small-angle root t = sgn(theta)/(|theta|+sqrt(theta^2+1)),
 * theta = (a_qq - a_pp)/(2 a_pq).
 *
 * Readings: eigenvalues sorted descending, equal values keep the lower
 * original index; each eigenvector's largest-magnitude component is made
 * positive, the lowest row index winning ties.
 *
 * Output: lam[c] and Q[i*d + c] (column c = eigenvector of channel c).
 * Returns the number of sweeps taken, or -1 if max_sweeps ran out. */
static double off_norm(const double* A, int d)
{
    double s = 0.0;
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j)
            if (i != j) s += A[i * d + j] * A[i * d + j];
    return sqrt(s);
}

static double fro_norm(const double* A, int d)
{
    double s = 0.0;
    for (int i = 0; i < d * d; ++i) s += A[i] * A[i];
    return sqrt(s);
}

int orc_jacobi(const double* G, int d, double tol, int max_sweeps,
               double* lam, double* Q)
{
    double* A = (double*)malloc(sizeof(double) * d * d);
    double* V = (double*)malloc(sizeof(double) * d * d);
    memcpy(A, G, sizeof(double) * d * d);
    for (int i = 0; i < d; ++i)
        for (int j = 0; j < d; ++j) V[i * d + j] = (i == j) ? 1.0 : 0.0;

    const double gf = fro_norm(A, d);
    int sweeps = 0, converged = 0;
    for (;;) {
        if (off_norm(A, d) <= tol * gf) { converged = 1; break; }
        if (sweeps >= max_sweeps) break;
        ++sweeps;
        for (int p = 0; p < d - 1; ++p)
            for (int q = p + 1; q < d; ++q) {
                const double apq = A[p * d + q];
                if (apq == 0.0) continue;
                const double theta = (A[q * d + q] - A[p * d + p]) / (2.0 * apq);
                const double t = (theta >= 0.0 ? 1.0 : -1.0) /
                                 (fabs(theta) + sqrt(theta * theta + 1.0));
                const double c = 1.0 / sqrt(t * t + 1.0);
                const double s = t * c;
                /* A <- A J  (columns p, q) */
                for (int k = 0; k < d; ++k) {
                    const double akp = A[k * d + p], akq = A[k * d + q];
                    A[k * d + p] = c * akp - s * akq;
                    A[k * d + q] = s * akp + c * akq;
                }
                /* A <- J^T A  (rows p, q) */
                for (int k = 0; k < d; ++k) {
                    const double apk = A[p * d + k], aqk = A[q * d + k];
                    A[p * d + k] = c * apk - s * aqk;
                    A[q * d + k] = s * apk + c * aqk;
                }
                /* V <- V J */
                for (int k = 0; k < d; ++k) {
                    const double vkp = V[k * d + p], vkq = V[k * d + q];
                    V[k * d + p] = c * vkp - s * vkq;
                    V[k * d + q] = s * vkp + c * vkq;
                }
            }
    }

    /* sort descending; ties keep the lower original index (stable) */
    int* order = (int*)malloc(sizeof(int) * d);
    for (int i = 0; i < d; ++i) order[i] = i;
    for (int i = 1; i < d; ++i) {           /* insertion sort: stable */
        int o = order[i], j = i - 1;
        while (j >= 0 && A[order[j] * d + order[j]] < A[o * d + o]) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = o;
    }
    for (int c = 0; c < d; ++c) {
        const int src = order[c];
        lam[c] = A[src * d + src];
        for (int i = 0; i < d; ++i) Q[i * d + c] = V[i * d + src];
        /* sign: largest |component| positive, lowest row on ties */
        int imax = 0;
        for (int i = 1; i < d; ++i)
            if (fabs(Q[i * d + c]) > fabs(Q[imax * d + c])) imax = i;
        if (Q[imax * d + c] < 0.0)
            for (int i = 0; i < d; ++i) Q[i * d + c] = -Q[i * d + c];
    }
    free(order);
    free(A);
    free(V);
    return converged ? sweeps : -1;
}

/* ------------------------------------------------------------------------ */
/* Bit allocation.  [SPECTRA] pipeline phase 2: reverse water-filling gives
 * more bits to high-variance latent coordinates and fewer, down to zero, to
 * low-variance ones, from their measured marginal variances; [SPECTRA]
 * "Metodologia" item 2: zero-bit channels are dropped.
 *
 * Reading: integer widths 0..8 under the high-rate model D_c(b) = lam_c 4^-b;
 * R_tot one-bit increments, each to the channel with the largest current
 * lam_c * 4^-b_c among channels below 8 bits, lowest channel index on ties.
 * Negative eigenvalues (round-off) count as 0.  Returns sum of bits. */
long orc_alloc(const double* lam, int d, long R_tot, uint8_t* bits)
{
    for (int c = 0; c < d; ++c) bits[c] = 0;
    long given = 0;
    for (long step = 0; step < R_tot; ++step) {
        int best = -1;
        double bv = -1.0;
        for (int c = 0; c < d; ++c) {
            if (bits[c] >= 8) continue;
            const double l = lam[c] > 0.0 ? lam[c] : 0.0;
            const double v = ldexp(l, -2 * (int)bits[c]);   /* exact */
            if (v > bv) { bv = v; best = c; }
        }
        if (best < 0) break;
        bits[best] += 1;
        ++given;
    }
    return given;
}

/* ------------------------------------------------------------------------ */
/* Grouped reverse water-filling.  [SPECTRA] "La Pipeline di SPECTRA" phase 2,
 * "Raggruppamento": adjacent latent coordinates share one bit width, which
 * keeps the cache append-only and streamable; [ABL] "Regime-Specifieke
 * Prestaties": the effective dimension is pruned (the channels past it take
 * no bits).  Readings: groups of g consecutive channels in the eigenvalue-
 * descending order; only the first `keep` channels take part, in
 * floor(keep / g) whole groups, every other channel gets 0 bits; a one-bit
 * step of a group gives all its g channels one bit and costs g bits; the
 * greedy takes floor(R_tot / g) steps, each to the group with the largest
 * Lam_G * 4^-b_G among groups below 8 bits (Lam_G = the sum of the group's
 * eigenvalues clipped at 0, added in ascending channel order in fp64),
 * lowest group index on ties.  g = 1 with keep = d is orc_alloc.
 * Returns the bits given. */
long orc_alloc_grouped(const double* lam, int d, long R_tot, int g, int keep, uint8_t* bits)
{
    for (int c = 0; c < d; ++c) bits[c] = 0;
    if (g < 1 || keep < 0) return 0;
    if (keep > d) keep = d;
    const int ng = keep / g;
    double* Lam = (double*)malloc(sizeof(double) * (ng > 0 ? ng : 1));
    int* bg = (int*)calloc(ng > 0 ? ng : 1, sizeof(int));
    for (int G = 0; G < ng; ++G) {
        double s = 0.0;
        for (int c = G * g; c < (G + 1) * g; ++c) s += lam[c] > 0.0 ? lam[c] : 0.0;
        Lam[G] = s;
    }
    long given = 0;
    for (long step = 0; step < R_tot / g; ++step) {
        int best = -1;
        double bv = -1.0;
        for (int G = 0; G < ng; ++G) {
            if (bg[G] >= 8) continue;
            const double v = ldexp(Lam[G], -2 * bg[G]);
            if (v > bv) { bv = v; best = G; }
        }
        if (best < 0) break;
        bg[best] += 1;
        given += g;
    }
    for (int G = 0; G < ng; ++G)
        for (int c = G * g; c < (G + 1) * g; ++c) bits[c] = (uint8_t)bg[G];
    free(Lam);
    free(bg);
    return given;
}

/* ------------------------------------------------------------------------ */
/* Effective dimension with spectral-gap pruning.  [ABL] "Regime-Specifieke
 * Prestaties": d_eff follows the calibration budget rather than the true
 * rank, and a single spurious eigenvalue can make the output anti-correlated,
 * so a spectral-gap criterion prunes the estimated dimension.  The page gives
 * no formula; readings (eigenvalues descending, clipped at 0):
 *   d_energy = the smallest k with lam_0 + ... + lam_{k-1} >= energy * sum(lam)
 *              (0 when the sum is 0), sums in ascending order in fp64;
 *   d_gap    = the k in 1 .. min(d_energy, d - 1) with the largest ratio
 *              lam_{k-1} / lam_k (a zero lam_k is an infinite ratio), the
 *              smallest such k on ties, compared exactly as cross products;
 *              d_energy when d_energy is 0 or d is 1. */
void orc_effective_dim(const double* lam_in, int d, double energy, int* d_energy, int* d_gap)
{
    double tot = 0.0;
    for (int c = 0; c < d; ++c) tot += lam_in[c] > 0.0 ? lam_in[c] : 0.0;
    int de = 0;
    if (tot > 0.0) {
        double cum = 0.0;
        for (de = 0; de < d;) {
            cum += lam_in[de] > 0.0 ? lam_in[de] : 0.0;
            ++de;
            if (cum >= energy * tot) break;
        }
    }
    *d_energy = de;
    int best = de;
    if (de > 0 && d > 1) {
        const int kmax = de < d - 1 ? de : d - 1;
        best = 1;
        for (int k = 2; k <= kmax; ++k) {
            const double a = lam_in[k - 1] > 0.0 ? lam_in[k - 1] : 0.0, b = lam_in[k] > 0.0 ? lam_in[k] : 0.0;
            const double ab = lam_in[best - 1] > 0.0 ? lam_in[best - 1] : 0.0;
            const double bb = lam_in[best] > 0.0 ? lam_in[best] : 0.0;
            /* a / b > ab / bb  <=>  a * bb > ab * b  (b, bb >= 0) */
            if (a * bb > ab * b) best = k;
        }
    }
    *d_gap = best;
}

/* ------------------------------------------------------------------------ */
/* Gaussian Lloyd-Max codebook (the Lloyd-Max codebook family of [ABL]
 * "Experimentele Opstelling", here for N(0,1) as the workload asks).
 * Lloyd's alternation: thresholds at midpoints of adjacent levels; each level
 * moved to the centroid of its cell,
 *     E[X | a < X < b] = (phi(a) - phi(b)) / (Phi(b) - Phi(a)),
 * until no level moves by more than tol.  Start: levels at the quantiles
 * (k + 1/2)/L of N(0,1).  Levels are kept exactly antisymmetric.
 * Output: levels[0..L-1] ascending, thresh[1..L-1] (thresh[0] unused).
 * Returns iterations, or -1 if max_iter ran out. */
static double phi(double x) { return exp(-0.5 * x * x) / sqrt(2.0 * M_PI); }
/* upper tail Q(x) = P(X > x), accurate in both tails */
static double qtail(double x) { return 0.5 * erfc(x / sqrt(2.0)); }
/* P(a < X < b) without cancellation */
static double cell_mass(double a, double b)
{
    if (a >= 0.0) return qtail(a) - qtail(b);
    if (b <= 0.0) return qtail(-b) - qtail(-a);
    return 1.0 - qtail(b) - qtail(-a);
}
static double normal_quantile(double p)
{
    /* bisection on the cdf: slow and obviously correct */
    double lo = -40.0, hi = 40.0;
    for (int it = 0; it < 200; ++it) {
        const double mid = 0.5 * (lo + hi);
        if (1.0 - qtail(mid) < p) lo = mid; else hi = mid;
    }
    return 0.5 * (lo + hi);
}

long orc_lloyd_max(int b, double tol, long max_iter, double* levels, double* thresh)
{
    const int L = 1 << b, H = L / 2;
    for (int k = 0; k < L; ++k) levels[k] = normal_quantile((k + 0.5) / L);
    for (int k = 0; k < H; ++k) {               /* exact antisymmetry */
        const double a = 0.5 * (levels[L - 1 - k] - levels[k]);
        levels[k] = -a;
        levels[L - 1 - k] = a;
    }
    long it = 0;
    for (; it < max_iter; ++it) {
        for (int k = 1; k < L; ++k) thresh[k] = 0.5 * (levels[k - 1] + levels[k]);
        double moved = 0.0;
        /* positive half; the negative half mirrors it */
        for (int k = H; k < L; ++k) {
            const double a = thresh[k];
            const double bb = (k == L - 1) ? INFINITY : thresh[k + 1];
            const double pa = phi(a), pb = (k == L - 1) ? 0.0 : phi(bb);
            const double c = (pa - pb) / cell_mass(a, bb);
            moved = fmax(moved, fabs(c - levels[k]));
            levels[k] = c;
        }
        for (int k = 0; k < H; ++k) levels[k] = -levels[L - 1 - k];
        if (moved <= tol) { ++it; break; }
    }
    for (int k = 1; k < L; ++k) thresh[k] = 0.5 * (levels[k - 1] + levels[k]);
    thresh[0] = -INFINITY;
    return (it >= max_iter) ? -1 : it;
}

/* mean squared error of a codebook on N(0,1), by its cells (closed form
 * of the second moment per cell: int_a^b (x - l)^2 phi). */
double orc_codebook_mse(int L, const double* levels, const double* thresh)
{
    double mse = 0.0;
    for (int k = 0; k < L; ++k) {
        const double a = (k == 0) ? -INFINITY : thresh[k];
        const double b = (k == L - 1) ? INFINITY : thresh[k + 1];
        const double P = cell_mass(a, b);
        const double pa = isinf(a) ? 0.0 : phi(a), pb = isinf(b) ? 0.0 : phi(b);
        const double m1 = pa - pb;                                 /* int x phi   */
        const double xa = isinf(a) ? 0.0 : a * pa, xb = isinf(b) ? 0.0 : b * pb;
        const double m2 = P + xa - xb;                             /* int x^2 phi */
        const double l = levels[k];
        mse += m2 - 2.0 * l * m1 + l * l * P;
    }
    return mse;
}

/* ------------------------------------------------------------------------ */
/* Projection onto the latent basis and reconstruction.  [SPECTRA] pipeline
 * phase 3: tokens are projected down, quantized per token, appended to the
 * latent cache; full keys/values are rebuilt on the fly.
 *   y[t][c] = sum_i Q[i][c] x[t][i]              (project)
 *   xh[t][i] = sum_c Q[i][c] yh[t][c]             (reconstruct)        */
void orc_project(const double* x, long T, long ldx, int d, const double* Q, double* y)
{
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            double s = 0.0;
            for (int i = 0; i < d; ++i) s += Q[i * d + c] * x[t * ldx + i];
            y[t * d + c] = s;
        }
}

void orc_reconstruct(const double* yh, long T, int d, const double* Q, double* xh)
{
    for (long t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) {
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += Q[i * d + c] * yh[t * d + c];
            xh[t * d + i] = s;
        }
}

/* ------------------------------------------------------------------------ */
/* Randomized Walsh-Hadamard rotation ([ABL] "Experimentele Opstelling",
 * TurboQuant: a randomized WHT spreads token energy evenly).  Reading:
 * Sylvester Hadamard in natural order, H[i][j] = (-1)^popcount(i & j),
 * D = diag(signs):  y = (1/sqrt d) H D x,  and its inverse
 * x = (1/sqrt d) D H y  (H is symmetric and H H = d I).  Explicit matrix
 * products, no fast transform. */
static int hsign(int i, int j) { return (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1; }

void orc_rwht(const double* x, long T, long ldx, int d, const int8_t* signs, double* y)
{
    const double s = 1.0 / sqrt((double)d);
    for (long t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += hsign(i, j) * signs[j] * x[t * ldx + j];
            y[t * d + i] = s * acc;
        }
}

void orc_irwht(const double* y, long T, int d, const int8_t* signs, double* x)
{
    const double s = 1.0 / sqrt((double)d);
    for (long t = 0; t < T; ++t)
        for (int i = 0; i < d; ++i) {
            double acc = 0.0;
            for (int j = 0; j < d; ++j) acc += hsign(i, j) * y[t * d + j];
            x[t * d + i] = s * signs[i] * acc;
        }
}

/* ------------------------------------------------------------------------ */
/* Scalar quantizers (per channel, per token).
 * Uniform ([SPECTRA] pipeline phase 2 widths; "clipped at +-3 sigma_c"):
 *   sigma = sqrt(max(lam,0)), Delta = 6 sigma / 2^b,
 *   code = clamp(floor((y + 3 sigma)/Delta), 0, 2^b - 1),
 *   recon = -3 sigma + (code + 1/2) Delta.
 * Reading: midrise cells, a value on a boundary goes to the upper cell;
 * when sigma == 0 the value is treated as 0 (middle cell, recon 0). */
void orc_quant_uniform(const double* y, long T, int d, const double* lam,
                       const uint8_t* bits, int32_t* codes)
{
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            const int b = bits[c];
            if (b == 0) { codes[t * d + c] = 0; continue; }
            const double sig = sqrt(lam[c] > 0.0 ? lam[c] : 0.0);
            const double L = ldexp(1.0, b);
            double u;
            if (sig > 0.0) u = floor((y[t * d + c] + 3.0 * sig) / (6.0 * sig / L));
            else u = L / 2;
            if (u < 0) u = 0;
            if (u > L - 1) u = L - 1;
            codes[t * d + c] = (int32_t)u;
        }
}

void orc_dequant_uniform(const int32_t* codes, long T, int d, const double* lam,
                         const uint8_t* bits, double* yh)
{
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            const int b = bits[c];
            if (b == 0) { yh[t * d + c] = 0.0; continue; }
            const double sig = sqrt(lam[c] > 0.0 ? lam[c] : 0.0);
            const double delta = 6.0 * sig / ldexp(1.0, b);
            yh[t * d + c] = -3.0 * sig + (codes[t * d + c] + 0.5) * delta;
        }
}

/* Lloyd-Max: code = number of thresholds tau_k <= y/sigma (ties go up),
 * recon = sigma * level[code].  sigma per (token, channel) is given by
 * sig[t*sig_ts + c*sig_cs] (per channel: sig_ts = 0; per token: sig_cs = 0).
 * Reading: sigma == 0 treats y/sigma as 0.
 * tables: levels/thresh for width b at offset (b-1)*256. */
void orc_quant_lm(const double* y, long T, int d, const double* sig, long sig_ts, long sig_cs,
                  const uint8_t* bits, const double* thresh_tab, int32_t* codes)
{
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            const int b = bits[c];
            if (b == 0) { codes[t * d + c] = 0; continue; }
            const double s = sig[t * sig_ts + c * sig_cs];
            const double u = (s > 0.0) ? y[t * d + c] / s : 0.0;
            const double* th = thresh_tab + (b - 1) * 256;
            int code = 0;
            for (int k = 1; k < (1 << b); ++k)
                if (th[k] <= u) ++code;
            codes[t * d + c] = code;
        }
}

void orc_dequant_lm(const int32_t* codes, long T, int d, const double* sig, long sig_ts, long sig_cs,
                    const uint8_t* bits, const double* level_tab, double* yh)
{
    for (long t = 0; t < T; ++t)
        for (int c = 0; c < d; ++c) {
            const int b = bits[c];
            if (b == 0) { yh[t * d + c] = 0.0; continue; }
            yh[t * d + c] = sig[t * sig_ts + c * sig_cs] *
                            level_tab[(b - 1) * 256 + codes[t * d + c]];
        }
}

/* ------------------------------------------------------------------------ */
/* Packing.  [SPECTRA] pipeline phases 2-3 describe an append-only latent
 * cache of per-token quantized coordinates; the pages give no bit layout.
 * Reading (bit-plane groups): tokens are taken in groups of 32; with
 * R = sum_c bits[c] and o_c = sum_{c'<c} bits[c'], group g holds R 32-bit
 * little-endian words; bit (t mod 32) of word g*R + o_c + k is bit k of the
 * code of channel c of token t.  Written bit by bit. */
long orc_stream_bytes(long T, long R)
{
    const long groups = (T + 31) / 32;
    const long raw = groups * 4 * R;
    return (raw + 15) / 16 * 16;
}

void orc_pack(const int32_t* codes, long T, int d, const uint8_t* bits, uint8_t* stream)
{
    long R = 0;
    for (int c = 0; c < d; ++c) R += bits[c];
    memset(stream, 0, (size_t)orc_stream_bytes(T, R));
    for (long t = 0; t < T; ++t) {
        long off = 0;
        for (int c = 0; c < d; ++c) {
            for (int k = 0; k < bits[c]; ++k) {
                if ((codes[t * d + c] >> k) & 1) {
                    const long word = (t / 32) * R + off + k;
                    const long bitpos = word * 32 + (t % 32);
                    stream[bitpos / 8] |= (uint8_t)(1u << (bitpos % 8));
                }
            }
            off += bits[c];
        }
    }
}

void orc_unpack(const uint8_t* stream, long T, int d, const uint8_t* bits, int32_t* codes)
{
    long R = 0;
    for (int c = 0; c < d; ++c) R += bits[c];
    for (long t = 0; t < T; ++t) {
        long off = 0;
        for (int c = 0; c < d; ++c) {
            int32_t v = 0;
            for (int k = 0; k < bits[c]; ++k) {
                const long word = (t / 32) * R + off + k;
                const long bitpos = word * 32 + (t % 32);
                if ((stream[bitpos / 8] >> (bitpos % 8)) & 1) v |= (1 << k);
            }
            codes[t * d + c] = v;
            off += bits[c];
        }
    }
}

/* Append to a stream.  [SPECTRA] "La Pipeline di SPECTRA" phase 2
 * ("Raggruppamento": the latent cache stays append-only and streamable) and
 * phase 3 (each new token is projected, quantized and appended): the codes of
 * n tokens are written at stream positions t0 .. t0+n-1, each bit of theirs
 * set or cleared one by one, every other bit of the stream left as it was.
 * The stream must hold at least t0 + n tokens. */
void orc_pack_into(const int32_t* codes, long n, int d, const uint8_t* bits, long t0, uint8_t* stream)
{
    long R = 0;
    for (int c = 0; c < d; ++c) R += bits[c];
    for (long i = 0; i < n; ++i) {
        const long t = t0 + i;
        long off = 0;
        for (int c = 0; c < d; ++c) {
            for (int k = 0; k < bits[c]; ++k) {
                const long word = (t / 32) * R + off + k;
                const long bitpos = word * 32 + (t % 32);
                const uint8_t m = (uint8_t)(1u << (bitpos % 8));
                if ((codes[i * d + c] >> k) & 1) stream[bitpos / 8] |= m;
                else stream[bitpos / 8] &= (uint8_t)~m;
            }
            off += bits[c];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* 1-bit Johnson-Lindenstrauss sketch of the key residual.  [ABL]
 * "Experimentele Opstelling" and "Belangrijkste Bijdragen" 1 (TQ-QKV: a 1-bit
 * QJL residual sketch on the key path): with a Gaussian matrix S (m x d,
 * i.i.d. N(0,1) entries, supplied by the caller), a residual r is kept as the
 * m signs z_j = sign(<s_j, r>) and its norm; an inner product with it is
 * estimated as
 *     <q, r>  ~  sqrt(pi / 2) / m * ||r|| * sum_j <s_j, q> z_j,
 * unbiased because E[<s, q> sign(<s, r>)] = sqrt(2 / pi) <q, r> / ||r|| for
 * Gaussian s.  Reading: the residual is taken in the latent coordinates
 * (r = y - yhat, the rotation is orthonormal so inner products and norms are
 * those of k - khat), sign(0) = +1, bits b_j = (z_j > 0).
 * r[T][d] -> bits[T][m] (0/1), norms[T]. */
void orc_qjl_sketch(const double* r, long T, int d, const double* S, int m, uint8_t* bits, double* norms)
{
    for (long t = 0; t < T; ++t) {
        double n2 = 0.0;
        for (int i = 0; i < d; ++i) n2 += r[t * d + i] * r[t * d + i];
        norms[t] = sqrt(n2);
        for (int j = 0; j < m; ++j) {
            double a = 0.0;
            for (int i = 0; i < d; ++i) a += S[(long)j * d + i] * r[t * d + i];
            bits[t * m + j] = (uint8_t)(a >= 0.0);
        }
    }
}

/* The estimate of <q, r> from a sketch (definition above). */
double orc_qjl_estimate(const double* q, int d, const double* S, int m, const uint8_t* bits, double norm)
{
    double acc = 0.0;
    for (int j = 0; j < m; ++j) {
        double sq = 0.0;
        for (int i = 0; i < d; ++i) sq += S[(long)j * d + i] * q[i];
        acc += bits[j] ? sq : -sq;
    }
    return sqrt(M_PI / 2.0) / (double)m * norm * acc;
}

/* ------------------------------------------------------------------------ */
/* Decode-step attention over reconstructed keys/values (the standard
 * attention that [SPECTRA] pipeline phase 3 feeds with rebuilt K/V):
 *   s_t = scale * <q, k_t>,  p = softmax(s) (max subtracted),
 *   o = sum_t p_t v_t.   One query vector; K, V are [ctx][d]. */
void orc_attention(const double* q, const double* K, const double* V, long ctx, int d,
                   double scale, double* out)
{
    double* s = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    double m = -INFINITY;
    for (long t = 0; t < ctx; ++t) {
        double a = 0.0;
        for (int i = 0; i < d; ++i) a += q[i] * K[t * d + i];
        s[t] = scale * a;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (long t = 0; t < ctx; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
    for (int i = 0; i < d; ++i) {
        double a = 0.0;
        for (long t = 0; t < ctx; ++t) a += s[t] * V[t * d + i];
        out[i] = (ctx > 0) ? a / l : 0.0;
    }
    free(s);
}
