/*
 * locks_oracle.c - plain float64 CPU oracle of the LOCKS decode step.
 *
 * TEST INFRASTRUCTURE. Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never
 * does. It shares no code, header, table or constant with the CUDA library:
 * everything below is written out again from the LOCKS pages and from the
 * textbook definitions it names.
 *
 * Sources (the LOCKS pages):
 *   [p1] "LOCKS: per-page SVD cuts KV cache reads 10x at 1M context"
 *        (wps.hkprog.org), sections "How LOCKS works" (summary contents and
 *        the score formula), "Code" (the PyTorch sketch of build, score,
 *        top-k and attention) and "Caveats".
 *   [p4] gist.science technical summary of the LOCKS paper (arXiv 2607.24555),
 *        section 2 "Method": 2.1 page-local spectral decomposition
 *        (eigendecomposition of the centred keys; int4 basis, int8
 *        coefficients and centroid), 2.2 reconstruction and selection (the
 *        score formula, no K/V read), 2.3 group-shared selection for GQA.
 *
 * Every computation is float64, one unit at a time, in the order the
 * definitions state. OpenMP only splits independent units across threads.
 *
 * Summary byte layout (per unit = one (physical page, kv head)):
 *   mu    int8[128]   element d at 32*t + 4*s + 2*h + e,
 *                     where s = d/16, w = d%16, h = w/8, t = (w%8)/2, e = w%2
 *   basis uint8[512]  int4 two's complement, element (d, r) in byte
 *                     64*r + 16*t + 4*(s/2) + p/2, nibble p%2 (0 = low),
 *                     p = 2*(s%2) + h + 4*e  (s, w, h, t, e as for mu)
 *   coef  int8[128]   element (token i, rank r) at
 *                     4*(4*(i%8) + r/2) + 2*(i/8) + r%2
 *   scales fp16[4]    absmax scales of mu, basis, coef, then 0
 * Dequantised value = code * (fp16 scale as a real number).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define LO_PAGE 16
#define LO_D 128
#define LO_R 8
#define LO_UNIT_BYTES 776

int lo_version(void) { return 1; }

int lo_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void lo_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ---------------------------------------------------------------- numbers */

/* bfloat16 bits -> real: the upper 16 bits of an IEEE binary32. */
double lo_bf16_to_f64(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* IEEE binary16 bits -> real, from the format's definition. */
double lo_f16_to_f64(uint16_t h) {
    int sign = (h >> 15) & 1;
    int ex = (h >> 10) & 0x1f;
    int man = h & 0x3ff;
    double v;
    if (ex == 0) {
        v = ldexp((double)man, -24);                /* subnormal: man * 2^-24 */
    } else if (ex == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexp(1.0 + man / 1024.0, ex - 15);
    }
    return sign ? -v : v;
}

/* real -> IEEE binary16 bits, round to nearest, ties to even. */
uint16_t lo_f64_to_f16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7e00;
    double a = fabs(x);
    if (a >= 65520.0) return sign | 0x7c00;         /* rounds past 65504 */
    if (a == 0.0) return sign;
    int e;
    frexp(a, &e);                                   /* a = m 2^e, m in [0.5, 1) */
    int ue = e - 1;                                 /* a in [2^ue, 2^(ue+1)) */
    if (ue < -14) ue = -14;                         /* subnormal quantum 2^-24 */
    double quantum = ldexp(1.0, ue - 10);
    double r = nearbyint(a / quantum) * quantum;    /* exact division by 2^k */
    if (r == 0.0) return sign;
    frexp(r, &e);
    ue = e - 1;
    if (ue < -14) return sign | (uint16_t)(r / ldexp(1.0, -24));
    uint16_t exf = (uint16_t)(ue + 15);
    uint16_t man = (uint16_t)((r / ldexp(1.0, ue) - 1.0) * 1024.0);
    return sign | (uint16_t)(exf << 10) | man;
}

static double lo_f16_round(double x) { return lo_f16_to_f64(lo_f64_to_f16(x)); }

/* ------------------------------------------------------------- Jacobi eig */

/*
 * Cyclic Jacobi eigenvalue method for a symmetric n x n matrix (Golub & Van
 * Loan, "Matrix Computations", the cyclic Jacobi algorithm of section 8.5):
 * sweep the off-diagonal pairs (p, q) row by row; each step applies the
 * symmetric Schur rotation that zeroes a[p][q]. Stops when the off-diagonal
 * Frobenius norm is <= tol * ||A||_F. On exit a holds the eigenvalues on its
 * diagonal and the columns of v the eigenvectors. Returns the sweeps used.
 */
int lo_jacobi_eig(int n, double* a, double* v, double tol, int max_sweeps) {
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) v[i * n + j] = (i == j) ? 1.0 : 0.0;
    double fro = 0.0;
    for (int i = 0; i < n * n; ++i) fro += a[i] * a[i];
    fro = sqrt(fro);
    int sweep;
    for (sweep = 0; sweep < max_sweeps; ++sweep) {
        double off = 0.0;
        for (int i = 0; i < n; ++i)
            for (int j = 0; j < n; ++j)
                if (i != j) off += a[i * n + j] * a[i * n + j];
        if (sqrt(off) <= tol * fro) break;
        for (int p = 0; p < n - 1; ++p) {
            for (int q = p + 1; q < n; ++q) {
                double apq = a[p * n + q];
                if (apq == 0.0) continue;
                double tau = (a[q * n + q] - a[p * n + p]) / (2.0 * apq);
                double t = (tau >= 0.0 ? 1.0 : -1.0) / (fabs(tau) + sqrt(1.0 + tau * tau));
                double c = 1.0 / sqrt(1.0 + t * t);
                double s = t * c;
                for (int k = 0; k < n; ++k) {          /* A <- A J */
                    double akp = a[k * n + p], akq = a[k * n + q];
                    a[k * n + p] = c * akp - s * akq;
                    a[k * n + q] = s * akp + c * akq;
                }
                for (int k = 0; k < n; ++k) {          /* A <- J^T A */
                    double apk = a[p * n + k], aqk = a[q * n + k];
                    a[p * n + k] = c * apk - s * aqk;
                    a[q * n + k] = s * apk + c * aqk;
                }
                for (int k = 0; k < n; ++k) {          /* V <- V J */
                    double vkp = v[k * n + p], vkq = v[k * n + q];
                    v[k * n + p] = c * vkp - s * vkq;
                    v[k * n + q] = s * vkp + c * vkq;
                }
            }
        }
    }
    return sweep;
}

/* ------------------------------------------------------------------ build */

/*
 * Unquantised page summary [p1 "How LOCKS works", "Code"; p4 2.1]:
 *   mu = mean of the 16 keys, D = K - mu,
 *   top-`rank` eigenpairs (lambda_r, u_r) of the 16 x 16 Gram G = D D^T
 *   (descending; equal eigenvalues keep the lower index first),
 *   V[:, r] = D^T u_r / sqrt(lambda_r)  (= right singular vector of D),
 *   C[:, r] = sqrt(lambda_r) u_r         (= D V[:, r]).
 * A direction with lambda_r <= 1e-12 lambda_1 (or lambda_1 <= 0) carries no
 * energy: its V and C columns are zero. Sign: the entry of V[:, r] with the
 * largest magnitude (first on ties) is made positive, and C[:, r] follows.
 * basis is [128][rank], coef is [16][rank], eigvals gets all 16 (descending).
 */
void lo_build_unit_f64(const uint16_t* k, int rank, double* mu, double* basis,
                       double* coef, double* eigvals) {
    double d[LO_PAGE][LO_D];
    double g[LO_PAGE * LO_PAGE], u[LO_PAGE * LO_PAGE];
    for (int c = 0; c < LO_D; ++c) {
        double s = 0.0;
        for (int i = 0; i < LO_PAGE; ++i) s += lo_bf16_to_f64(k[i * LO_D + c]);
        mu[c] = s / LO_PAGE;
    }
    for (int i = 0; i < LO_PAGE; ++i)
        for (int c = 0; c < LO_D; ++c) d[i][c] = lo_bf16_to_f64(k[i * LO_D + c]) - mu[c];
    for (int i = 0; i < LO_PAGE; ++i)
        for (int j = 0; j < LO_PAGE; ++j) {
            double s = 0.0;
            for (int c = 0; c < LO_D; ++c) s += d[i][c] * d[j][c];
            g[i * LO_PAGE + j] = s;
        }
    lo_jacobi_eig(LO_PAGE, g, u, 1e-14, 100);
    int order[LO_PAGE];
    for (int i = 0; i < LO_PAGE; ++i) order[i] = i;
    for (int i = 1; i < LO_PAGE; ++i) {               /* stable insertion sort, descending */
        int x = order[i], j = i - 1;
        while (j >= 0 && g[order[j] * LO_PAGE + order[j]] < g[x * LO_PAGE + x]) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = x;
    }
    if (eigvals)
        for (int i = 0; i < LO_PAGE; ++i) eigvals[i] = g[order[i] * LO_PAGE + order[i]];
    double lam1 = g[order[0] * LO_PAGE + order[0]];
    for (int r = 0; r < rank; ++r) {
        double lam = g[order[r] * LO_PAGE + order[r]];
        int col = order[r];
        if (lam1 <= 0.0 || lam <= 1e-12 * lam1) {
            for (int c = 0; c < LO_D; ++c) basis[c * rank + r] = 0.0;
            for (int i = 0; i < LO_PAGE; ++i) coef[i * rank + r] = 0.0;
            continue;
        }
        double sigma = sqrt(lam);
        for (int c = 0; c < LO_D; ++c) {
            double s = 0.0;
            for (int i = 0; i < LO_PAGE; ++i) s += d[i][c] * u[i * LO_PAGE + col];
            basis[c * rank + r] = s / sigma;
        }
        for (int i = 0; i < LO_PAGE; ++i) coef[i * rank + r] = sigma * u[i * LO_PAGE + col];
        int best = 0;
        for (int c = 1; c < LO_D; ++c)
            if (fabs(basis[c * rank + r]) > fabs(basis[best * rank + r])) best = c;
        if (basis[best * rank + r] < 0.0) {
            for (int c = 0; c < LO_D; ++c) basis[c * rank + r] = -basis[c * rank + r];
            for (int i = 0; i < LO_PAGE; ++i) coef[i * rank + r] = -coef[i * rank + r];
        }
    }
}

/* Symmetric absmax quantiser: scale = fp16(absmax / qmax); code = clamp(rne(x / scale)). */
static uint16_t lo_quantise(const double* x, int n, int qmax, int* codes) {
    double amax = 0.0;
    for (int i = 0; i < n; ++i)
        if (fabs(x[i]) > amax) amax = fabs(x[i]);
    uint16_t sbits = lo_f64_to_f16(amax / qmax);
    double s = lo_f16_to_f64(sbits);
    for (int i = 0; i < n; ++i) {
        if (!(s > 0.0) || isinf(s)) {
            codes[i] = 0;
            continue;
        }
        double c = nearbyint(x[i] / s);
        if (c > qmax) c = qmax;
        if (c < -qmax) c = -qmax;
        codes[i] = (int)c;
    }
    return sbits;
}

/* Byte offsets of the layout described at the top of this file. */
static int lo_mu_offset(int dd) {
    int s = dd / 16, w = dd % 16, h = w / 8, t = (w % 8) / 2, e = w % 2;
    return 32 * t + 4 * s + 2 * h + e;
}
static void lo_basis_pos(int dd, int r, int* byte, int* nibble) {
    int s = dd / 16, w = dd % 16, h = w / 8, t = (w % 8) / 2, e = w % 2;
    int p = 2 * (s % 2) + h + 4 * e;
    *byte = 64 * r + 16 * t + 4 * (s / 2) + p / 2;
    *nibble = p % 2;
}
static int lo_coef_offset(int i, int r) { return 4 * (4 * (i % 8) + r / 2) + 2 * (i / 8) + r % 2; }

/* Encode dequantisable arrays into one unit's bytes. */
void lo_encode_unit(const double* mu, const double* basis /*[128][8]*/, const double* coef /*[16][8]*/,
                    int8_t* mu_out, uint8_t* basis_out, int8_t* coef_out, uint16_t* scales_out) {
    int codes[LO_D * LO_R];
    scales_out[0] = lo_quantise(mu, LO_D, 127, codes);
    for (int c = 0; c < LO_D; ++c) mu_out[lo_mu_offset(c)] = (int8_t)codes[c];
    scales_out[1] = lo_quantise(basis, LO_D * LO_R, 7, codes);
    memset(basis_out, 0, 512);
    for (int c = 0; c < LO_D; ++c)
        for (int r = 0; r < LO_R; ++r) {
            int byte, nib;
            lo_basis_pos(c, r, &byte, &nib);
            uint8_t v = (uint8_t)(codes[c * LO_R + r] & 0xf);
            basis_out[byte] |= (uint8_t)(nib ? (v << 4) : v);
        }
    scales_out[2] = lo_quantise(coef, LO_PAGE * LO_R, 127, codes);
    for (int i = 0; i < LO_PAGE; ++i)
        for (int r = 0; r < LO_R; ++r) coef_out[lo_coef_offset(i, r)] = (int8_t)codes[i * LO_R + r];
    scales_out[3] = 0;
}

/* Decode one unit's bytes into dequantised float64 arrays. */
void lo_decode_unit(const int8_t* mu, const uint8_t* basis, const int8_t* coef, const uint16_t* scales,
                    double* mu_hat, double* basis_hat /*[128][8]*/, double* coef_hat /*[16][8]*/) {
    double smu = lo_f16_to_f64(scales[0]), sv = lo_f16_to_f64(scales[1]), sc = lo_f16_to_f64(scales[2]);
    for (int c = 0; c < LO_D; ++c) mu_hat[c] = mu[lo_mu_offset(c)] * smu;
    for (int c = 0; c < LO_D; ++c)
        for (int r = 0; r < LO_R; ++r) {
            int byte, nib;
            lo_basis_pos(c, r, &byte, &nib);
            int v = nib ? (basis[byte] >> 4) & 0xf : basis[byte] & 0xf;
            if (v >= 8) v -= 16;
            basis_hat[c * LO_R + r] = v * sv;
        }
    for (int i = 0; i < LO_PAGE; ++i)
        for (int r = 0; r < LO_R; ++r) coef_hat[i * LO_R + r] = coef[lo_coef_offset(i, r)] * sc;
}

/* Build and quantise n units ([n][16][128] bf16 keys) into the byte layout. */
void lo_build_units(int64_t n, const uint16_t* k, int8_t* mu, uint8_t* basis, int8_t* coef,
                    uint16_t* scales) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t u = 0; u < n; ++u) {
        double m[LO_D], v[LO_D * LO_R], c[LO_PAGE * LO_R];
        lo_build_unit_f64(k + u * LO_PAGE * LO_D, LO_R, m, v, c, NULL);
        lo_encode_unit(m, v, c, mu + u * LO_D, basis + u * 512, coef + u * 128, scales + u * 4);
    }
}

/* ------------------------------------------------------------------ score */

/*
 * Summary-only page score [p1 "How LOCKS works"; p4 2.2]:
 *   s = log sum_i exp[(q . mu + (V^T q) . c_i) / sqrt(d)],  d = 128,
 * over the 16 tokens i of the page, evaluated with the maximum factored out.
 */
double lo_score_unit(const double* q, const double* mu, const double* basis, const double* coef,
                     int rank) {
    double a = 0.0;
    for (int c = 0; c < LO_D; ++c) a += q[c] * mu[c];
    double w[LO_PAGE];
    for (int r = 0; r < rank; ++r) {
        double s = 0.0;
        for (int c = 0; c < LO_D; ++c) s += basis[c * rank + r] * q[c];
        w[r] = s;
    }
    double t[LO_PAGE], mx = -INFINITY;
    for (int i = 0; i < LO_PAGE; ++i) {
        double s = a;
        for (int r = 0; r < rank; ++r) s += w[r] * coef[i * rank + r];
        t[i] = s / sqrt((double)LO_D);
        if (t[i] > mx) mx = t[i];
    }
    if (isnan(mx) || isinf(mx)) {
        double z = 0.0;
        for (int i = 0; i < LO_PAGE; ++i) z += exp(t[i]);
        return log(z);
    }
    double z = 0.0;
    for (int i = 0; i < LO_PAGE; ++i) z += exp(t[i] - mx);
    return mx + log(z);
}

/*
 * Scores of every (request b, query head h, logical page j < seq_pages[b]) from
 * the summary bytes of physical page page_table[b][j], kv head h / g.
 * scores is [B][Hq][max_pages]; entries j >= seq_pages[b] are left untouched.
 */
void lo_scores(int batch, int hq, int hkv, int max_pages, const float* q, const int8_t* mu,
               const uint8_t* basis, const int8_t* coef, const uint16_t* scales,
               const int32_t* page_table, const int32_t* seq_pages, double* scores) {
    int g = hq / hkv;
    int64_t total = (int64_t)batch * hkv * max_pages;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t idx = 0; idx < total; ++idx) {
        int b = (int)(idx / ((int64_t)hkv * max_pages));
        int kvh = (int)((idx / max_pages) % hkv);
        int j = (int)(idx % max_pages);
        if (j >= seq_pages[b]) continue;
        int64_t unit = (int64_t)page_table[(int64_t)b * max_pages + j] * hkv + kvh;
        double m[LO_D], v[LO_D * LO_R], c[LO_PAGE * LO_R], qq[LO_D];
        lo_decode_unit(mu + unit * LO_D, basis + unit * 512, coef + unit * 128, scales + unit * 4, m, v, c);
        for (int hh = 0; hh < g; ++hh) {
            int h = kvh * g + hh;
            for (int d = 0; d < LO_D; ++d) qq[d] = q[((int64_t)b * hq + h) * LO_D + d];
            scores[((int64_t)b * hq + h) * max_pages + j] = lo_score_unit(qq, m, v, c, LO_R);
        }
    }
}

/* Scores of n sampled (b, h, j) triples; out[i] is the score of sample i. */
void lo_scores_sampled(int batch, int hq, int hkv, int max_pages, const float* q, const int8_t* mu,
                       const uint8_t* basis, const int8_t* coef, const uint16_t* scales,
                       const int32_t* page_table, int64_t n, const int32_t* sb, const int32_t* sh,
                       const int32_t* sj, double* out) {
    (void)batch;
    int g = hq / hkv;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t i = 0; i < n; ++i) {
        int b = sb[i], h = sh[i], j = sj[i];
        int64_t unit = (int64_t)page_table[(int64_t)b * max_pages + j] * hkv + h / g;
        double m[LO_D], v[LO_D * LO_R], c[LO_PAGE * LO_R], qq[LO_D];
        lo_decode_unit(mu + unit * LO_D, basis + unit * 512, coef + unit * 128, scales + unit * 4, m, v, c);
        for (int d = 0; d < LO_D; ++d) qq[d] = q[((int64_t)b * hq + h) * LO_D + d];
        out[i] = lo_score_unit(qq, m, v, c, LO_R);
    }
}

/* ---------------------------------------------------------- group, select */

/*
 * Group-shared selection key [p4 2.3: average the estimated mass shares over
 * the query heads of a GQA group]. Per head the estimated mass share of page j
 * is exp(s_hj - L_h) with L_h = log sum_j exp(s_hj) over the sequence's pages;
 * the key is the log of the group mean of the shares:
 *   key_j = log( (1/g) sum_{h in group} exp(s_hj - L_h) ).
 * keys is [B][Hkv][max_pages], head_lse [B][Hq] (may be NULL).
 */
void lo_group_keys(int batch, int hq, int hkv, int max_pages, const double* scores,
                   const int32_t* seq_pages, double* keys, double* head_lse) {
    int g = hq / hkv;
    for (int b = 0; b < batch; ++b) {
        int P = seq_pages[b];
        for (int kvh = 0; kvh < hkv; ++kvh) {
            double L[64];
            for (int hh = 0; hh < g; ++hh) {
                const double* s = scores + ((int64_t)b * hq + kvh * g + hh) * max_pages;
                double mx = -INFINITY;
                for (int j = 0; j < P; ++j)
                    if (s[j] > mx) mx = s[j];
                double z = 0.0;
                for (int j = 0; j < P; ++j) z += exp(s[j] - mx);
                L[hh] = (P > 0) ? mx + log(z) : -INFINITY;
                if (head_lse) head_lse[(int64_t)b * hq + kvh * g + hh] = L[hh];
            }
            double* out = keys + ((int64_t)b * hkv + kvh) * max_pages;
            for (int j = 0; j < P; ++j) {
                double mx = -INFINITY, z = 0.0, x[64];
                for (int hh = 0; hh < g; ++hh) {
                    x[hh] = scores[((int64_t)b * hq + kvh * g + hh) * max_pages + j] - L[hh];
                    if (x[hh] > mx) mx = x[hh];
                }
                if (isinf(mx) && mx < 0) {
                    out[j] = -INFINITY;
                    continue;
                }
                for (int hh = 0; hh < g; ++hh) z += exp(x[hh] - mx);
                out[j] = mx + log(z / g);
            }
        }
    }
}

static const double* lo_sort_keys;
static int lo_cmp_desc(const void* pa, const void* pb) {
    int a = *(const int*)pa, b = *(const int*)pb;
    double ka = lo_sort_keys[a], kb = lo_sort_keys[b];
    if (isnan(ka)) ka = -INFINITY;
    if (isnan(kb)) kb = -INFINITY;
    if (ka > kb) return -1;
    if (ka < kb) return 1;
    return (a > b) - (a < b);                    /* equal keys: lower page id first */
}
static int lo_cmp_int(const void* pa, const void* pb) {
    int a = *(const int*)pa, b = *(const int*)pb;
    return (a > b) - (a < b);
}

/*
 * Top-k page selection [p1 "Code": k = budget // 16 pages, the chosen indices
 * sorted ascending]. k = min(budget // 16, seq_pages[b]); the k pages with the
 * largest keys, equal keys ordered by lower page id, NaN ranked as -inf.
 * selected is [B][Hkv][k_cap] (ascending page ids), n_selected [B][Hkv].
 */
void lo_select(int batch, int hkv, int max_pages, const double* keys, const int32_t* seq_pages,
               int budget_tokens, int k_cap, int32_t* selected, int32_t* n_selected) {
    int* idx = (int*)malloc(sizeof(int) * (max_pages > 0 ? max_pages : 1));
    for (int b = 0; b < batch; ++b)
        for (int kvh = 0; kvh < hkv; ++kvh) {
            int P = seq_pages[b];
            int k = budget_tokens / LO_PAGE;
            if (k > P) k = P;
            if (k > k_cap) k = k_cap;
            if (k < 0) k = 0;
            for (int j = 0; j < P; ++j) idx[j] = j;
            lo_sort_keys = keys + ((int64_t)b * hkv + kvh) * max_pages;
            qsort(idx, (size_t)P, sizeof(int), lo_cmp_desc);
            qsort(idx, (size_t)k, sizeof(int), lo_cmp_int);
            int32_t* out = selected + ((int64_t)b * hkv + kvh) * k_cap;
            for (int i = 0; i < k; ++i) out[i] = idx[i];
            n_selected[b * hkv + kvh] = k;
        }
    free(idx);
}

/* -------------------------------------------------------------- attention */

/*
 * Attention over the selected pages [p1 "Code": scaled dot-product attention of
 * q over the gathered keys/values of the chosen pages, default scale 1/sqrt(d)],
 * plus, when tail_tokens is given, the sequence's tail_tokens[b] tokens that
 * have no summary yet: logical pages seq_pages[b], seq_pages[b] + 1, ... (16
 * tokens each, the last one partial). A page gets its summary only once it fills
 * [p1 "How LOCKS works": the decomposition runs when a page fills, every 16
 * tokens, off the decode critical path], so the page being filled, and a filled
 * page whose summary is still being built, cannot be scored; they are attended
 * whole (the pages are silent on them; this is the plain reading).
 * For every (b, query head h) with kv head h / g, over that token set:
 *   l_i = q . k_i / sqrt(128),  out = sum_i softmax(l)_i v_i,  lse = log sum_i exp(l_i).
 * An empty set gives out = 0 and lse = -inf.
 * out is [B][Hq][128], lse [B][Hq] (may be NULL); seq_pages and tail_tokens may
 * both be NULL (no tail).
 */
void lo_attend(int batch, int hq, int hkv, int max_pages, const float* q, const uint16_t* k_cache,
               const uint16_t* v_cache, const int32_t* page_table, const int32_t* selected,
               const int32_t* n_selected, int k_cap, const int32_t* seq_pages, const int32_t* tail_tokens,
               double* out, double* lse) {
    int g = hq / hkv;
    int64_t total = (int64_t)batch * hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t bh = 0; bh < total; ++bh) {
        int b = (int)(bh / hq), h = (int)(bh % hq), kvh = h / g;
        int n = n_selected[b * hkv + kvh];
        const int32_t* sel = selected + ((int64_t)b * hkv + kvh) * k_cap;
        int tail = (tail_tokens && seq_pages) ? tail_tokens[b] : 0;
        const float* qv = q + bh * LO_D;
        double* o = out + bh * LO_D;
        for (int c = 0; c < LO_D; ++c) o[c] = 0.0;
        if (n < 0) n = 0;
        if (n == 0 && tail <= 0) {
            if (lse) lse[bh] = -INFINITY;
            continue;
        }
        /* the token set: (physical page, tokens used) for each selected page, then the tail pages */
        int ntail = (tail + LO_PAGE - 1) / LO_PAGE;
        int npages = n + ntail;
        int64_t* phys = (int64_t*)malloc(sizeof(int64_t) * npages);
        int* ntok = (int*)malloc(sizeof(int) * npages);
        for (int p = 0; p < n; ++p) {
            phys[p] = page_table[(int64_t)b * max_pages + sel[p]];
            ntok[p] = LO_PAGE;
        }
        for (int j = 0; j < ntail; ++j) {
            phys[n + j] = page_table[(int64_t)b * max_pages + seq_pages[b] + j];
            ntok[n + j] = tail - j * LO_PAGE < LO_PAGE ? tail - j * LO_PAGE : LO_PAGE;
        }
        double* logit = (double*)malloc(sizeof(double) * npages * LO_PAGE);
        double mx = -INFINITY;
        for (int p = 0; p < npages; ++p) {
            const uint16_t* kp = k_cache + (phys[p] * hkv + kvh) * LO_PAGE * LO_D;
            for (int i = 0; i < ntok[p]; ++i) {
                double s = 0.0;
                for (int c = 0; c < LO_D; ++c) s += (double)qv[c] * lo_bf16_to_f64(kp[i * LO_D + c]);
                logit[p * LO_PAGE + i] = s / sqrt((double)LO_D);
                if (logit[p * LO_PAGE + i] > mx) mx = logit[p * LO_PAGE + i];
            }
        }
        double z = 0.0;
        for (int p = 0; p < npages; ++p) {
            const uint16_t* vp = v_cache + (phys[p] * hkv + kvh) * LO_PAGE * LO_D;
            for (int i = 0; i < ntok[p]; ++i) {
                double w = exp(logit[p * LO_PAGE + i] - mx);
                z += w;
                for (int c = 0; c < LO_D; ++c) o[c] += w * lo_bf16_to_f64(vp[i * LO_D + c]);
            }
        }
        for (int c = 0; c < LO_D; ++c) o[c] /= z;
        if (lse) lse[bh] = mx + log(z);
        free(logit);
        free(ntok);
        free(phys);
    }
}

/* Rounds a real to the nearest fp16 value (exposed for the quantiser pins). */
double lo_round_f16(double x) { return lo_f16_round(x); }

/* -------------------------------------------------------------- ablations */

/*
 * Exact page score, the selector that reads every key ([p4] section 1, the
 * "exact selection" that reads all keys; section 3, the read-all-keys
 * selector LOCKS is measured against):
 *   s = log sum_i exp(q . k_i / sqrt(d)) over the 16 keys of the page.
 * k is one unit's [16][128] bf16 keys.
 */
double lo_exact_score_unit(const double* q, const uint16_t* k) {
    double t[LO_PAGE], mx = -INFINITY;
    for (int i = 0; i < LO_PAGE; ++i) {
        double s = 0.0;
        for (int c = 0; c < LO_D; ++c) s += q[c] * lo_bf16_to_f64(k[i * LO_D + c]);
        t[i] = s / sqrt((double)LO_D);
        if (t[i] > mx) mx = t[i];
    }
    double z = 0.0;
    for (int i = 0; i < LO_PAGE; ++i) z += exp(t[i] - mx);
    return mx + log(z);
}

/* The physical unit of (b, kv head, logical page j); NULL when j is past the sequence. */
static const uint16_t* lo_unit_keys(const uint16_t* k_cache, const int32_t* table, const int32_t* seq_pages,
                                    int hkv, int max_pages, int b, int kvh, int j) {
    if (j >= seq_pages[b]) return NULL;
    int64_t phys = table[(int64_t)b * max_pages + j];
    return k_cache + (phys * hkv + kvh) * (int64_t)(LO_PAGE * LO_D);
}

/* Exact scores of every (b, h, j < seq_pages[b]); out is [B][Hq][max_pages]. */
void lo_exact_scores(int batch, int hq, int hkv, int max_pages, const float* q, const uint16_t* k_cache,
                     const int32_t* table, const int32_t* seq_pages, double* out) {
    int g = hq / hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
    for (int b = 0; b < batch; ++b)
        for (int j = 0; j < max_pages; ++j)
            for (int kvh = 0; kvh < hkv; ++kvh) {
                const uint16_t* k = lo_unit_keys(k_cache, table, seq_pages, hkv, max_pages, b, kvh, j);
                if (!k) continue;
                for (int hh = 0; hh < g; ++hh) {
                    int h = kvh * g + hh;
                    double qq[LO_D];
                    for (int c = 0; c < LO_D; ++c) qq[c] = q[((int64_t)b * hq + h) * LO_D + c];
                    out[((int64_t)b * hq + h) * max_pages + j] = lo_exact_score_unit(qq, k);
                }
            }
}

/*
 * Replaces x[0..n) by its dequantised absmax codes of `bits` bits
 * (symmetric: qmax = 2^(bits-1) - 1, so int8 -> 127, int4 -> 7, int2 -> 1);
 * bits = 0 leaves x unquantised. The quantiser is the one of the shipped
 * summary ([p1] "How LOCKS works": int8 centroid, int4 basis, int8
 * coefficients), with the width as the ablated parameter ([p1] "Caveats").
 */
void lo_quant_dequant(double* x, int n, int bits) {
    if (bits == 0) return;
    int codes[LO_D * LO_PAGE];
    int qmax = (1 << (bits - 1)) - 1;
    double s = lo_f16_to_f64(lo_quantise(x, n, qmax, codes));
    for (int i = 0; i < n; ++i) x[i] = (s > 0.0 && !isinf(s)) ? codes[i] * s : 0.0;
}

/*
 * Ablation variant of the summary score: the page-local summary of rank
 * `rank` (1..15; 15 spans all 16 centred keys) built as lo_build_unit_f64
 * does, mu / V / C each quantised to bits_mu / bits_v / bits_c (8, 4, 2, or
 * 0 for unquantised, the setting Theorem 1 covers), dequantised and scored
 * with the summary score formula. Rank 8 with bits (8, 4, 8) is the shipped
 * summary. out is [B][Hq][max_pages].
 */
void lo_variant_scores(int batch, int hq, int hkv, int max_pages, const float* q, const uint16_t* k_cache,
                       const int32_t* table, const int32_t* seq_pages, int rank, int bits_mu, int bits_v,
                       int bits_c, double* out) {
    int g = hq / hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 16)
    for (int b = 0; b < batch; ++b)
        for (int j = 0; j < max_pages; ++j)
            for (int kvh = 0; kvh < hkv; ++kvh) {
                const uint16_t* k = lo_unit_keys(k_cache, table, seq_pages, hkv, max_pages, b, kvh, j);
                if (!k) continue;
                double mu[LO_D], basis[LO_D * LO_PAGE], coef[LO_PAGE * LO_PAGE];
                lo_build_unit_f64(k, rank, mu, basis, coef, NULL);
                lo_quant_dequant(mu, LO_D, bits_mu);
                lo_quant_dequant(basis, LO_D * rank, bits_v);
                lo_quant_dequant(coef, LO_PAGE * rank, bits_c);
                for (int hh = 0; hh < g; ++hh) {
                    int h = kvh * g + hh;
                    double qq[LO_D];
                    for (int c = 0; c < LO_D; ++c) qq[c] = q[((int64_t)b * hq + h) * LO_D + c];
                    out[((int64_t)b * hq + h) * max_pages + j] = lo_score_unit(qq, mu, basis, coef, rank);
                }
            }
}

/*
 * Shared basis of the kind shared-projection selectors use ([p1] "Why
 * shared-basis sparse attention is structurally broken": one low-rank basis
 * built from the full sequence): per (request b, kv head), the `rank`
 * eigenvectors of largest eigenvalue of M = sum_t k_t k_t^T over every token
 * of the sequence's seq_pages[b] pages (the top right singular vectors of the
 * sequence's key matrix), by the cyclic Jacobi method, descending (equal
 * eigenvalues keep the lower index first). A direction with
 * lambda <= 1e-12 lambda_1 is returned as zeros. Sign: the largest-magnitude
 * entry (first on ties) is positive. basis is [B][Hkv][rank][128]; eigvals,
 * if not NULL, gets all 128 eigenvalues of each M ([B][Hkv][128], descending).
 */
void lo_shared_basis(int batch, int hkv, int max_pages, const uint16_t* k_cache, const int32_t* table,
                     const int32_t* seq_pages, int rank, double* basis, double* eigvals) {
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int b = 0; b < batch; ++b)
        for (int kvh = 0; kvh < hkv; ++kvh) {
            double* m = (double*)calloc(LO_D * LO_D, sizeof(double));
            double* u = (double*)malloc(LO_D * LO_D * sizeof(double));
            double kt[LO_D];
            for (int j = 0; j < seq_pages[b]; ++j) {
                const uint16_t* k = lo_unit_keys(k_cache, table, seq_pages, hkv, max_pages, b, kvh, j);
                for (int i = 0; i < LO_PAGE; ++i) {
                    for (int c = 0; c < LO_D; ++c) kt[c] = lo_bf16_to_f64(k[i * LO_D + c]);
                    for (int r = 0; r < LO_D; ++r)
                        for (int c = 0; c < LO_D; ++c) m[r * LO_D + c] += kt[r] * kt[c];
                }
            }
            lo_jacobi_eig(LO_D, m, u, 1e-14, 100);
            int order[LO_D];
            for (int i = 0; i < LO_D; ++i) order[i] = i;
            for (int i = 1; i < LO_D; ++i) {           /* stable insertion sort, descending */
                int x = order[i], p = i - 1;
                while (p >= 0 && m[order[p] * LO_D + order[p]] < m[x * LO_D + x]) {
                    order[p + 1] = order[p];
                    --p;
                }
                order[p + 1] = x;
            }
            double* out = basis + ((int64_t)b * hkv + kvh) * rank * LO_D;
            if (eigvals)
                for (int i = 0; i < LO_D; ++i)
                    eigvals[((int64_t)b * hkv + kvh) * LO_D + i] = m[order[i] * LO_D + order[i]];
            double lam1 = m[order[0] * LO_D + order[0]];
            for (int r = 0; r < rank; ++r) {
                int col = order[r];
                double lam = m[col * LO_D + col];
                int best = 0;
                for (int c = 1; c < LO_D; ++c)
                    if (fabs(u[c * LO_D + col]) > fabs(u[best * LO_D + col])) best = c;
                double sgn = u[best * LO_D + col] < 0.0 ? -1.0 : 1.0;
                int keep = lam1 > 0.0 && lam > 1e-12 * lam1;
                for (int c = 0; c < LO_D; ++c) out[r * LO_D + c] = keep ? sgn * u[c * LO_D + col] : 0.0;
            }
            free(m);
            free(u);
        }
}

/*
 * Shared-basis page score: the keys seen through the fixed projection
 * P = W W^T of the basis W ([rank][128] rows per (b, kv head)),
 *   s = log sum_i exp(q . (P k_i) / sqrt(d)),
 * so a page whose keys lie in the null space of W^T scores log 16 whatever
 * the query ([p1] "Why shared-basis sparse attention is structurally broken";
 * Proposition 1 of [p4] section 3). out is [B][Hq][max_pages].
 */
void lo_shared_scores(int batch, int hq, int hkv, int max_pages, const float* q, const uint16_t* k_cache,
                      const int32_t* table, const int32_t* seq_pages, const double* basis, int rank,
                      double* out) {
    int g = hq / hkv;
#pragma omp parallel for collapse(2) schedule(dynamic, 64)
    for (int b = 0; b < batch; ++b)
        for (int j = 0; j < max_pages; ++j)
            for (int kvh = 0; kvh < hkv; ++kvh) {
                const uint16_t* k = lo_unit_keys(k_cache, table, seq_pages, hkv, max_pages, b, kvh, j);
                if (!k) continue;
                const double* w = basis + ((int64_t)b * hkv + kvh) * rank * LO_D;
                double pk[LO_PAGE][LO_D];
                for (int i = 0; i < LO_PAGE; ++i) {
                    for (int c = 0; c < LO_D; ++c) pk[i][c] = 0.0;
                    for (int r = 0; r < rank; ++r) {
                        double a = 0.0;
                        for (int c = 0; c < LO_D; ++c) a += w[r * LO_D + c] * lo_bf16_to_f64(k[i * LO_D + c]);
                        for (int c = 0; c < LO_D; ++c) pk[i][c] += a * w[r * LO_D + c];
                    }
                }
                for (int hh = 0; hh < g; ++hh) {
                    int h = kvh * g + hh;
                    double t[LO_PAGE], mx = -INFINITY;
                    for (int i = 0; i < LO_PAGE; ++i) {
                        double s = 0.0;
                        for (int c = 0; c < LO_D; ++c) s += q[((int64_t)b * hq + h) * LO_D + c] * pk[i][c];
                        t[i] = s / sqrt((double)LO_D);
                        if (t[i] > mx) mx = t[i];
                    }
                    double z = 0.0;
                    for (int i = 0; i < LO_PAGE; ++i) z += exp(t[i] - mx);
                    out[((int64_t)b * hq + h) * max_pages + j] = mx + log(z);
                }
            }
}
