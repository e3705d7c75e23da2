/*
 * PuzzleKV oracle: a plain, slow, fp64 CPU statement of what the hot path
 * computes.  TEST INFRASTRUCTURE ONLY -- the product library neither links
 * nor calls anything here; only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it.  It shares no code, header or table
 * with the CUDA path.
 *
 * Citations name sections and equations of the page "PuzzleKV: Page-Wise
 * Low-Rank Decomposition for KV Cache Compression" (written [PuzzleKV] below).
 *
 * What it computes:
 *   - the page classification (sink page, dense local window, partial last
 *     page, everything else factorized)            [PuzzleKV §3.3 ①②③, ⑤]
 *   - the rank-r truncated SVD of every eligible page, by the plain
 *     definition: a one-sided (Hestenes) Jacobi SVD of the P x d page in
 *     fp64, singular values sorted descending, factors in the eq. (2) form
 *     L = U_r, R = Sigma_r W_r^T                    [PuzzleKV §3.2, eq. (2)]
 *   - decode attention as the plain softmax of eq. (1) over the cache with
 *     every factorized page replaced by its reconstruction L R; eqs. (4)-(5)
 *     are an exact regrouping of this, so no online softmax appears here.
 *                                                   [PuzzleKV §3.2 eq. (1), §3.3 ④]
 *   - INT4 factors: singular values absorbed into both factors, symmetric
 *     INT4 codes with one scale per column (L_K, R_K, R_V) or per row (L_V),
 *     and their dequantization                     [PuzzleKV §4.3]
 *   - the rotary position embedding applied to keys at cache access when
 *     keys are factorized before it          [PuzzleKV §4.1, Appendix D.3]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_FACTORED 0
#define ORACLE_DENSE 1

/*
 * Page classification [PuzzleKV §3.3 ①②③ and ⑤].  A cache of T tokens is cut
 * into ceil(T/P) pages.  Dense: the sink pages (those holding the first
 * `sink_tokens` tokens), every page holding a token of the local window
 * [T - window_tokens, T), and the incomplete last page.  Every other page
 * is a completed page outside both regions and is factorized.
 * Writes one kind per page into kinds[0..n) and returns the page count, or
 * -1 if `cap` is too small.
 */
int oracle_page_kinds(int T, int P, int sink_tokens, int window_tokens, int *kinds, int cap)
{
    int n_pages = (T + P - 1) / P;
    int sink_pages = (sink_tokens + P - 1) / P;
    int window_lo = T - window_tokens;
    if (n_pages > cap)
        return -1;
    for (int p = 0; p < n_pages; ++p) {
        int first = p * P;
        int end = first + P < T ? first + P : T; /* one past the last token */
        int is_sink = p < sink_pages;
        int is_partial = (end - first) < P;
        int in_window = end > window_lo;
        kinds[p] = (is_sink || is_partial || in_window) ? ORACLE_DENSE : ORACLE_FACTORED;
    }
    return n_pages;
}

static double dot(const double *a, const double *b, int n)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i)
        s += a[i] * b[i];
    return s;
}

/*
 * Singular value decomposition X = U Sigma W^T of an n x d matrix (row-major,
 * n <= d) by one-sided Jacobi on the rows [PuzzleKV §3.2 "Truncated SVD"].
 *
 * Rows y_p, y_q of Y (initially X) are rotated until all rows are mutually
 * orthogonal; the same plane rotations accumulate into U (initially I), so
 * that X = U Y holds throughout.  At the end row i of Y equals
 * sigma_i w_i^T.  Rows are then ordered by descending norm, ties keeping the
 * lower original index.
 *
 * Outputs: U (n x n, row-major, columns = left singular vectors),
 * S (n, descending), Y (n x d, row i = sigma_i w_i^T, i.e. Sigma W^T).
 * Returns the number of sweeps, or -1 when it did not converge within
 * the sweep cap.
 */
int oracle_svd(const double *X, int n, int d, double *U, double *S, double *Y)
{
    double *y = (double *)malloc(sizeof(double) * (size_t)n * d);
    double *u = (double *)malloc(sizeof(double) * (size_t)n * n);
    double *norm2 = (double *)malloc(sizeof(double) * n);
    int *order = (int *)malloc(sizeof(int) * n);
    int sweeps = 0, converged = 0;
    const int max_sweeps = 100;
    const double tol = 1e-15;

    memcpy(y, X, sizeof(double) * (size_t)n * d);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j)
            u[i * n + j] = (i == j) ? 1.0 : 0.0;
    /* Rows whose norm falls below 1e-14 ||X||_F are zero to working
     * precision (what is left of them is rounding noise); rotating them
     * changes nothing in exact arithmetic and can go on forever in floating
     * point, so they take part in no rotation. */
    double frob2 = 0.0;
    for (size_t i = 0; i < (size_t)n * d; ++i)
        frob2 += X[i] * X[i];
    const double negligible = 1e-28 * frob2;

    while (!converged && sweeps < max_sweeps) {
        int rotated = 0;
        for (int p = 0; p < n - 1; ++p) {
            for (int q = p + 1; q < n; ++q) {
                double *yp = y + (size_t)p * d, *yq = y + (size_t)q * d;
                double alpha = dot(yp, yp, d);
                double beta = dot(yq, yq, d);
                double gamma = dot(yp, yq, d);
                if (gamma == 0.0 || fabs(gamma) <= tol * sqrt(alpha * beta) || alpha <= negligible ||
                    beta <= negligible)
                    continue;
                /* tan of the angle that zeroes the rotated rows' inner product
                 * (smaller root of t^2 + 2 zeta t - 1 = 0). */
                double zeta = (beta - alpha) / (2.0 * gamma);
                double t = (zeta >= 0.0 ? 1.0 : -1.0) / (fabs(zeta) + sqrt(1.0 + zeta * zeta));
                double c = 1.0 / sqrt(1.0 + t * t);
                double s = c * t;
                for (int k = 0; k < d; ++k) {
                    double a = yp[k], b = yq[k];
                    yp[k] = c * a - s * b;
                    yq[k] = s * a + c * b;
                }
                for (int k = 0; k < n; ++k) {
                    double a = u[k * n + p], b = u[k * n + q];
                    u[k * n + p] = c * a - s * b;
                    u[k * n + q] = s * a + c * b;
                }
                rotated = 1;
            }
        }
        ++sweeps;
        if (!rotated)
            converged = 1;
    }

    for (int i = 0; i < n; ++i) {
        norm2[i] = dot(y + (size_t)i * d, y + (size_t)i * d, d);
        order[i] = i;
    }
    /* insertion sort: descending norm, stable (lower index first on ties) */
    for (int i = 1; i < n; ++i) {
        int key = order[i], j = i - 1;
        while (j >= 0 && norm2[order[j]] < norm2[key]) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = key;
    }
    for (int i = 0; i < n; ++i) {
        int src = order[i];
        S[i] = sqrt(norm2[src]);
        memcpy(Y + (size_t)i * d, y + (size_t)src * d, sizeof(double) * d);
        for (int k = 0; k < n; ++k)
            U[k * n + i] = u[k * n + src];
    }
    free(y);
    free(u);
    free(norm2);
    free(order);
    return converged ? sweeps : -1;
}

/*
 * Rank-r truncated factors of one P x d page in the form of eq. (2):
 * L = U_r (P x r), R = Sigma_r W_r^T (r x d)          [PuzzleKV §3.3 eq. (2)]
 * Also returns all P singular values in S.  Returns the SVD's status.
 */
int oracle_factorize_page(const double *X, int P, int d, int r, double *L, double *R, double *S)
{
    double *U = (double *)malloc(sizeof(double) * (size_t)P * P);
    double *Y = (double *)malloc(sizeof(double) * (size_t)P * d);
    int st = oracle_svd(X, P, d, U, S, Y);
    for (int i = 0; i < P; ++i)
        for (int j = 0; j < r; ++j)
            L[i * r + j] = U[i * P + j];
    memcpy(R, Y, sizeof(double) * (size_t)r * d);
    free(U);
    free(Y);
    return st;
}

/* Many independent pages X[n][P][d]; pages are independent units
 * [PuzzleKV §3.3 ③], so they may run on several host threads. Returns the
 * number of pages whose SVD did not converge. */
int oracle_factorize_pages(const double *X, long n, int P, int d, int r,
                           double *L, double *R, double *S, int nthreads)
{
    int failures = 0;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads) reduction(+ : failures)
#endif
    for (long i = 0; i < n; ++i) {
        int st = oracle_factorize_page(X + (size_t)i * P * d, P, d, r,
                                       L + (size_t)i * P * r, R + (size_t)i * r * d,
                                       S + (size_t)i * P);
        if (st < 0)
            failures += 1;
    }
    (void)nthreads;
    return failures;
}

/*
 * Attention for G query rows over T keys/values, eq. (1):
 * out = softmax(q K^T / sqrt(d)) V.  q: G x d, K, V: T x d, out: G x d.
 *                                                  [PuzzleKV §3.2 eq. (1)]
 */
void oracle_attention(const double *q, const double *K, const double *V,
                      int G, int T, int d, double *out)
{
    double *s = (double *)malloc(sizeof(double) * (T > 0 ? T : 1));
    double scale = 1.0 / sqrt((double)d);
    for (int g = 0; g < G; ++g) {
        const double *qg = q + (size_t)g * d;
        double m = -INFINITY, denom = 0.0;
        for (int j = 0; j < T; ++j) {
            s[j] = dot(qg, K + (size_t)j * d, d) * scale;
            if (s[j] > m)
                m = s[j];
        }
        for (int j = 0; j < T; ++j) {
            s[j] = exp(s[j] - m);
            denom += s[j];
        }
        for (int k = 0; k < d; ++k) {
            double acc = 0.0;
            for (int j = 0; j < T; ++j)
                acc += s[j] * V[(size_t)j * d + k];
            out[(size_t)g * d + k] = acc / denom;
        }
    }
    free(s);
}

/*
 * Decode attention of one (sequence, layer, KV head) over a hybrid cache
 * [PuzzleKV §3.3 ④]: every factorized page is replaced by its reconstruction
 * K_p = L_K R_K, V_p = L_V R_V, every dense page is used as stored, and the
 * plain softmax attention of eq. (1) runs over the T reconstructed rows.
 *
 *   q:       G x d query rows of the heads sharing this KV head
 *   kinds:   per page, ORACLE_FACTORED or ORACLE_DENSE
 *   Kd, Vd:  T x d stored dense rows (only rows of dense pages are read)
 *   LK, RK:  per page P x rk and rk x d key factors (read for factorized pages)
 *   LV, RV:  per page P x rv and rv x d value factors
 */
void oracle_decode_head(const double *q, int G, int d, int T, int P,
                        const int *kinds, const double *Kd, const double *Vd,
                        const double *LK, const double *RK, int rk,
                        const double *LV, const double *RV, int rv, double *out)
{
    double *K = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
    double *V = (double *)malloc(sizeof(double) * (size_t)(T > 0 ? T : 1) * d);
    int n_pages = (T + P - 1) / P;
    for (int p = 0; p < n_pages; ++p) {
        int first = p * P;
        int rows = (first + P < T ? first + P : T) - first;
        for (int i = 0; i < rows; ++i) {
            double *krow = K + (size_t)(first + i) * d;
            double *vrow = V + (size_t)(first + i) * d;
            if (kinds[p] == ORACLE_DENSE) {
                memcpy(krow, Kd + (size_t)(first + i) * d, sizeof(double) * d);
                memcpy(vrow, Vd + (size_t)(first + i) * d, sizeof(double) * d);
            } else {
                const double *lk = LK + (size_t)p * P * rk + (size_t)i * rk;
                const double *lv = LV + (size_t)p * P * rv + (size_t)i * rv;
                const double *Rk = RK + (size_t)p * rk * d;
                const double *Rv = RV + (size_t)p * rv * d;
                for (int k = 0; k < d; ++k) {
                    double a = 0.0, b = 0.0;
                    for (int j = 0; j < rk; ++j)
                        a += lk[j] * Rk[(size_t)j * d + k];
                    for (int j = 0; j < rv; ++j)
                        b += lv[j] * Rv[(size_t)j * d + k];
                    krow[k] = a;
                    vrow[k] = b;
                }
            }
        }
    }
    oracle_attention(q, K, V, G, T, d, out);
    free(K);
    free(V);
}

/*
 * Singular values absorbed into both factors [PuzzleKV §4.3]: from
 * L = U_r and R = Sigma_r W_r^T (the eq. (2) form), Lt = U_r Sigma_r^{1/2} and
 * Rt = Sigma_r^{1/2} W_r^T, so that Lt Rt = L R.  Sigma_r is read off R as the
 * norms of its rows (L has orthonormal columns); a zero row leaves both
 * factors' j-th column / row zero.
 *   L: [P][r], R: [r][d] in; Lt: [P][r], Rt: [r][d] out (may alias L, R).
 */
void oracle_absorb_sigma(const double *L, const double *R, int P, int d, int r, double *Lt, double *Rt)
{
    for (int j = 0; j < r; ++j) {
        const double s = sqrt(dot(R + (size_t)j * d, R + (size_t)j * d, d));
        const double rs = sqrt(s);
        for (int i = 0; i < P; ++i) Lt[(size_t)i * r + j] = rs > 0.0 ? L[(size_t)i * r + j] * rs : 0.0;
        for (int k = 0; k < d; ++k) Rt[(size_t)j * d + k] = rs > 0.0 ? R[(size_t)j * d + k] / rs : 0.0;
    }
}

/*
 * Symmetric INT4 quantization of one matrix [PuzzleKV §4.3]: each group (a
 * row when per_row, else a column) gets one scale s = max|x| / 7 and codes
 * c = round(x / s) in [-7, 7] (no zero point; the 15 symmetric levels),
 * so that |x - c s| <= s / 2.  An all-zero group gets s = 0 and zero codes.
 *   x: [rows][cols] in; codes: [rows][cols] out; scales: [rows] or [cols] out.
 */
void oracle_quantize_int4(const double *x, int rows, int cols, int per_row, signed char *codes, double *scales)
{
    const int ng = per_row ? rows : cols, glen = per_row ? cols : rows;
    for (int g = 0; g < ng; ++g) {
        double amax = 0.0;
        for (int t = 0; t < glen; ++t) {
            const double v = per_row ? x[(size_t)g * cols + t] : x[(size_t)t * cols + g];
            if (fabs(v) > amax) amax = fabs(v);
        }
        const double s = amax / 7.0;
        scales[g] = s;
        for (int t = 0; t < glen; ++t) {
            const size_t idx = per_row ? (size_t)g * cols + t : (size_t)t * cols + g;
            double c = s > 0.0 ? nearbyint(x[idx] / s) : 0.0;
            if (c > 7.0) c = 7.0;
            if (c < -7.0) c = -7.0;
            codes[idx] = (signed char)c;
        }
    }
}

/* x = c s, the dequantized matrix of oracle_quantize_int4's output. */
void oracle_dequantize_int4(const signed char *codes, const double *scales, int rows, int cols, int per_row,
                            double *x)
{
    for (int i = 0; i < rows; ++i)
        for (int k = 0; k < cols; ++k)
            x[(size_t)i * cols + k] = codes[(size_t)i * cols + k] * scales[per_row ? i : k];
}

/*
 * Rotary position embedding of n rows of X (n x d) [PuzzleKV §4.1 and
 * Appendix D.3: keys factorized before RoPE are rotated at cache access].
 * Rotate-half pairing: row t sits at position pos[t]; for each i < d/2 the
 * pair (x_i, x_{i+d/2}) turns by the angle pos[t] * theta^(-2i/d):
 *     x'_i       = x_i cos(a) - x_{i+d/2} sin(a)
 *     x'_{i+d/2} = x_{i+d/2} cos(a) + x_i sin(a)
 * out may not alias X.
 */
void oracle_rope(const double *X, const long *pos, long n, int d, double theta, double *out)
{
    int h = d / 2;
    for (long t = 0; t < n; ++t) {
        const double *x = X + t * (long)d;
        double *y = out + t * (long)d;
        for (int i = 0; i < h; ++i) {
            double a = (double)pos[t] * pow(theta, -2.0 * (double)i / (double)d);
            double c = cos(a), s = sin(a);
            y[i] = x[i] * c - x[i + h] * s;
            y[i + h] = x[i + h] * c + x[i] * s;
        }
    }
}
