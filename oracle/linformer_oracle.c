/*
 * Linformer attention forward: plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark do. It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (one "unit" = one (batch, head) pair):
 *   Xbar = Ehat . X               sequence-axis projection, Ehat is k x n
 *   S    = Q . Kbar^T / sqrt(d)    n x k compressed scores
 *   P    = row-softmax(S)          over the k projected positions
 *   O    = P . Vbar                n x d output, one row per query position
 * Sources:
 *   - "Linformer(Self-Attention with Linear Complexity) 요약 설명", section Model:
 *     E, F are k x n; row j of E merges the n keys into one compressed key;
 *     queries are not compressed, so the output stays n x d; worked shapes
 *     n=4096, d=64, k=256 -> Kbar 256x64, attention 4096x256, output 4096x64.
 *   - same page, section Transformer and Self-Attention: P is applied row-wise,
 *     softmax runs along the key axis of each query.
 *   - PaperWeekly efficient-Transformer survey, section 2.1 Multi-Head
 *     Self-Attention: the attention is a scaled dot product (scale 1/sqrt(d)).
 *   - "Linformer: Self-Attention with Linear Complexity - 中文验证版", section 方法适配:
 *     projections may be shared headwise, key-value (E = F) or layerwise.
 *   - 요약 설명, section Model (padding paragraph): the projection is tied to the
 *     maximum length, so short inputs are padded; padded rows of K and V count as
 *     zero before the projection and padded query rows produce zero output.
 *
 * All arithmetic is in double precision, in the order the definition states it:
 * no blocking, no fusion, no reordering.  Parity: pinned (see tests/test_oracle.py):
 * golden hand-derived cases, the k = n, E = F = I reduction to library softmax
 * attention, projection against a library matmul, closed forms (Q = 0, k = 1),
 * and invariants (row sums, sharing modes, padding, permutation, linearity).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Sharing modes, numbered as the library's public header numbers them. */
enum { OR_PER_HEAD = 0, OR_KV = 1, OR_HEADWISE = 2, OR_LAYERWISE = 3 };

/* Kbar[j][c] = sum_{t < L} Ehat[j][t] * X[t][c]   (Ehat: k x n row-major, X: n x d)
 * Rows t >= L of X are never read: they count as zero whatever they hold. */
static void project_row(int n, int d, int j, int L, const double *Ehat, const double *X,
                        double *Xbar)
{
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int t = 0; t < L; ++t)
            acc += Ehat[(int64_t)j * n + t] * X[(int64_t)t * d + c];
        Xbar[(int64_t)j * d + c] = acc;
    }
}

void oracle_project(int n, int d, int k, int L, const double *Ehat, const double *X,
                    double *Xbar)
{
    for (int j = 0; j < k; ++j) project_row(n, d, j, L, Ehat, X, Xbar);
}

/* One query row i (0 <= i < n) of the compressed attention.
 * i >= L: zero output row (and zero P row if P is given). */
static void attend_row(int d, int k, int L, int i, const double *Q, const double *Kbar,
                       const double *Vbar, double *s, double *Orow, double *Prow)
{
    if (i >= L) {
        for (int c = 0; c < d; ++c) Orow[c] = 0.0;
        if (Prow) for (int j = 0; j < k; ++j) Prow[j] = 0.0;
        return;
    }
    const double scale = 1.0 / sqrt((double)d);
    const double *q = Q + (int64_t)i * d;
    for (int j = 0; j < k; ++j) {
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += q[c] * Kbar[(int64_t)j * d + c];
        s[j] = dot * scale;
    }
    double m = s[0];
    for (int j = 1; j < k; ++j) if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int j = 0; j < k; ++j) { s[j] = exp(s[j] - m); sum += s[j]; }
    for (int j = 0; j < k; ++j) s[j] /= sum;
    for (int c = 0; c < d; ++c) {
        double acc = 0.0;
        for (int j = 0; j < k; ++j) acc += s[j] * Vbar[(int64_t)j * d + c];
        Orow[c] = acc;
    }
    if (Prow) for (int j = 0; j < k; ++j) Prow[j] = s[j];
}

/* Selected query rows of one unit: O[r][:] (and P[r][:] if P != NULL) for
 * query row rows[r].  Q is that unit's n x d query block. */
int oracle_attend(int n, int d, int k, int L, const double *Q, const double *Kbar,
                  const double *Vbar, const int64_t *rows, int64_t nrows, double *O,
                  double *P)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(k > 0 ? k : 1));
    if (!s) return -1;
    for (int64_t r = 0; r < nrows; ++r) {
        if (rows[r] < 0 || rows[r] >= n) { free(s); return -2; }
        attend_row(d, k, L, (int)rows[r], Q, Kbar, Vbar, s, O + r * d, P ? P + r * k : NULL);
    }
    free(s);
    return 0;
}

/* Which projection a unit uses.  E, F are [h][k][n] in PER_HEAD and KV modes and
 * [k][n] in HEADWISE and LAYERWISE modes; KV and LAYERWISE use F = E. */
static void pick_projections(int share_mode, int head, int k, int n, const double *E,
                             const double *F, const double **Eh, const double **Fh)
{
    int64_t off = (share_mode == OR_PER_HEAD || share_mode == OR_KV)
                      ? (int64_t)head * k * n : 0;
    *Eh = E + off;
    *Fh = (share_mode == OR_KV || share_mode == OR_LAYERWISE) ? *Eh : F + off;
}

static int valid_length(const int32_t *pad_lengths, int batch, int n)
{
    if (!pad_lengths) return n;
    int L = pad_lengths[batch];
    return L < 0 ? 0 : (L > n ? n : L);
}

/* Whole problem.  Q, K, V, O: [b][h][n][d]; pad_lengths: int32[b] or NULL
 * (values clamped to [0, n]); Kbar_out / Vbar_out: optional [b][h][k][d].
 * nthreads <= 0 uses the OpenMP default.  Returns the thread count used. */
int oracle_linformer_fwd(const double *Q, const double *K, const double *V,
                         const double *E, const double *F, const int32_t *pad_lengths,
                         double *O, double *Kbar_out, double *Vbar_out, int b, int h, int n,
                         int d, int k, int share_mode, int nthreads)
{
    if (b < 1 || h < 1 || n < 1 || d < 1 || k < 1) return -2;
    if (share_mode < 0 || share_mode > 3) return -4;
    const int64_t units = (int64_t)b * h;
    const int64_t nd = (int64_t)n * d, kd = (int64_t)k * d;
    double *Kb = Kbar_out ? Kbar_out : (double *)malloc(sizeof(double) * units * kd);
    double *Vb = Vbar_out ? Vbar_out : (double *)malloc(sizeof(double) * units * kd);
    if (!Kb || !Vb) return -1;
    int used = 1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#endif
    /* Step 1: projections, one projected row of one unit per iteration. */
#pragma omp parallel
    {
#ifdef _OPENMP
#pragma omp single
        used = omp_get_num_threads();
#endif
#pragma omp for schedule(dynamic, 4)
        for (int64_t uj = 0; uj < units * k; ++uj) {
            const int64_t u = uj / k;
            const int j = (int)(uj % k);
            const int batch = (int)(u / h), head = (int)(u % h);
            const int L = valid_length(pad_lengths, batch, n);
            const double *Eh, *Fh;
            pick_projections(share_mode, head, k, n, E, F, &Eh, &Fh);
            project_row(n, d, j, L, Eh, K + u * nd, Kb + u * kd);
            project_row(n, d, j, L, Fh, V + u * nd, Vb + u * kd);
        }
        /* Step 2: compressed attention, one query row per iteration. */
        double *s = (double *)malloc(sizeof(double) * (size_t)k);
#pragma omp for schedule(static)
        for (int64_t ui = 0; ui < units * n; ++ui) {
            const int64_t u = ui / n;
            const int i = (int)(ui % n);
            const int L = valid_length(pad_lengths, (int)(u / h), n);
            attend_row(d, k, L, i, Q + u * nd, Kb + u * kd, Vb + u * kd, s,
                       O + u * nd + (int64_t)i * d, NULL);
        }
        free(s);
    }
    if (!Kbar_out) free(Kb);
    if (!Vbar_out) free(Vb);
    return used;
}

/* Plain full softmax attention (no projection), for small pins only:
 * O = softmax(Q K^T / sqrt(d)) V over all n keys.  Q, K, V, O: n x d. */
void oracle_full_attention(int n, int d, const double *Q, const double *K, const double *V,
                           double *O)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    const double scale = 1.0 / sqrt((double)d);
    for (int i = 0; i < n; ++i) {
        for (int j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int c = 0; c < d; ++c) dot += Q[(int64_t)i * d + c] * K[(int64_t)j * d + c];
            s[j] = dot * scale;
        }
        double m = s[0];
        for (int j = 1; j < n; ++j) if (s[j] > m) m = s[j];
        double sum = 0.0;
        for (int j = 0; j < n; ++j) { s[j] = exp(s[j] - m); sum += s[j]; }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < n; ++j) acc += (s[j] / sum) * V[(int64_t)j * d + c];
            O[(int64_t)i * d + c] = acc;
        }
    }
    free(s);
}
