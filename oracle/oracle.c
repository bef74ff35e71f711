/*
 * oracle.c -- plain CPU reference for distance-bound smoothing.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline of the benchmark call this code.  It shares no source, header,
 * table or helper with the CUDA library, and the library never calls it.
 *
 * What it computes (GPU Gems 2, ch. 43, "GPU Computing for Protein Structure
 * Prediction"):
 *   section 2 (triangle inequality): through a middle atom k,
 *       u_ij <- min(u_ij, u_ik + u_kj)
 *       l_ij <- max(l_ij, l_ik - u_kj, l_kj - u_ik)
 *     and the upper bound is tightened before the lower bound uses it;
 *   section 3 (Floyd-Warshall rounds): k runs 0..n-1 in order, every pair
 *     (i, j) is updated in each round, and round k+1 sees the whole matrix that
 *     round k produced;
 *   section 5 (stepping through rounds): each round is computed from a copy of
 *     the matrix taken at the start of the round, so no new value of round k is
 *     read inside round k.
 *
 * Only row k and column k are read by other cells in round k, so the "copy of
 * the matrix" is kept as copies of row k and column k of U and L.  Every cell,
 * the diagonal included, is updated.
 *
 * Rules for the lower bound:
 *   ORACLE_RULE_LITERAL  -- the section-2 formula as printed:
 *       l_ij <- max(l_ij, l_ik - u_kj, l_kj - u_ik)
 *   ORACLE_RULE_CLOSURE  -- the same formula with the column value first raised
 *       by the path i -> k -> k' (the pair (k, k) itself):
 *       lc_i  = max(l_ik, l_kk - u_ik)
 *       l_ij <- max(l_ij, l_kj - u_ik, lc_i - u_kj)
 *     The two coincide whenever l_kk = 0, which holds for every consistent set
 *     of bounds.  CLOSURE makes the result the exact fixed point of the
 *     triangle inequalities (shortest paths on the bound graph with a doubled
 *     vertex set), independent of the order the cells are visited in.
 *
 * Arithmetic: fp32 (the chapter's precision), int32 in 1/1024 A units (sums
 * formed in int64), and fp64 for diagnostics.  No FMA contraction, no fast
 * math; fp32 operations round to nearest-even.
 *
 * oracle_closure_rows() gives single rows of the fixed point at any size by a
 * different route (Dijkstra on the bound graph) for sampled checks of large
 * matrices.
 *
 * oracle_smooth_track_f64() is the fp64 closure-rule smoothing that also keeps,
 * for every cell, which path its value is the length of: the number of edges
 * and, for the lower bound, the sum of the magnitudes of the edge weights.
 * Rounding bounds for fp32 results off the 1/1024 grid are stated in those
 * terms (see that function).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_RULE_CLOSURE = 0, ORACLE_RULE_LITERAL = 1 };

int oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads for the following calls (timing only: results never depend on it). */
void oracle_set_threads(int t) {
#ifdef _OPENMP
    if (t > 0) omp_set_num_threads(t);
#else
    (void)t;
#endif
}

/* One implementation per arithmetic type.  T is the stored type, W the type in
 * which a sum or a difference is formed (int64 for int32 storage, so the oracle
 * itself never overflows), and the result of a min or max is always one of the
 * stored operands or a formed value that fits T because it lies between stored
 * values. */
#define DEFINE_SMOOTH(NAME, T, W)                                                   \
int NAME(T *U, T *L, int64_t n, int64_t ld, int rule, int64_t k_begin,             \
         int64_t k_end)                                                            \
{                                                                                  \
    if (n < 0 || ld < n || k_begin < 0 || k_end > n || k_begin > k_end)           \
        return 1;                                                                  \
    if (n == 0) return 0;                                                          \
    T *urow = (T *)malloc(sizeof(T) * (size_t)n);                                  \
    T *ucol = (T *)malloc(sizeof(T) * (size_t)n);                                  \
    T *lrow = (T *)malloc(sizeof(T) * (size_t)n);                                  \
    T *lcol = (T *)malloc(sizeof(T) * (size_t)n);                                  \
    if (!urow || !ucol || !lrow || !lcol) {                                        \
        free(urow); free(ucol); free(lrow); free(lcol);                            \
        return 2;                                                                  \
    }                                                                              \
    for (int64_t k = k_begin; k < k_end; ++k) {                                    \
        /* copies taken at the start of round k */                                 \
        for (int64_t j = 0; j < n; ++j) urow[j] = U[k * ld + j];                   \
        for (int64_t i = 0; i < n; ++i) ucol[i] = U[i * ld + k];                   \
        if (L) {                                                                   \
            for (int64_t j = 0; j < n; ++j) lrow[j] = L[k * ld + j];               \
            for (int64_t i = 0; i < n; ++i) lcol[i] = L[i * ld + k];               \
            if (rule == ORACLE_RULE_CLOSURE) {                                     \
                T lkk = L[k * ld + k];                                             \
                for (int64_t i = 0; i < n; ++i) {                                  \
                    W c = (W)lkk - (W)ucol[i];                                     \
                    if (c > (W)lcol[i]) lcol[i] = (T)c;                            \
                }                                                                  \
            }                                                                      \
        }                                                                          \
        _Pragma("omp parallel for schedule(static)")                               \
        for (int64_t i = 0; i < n; ++i) {                                          \
            T *Ui = U + i * ld;                                                    \
            const W uik = (W)ucol[i];                                              \
            for (int64_t j = 0; j < n; ++j) {                                      \
                /* upper bound first */                                            \
                W s = uik + (W)urow[j];                                            \
                if (s < (W)Ui[j]) Ui[j] = (T)s;                                    \
            }                                                                      \
            if (L) {                                                               \
                T *Li = L + i * ld;                                                \
                const W lik = (W)lcol[i];                                          \
                for (int64_t j = 0; j < n; ++j) {                                  \
                    W a = (W)lrow[j] - uik;      /* l_kj - u_ik */                 \
                    W b = lik - (W)urow[j];      /* l_ik - u_kj */                 \
                    W m = a > b ? a : b;                                           \
                    if (m > (W)Li[j]) Li[j] = (T)m;                                \
                }                                                                  \
            }                                                                      \
        }                                                                          \
    }                                                                              \
    free(urow); free(ucol); free(lrow); free(lcol);                                \
    return 0;                                                                      \
}

DEFINE_SMOOTH(oracle_smooth_f32, float, float)
DEFINE_SMOOTH(oracle_smooth_f64, double, double)
DEFINE_SMOOTH(oracle_smooth_i32, int32_t, int64_t)

/* Count of cells (diagonal included) with L > U: the infeasibility flags. */
int64_t oracle_count_infeasible_f32(const float *U, const float *L, int64_t n, int64_t ld)
{
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            c += L[i * ld + j] > U[i * ld + j];
    return c;
}

int64_t oracle_count_infeasible_i32(const int32_t *U, const int32_t *L, int64_t n,
                                    int64_t ld)
{
    int64_t c = 0;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j)
            c += L[i * ld + j] > U[i * ld + j];
    return c;
}

/*
 * Single rows of the smoothing fixed point, by shortest paths.
 *
 * The triangle inequalities of section 2 are the shortest-path conditions of a
 * graph with two copies a', a'' of every atom: edge a'->b' and a''->b'' weigh
 * u_ab, edge a'->b'' weighs -l_ab, and no edge returns from the '' copies.  The
 * smoothed upper bound u*_ij is the distance i'->j'; the smoothed lower bound
 * l*_ij is minus the distance i'->j''.  A path i'->j'' runs in the ' copy, takes
 * one -l edge, and ends in the '' copy, so for source i:
 *   1. Dijkstra from i over the u edges gives u*_i. (all weights >= 0);
 *   2. t_b = max_a (l_ab - u*_ia) is the best entry into b'';
 *   3. Dijkstra in the '' copy started from labels -t_b gives -l*_i. .
 * Inputs and outputs are fp64 (exact for Q10 values and for fp32 values on the
 * 1/1024 grid).  rows[] lists the sources; U_out and L_out are nrows x n.
 * With L0 == NULL only the upper rows are produced.
 */
static void dijkstra_dense(const double *W, int64_t n, int64_t ld, double *dist,
                           unsigned char *done)
{
    /* dist[] holds the initial labels on entry and the distances on exit */
    memset(done, 0, (size_t)n);
    for (int64_t it = 0; it < n; ++it) {
        int64_t a = -1;
        double best = 0;
        for (int64_t v = 0; v < n; ++v)
            if (!done[v] && (a < 0 || dist[v] < best)) { a = v; best = dist[v]; }
        done[a] = 1;
        const double *Wa = W + a * ld;
        for (int64_t v = 0; v < n; ++v) {
            if (done[v]) continue;
            double c = best + Wa[v];
            if (c < dist[v]) dist[v] = c;
        }
    }
}

int oracle_closure_rows(const double *U0, const double *L0, int64_t n, int64_t ld,
                        const int64_t *rows, int64_t nrows, double *U_out,
                        double *L_out)
{
    if (n <= 0 || ld < n) return 1;
    int bad = 0;
    _Pragma("omp parallel for schedule(dynamic, 1)")
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = rows[r];
        double *du = U_out + r * n;
        unsigned char *done = (unsigned char *)malloc((size_t)n);
        double *t = (double *)malloc(sizeof(double) * (size_t)n);
        if (!done || !t || i < 0 || i >= n) {
            free(done); free(t);
            _Pragma("omp atomic write") bad = 1;
            continue;
        }
        const double inf = 1.0 / 0.0;
        for (int64_t v = 0; v < n; ++v) du[v] = inf;
        du[i] = 0.0;
        dijkstra_dense(U0, n, ld, du, done);
        if (L0 && L_out) {
            double *dl = L_out + r * n;
            for (int64_t b = 0; b < n; ++b) t[b] = -inf;
            for (int64_t a = 0; a < n; ++a) {
                const double *La = L0 + a * ld;
                const double ua = du[a];
                for (int64_t b = 0; b < n; ++b) {
                    double c = La[b] - ua;
                    if (c > t[b]) t[b] = c;
                }
            }
            for (int64_t b = 0; b < n; ++b) dl[b] = -t[b];
            dijkstra_dense(U0, n, ld, dl, done);
            for (int64_t b = 0; b < n; ++b) dl[b] = -dl[b];
        }
        free(done); free(t);
    }
    return bad ? 1 : 0;
}

/*
 * fp64 closure-rule smoothing with path provenance.
 *
 * Same rounds as oracle_smooth_f64 (ORACLE_RULE_CLOSURE, copies of row and
 * column k taken at the start of round k), and in addition, per cell:
 *   HU[i,j]  edges of a path i -> j whose upper-bound length is U[i,j];
 *   HL[i,j]  edges of a path i' -> j'' (one -l edge, u edges before and after
 *            it) whose length is -L[i,j];
 *   ML[i,j]  the sum of |edge weight| along that path.
 * A candidate formed through k combines the provenance of its two parts
 * (edges add, magnitudes add; a u part contributes its own length, since u
 * weights are >= 0).  Among candidates of equal length the one with fewer
 * edges is kept, so HU and HL are the fewest edges over all shortest paths
 * (lexicographic Floyd-Warshall).  Start: HU = 1 off the diagonal, 0 on it
 * (the empty path); HL = 1 and ML = L0 everywhere (the single -l edge).
 *
 * Why these numbers bound rounding: every value a schedule computes is a
 * rounded sum or difference of two computed values, and rounding is monotone,
 * so the computed upper bound is at most the rounded length of a shortest
 * path, summed in some order, and the computed lower bound at least that of
 * the best lower-bound path.  A sum of h terms rounded in any order is within
 * (h-1) u / (1 - (h-1) u) of the exact sum times the sum of the terms'
 * magnitudes (u = unit roundoff).  U, L: n x n fp64 (row stride ld), updated
 * in place; HU, HL: int32; ML: fp64, all with stride ld.
 */
int oracle_smooth_track_f64(double *U, double *L, int32_t *HU, int32_t *HL, double *ML,
                            int64_t n, int64_t ld)
{
    if (n < 0 || ld < n) return 1;
    if (n == 0) return 0;
    for (int64_t i = 0; i < n; ++i)
        for (int64_t j = 0; j < n; ++j) {
            HU[i * ld + j] = i == j ? 0 : 1;
            HL[i * ld + j] = 1;
            ML[i * ld + j] = L[i * ld + j];
        }
    size_t bytes = sizeof(double) * (size_t)n, ibytes = sizeof(int32_t) * (size_t)n;
    double *urow = malloc(bytes), *ucol = malloc(bytes), *lrow = malloc(bytes),
           *lcol = malloc(bytes), *mrow = malloc(bytes), *mcol = malloc(bytes);
    int32_t *hurow = malloc(ibytes), *hucol = malloc(ibytes), *hlrow = malloc(ibytes),
            *hlcol = malloc(ibytes);
    int rc = 0;
    if (!urow || !ucol || !lrow || !lcol || !mrow || !mcol || !hurow || !hucol || !hlrow ||
        !hlcol) {
        rc = 2;
        goto out;
    }
    for (int64_t k = 0; k < n; ++k) {
        for (int64_t j = 0; j < n; ++j) {
            urow[j] = U[k * ld + j];
            hurow[j] = HU[k * ld + j];
            lrow[j] = L[k * ld + j];
            hlrow[j] = HL[k * ld + j];
            mrow[j] = ML[k * ld + j];
        }
        const double lkk = L[k * ld + k];
        const int32_t hlkk = HL[k * ld + k];
        const double mkk = ML[k * ld + k];
        for (int64_t i = 0; i < n; ++i) {
            ucol[i] = U[i * ld + k];
            hucol[i] = HU[i * ld + k];
            /* the column value, raised through the pair (k, k) */
            double lc = L[i * ld + k], mc = ML[i * ld + k];
            int32_t hc = HL[i * ld + k];
            const double r = lkk - ucol[i];
            const int32_t hr = hlkk + hucol[i];
            if (r > lc || (r == lc && hr < hc)) {
                lc = r;
                hc = hr;
                mc = mkk + ucol[i];
            }
            lcol[i] = lc;
            hlcol[i] = hc;
            mcol[i] = mc;
        }
        _Pragma("omp parallel for schedule(static)")
        for (int64_t i = 0; i < n; ++i) {
            for (int64_t j = 0; j < n; ++j) {
                const int64_t c = i * ld + j;
                const double s = ucol[i] + urow[j];
                const int32_t hs = hucol[i] + hurow[j];
                if (s < U[c] || (s == U[c] && hs < HU[c])) {
                    U[c] = s;
                    HU[c] = hs;
                }
                /* l_kj - u_ik, then lc_i - u_kj */
                const double a = lrow[j] - ucol[i];
                const int32_t ha = hlrow[j] + hucol[i];
                const double b = lcol[i] - urow[j];
                const int32_t hb = hlcol[i] + hurow[j];
                if (a > L[c] || (a == L[c] && ha < HL[c])) {
                    L[c] = a;
                    HL[c] = ha;
                    ML[c] = mrow[j] + ucol[i];
                }
                if (b > L[c] || (b == L[c] && hb < HL[c])) {
                    L[c] = b;
                    HL[c] = hb;
                    ML[c] = mcol[i] + urow[j];
                }
            }
        }
    }
out:
    free(urow); free(ucol); free(lrow); free(lcol); free(mrow); free(mcol);
    free(hurow); free(hucol); free(hlrow); free(hlcol);
    return rc;
}
