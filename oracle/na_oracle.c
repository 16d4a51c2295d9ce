/*
 * na_oracle.c -- plain fp64 CPU oracle for multi-dimensional neighborhood attention (NA),
 * forward and analytic backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load this library.  The product path (the CUDA library) never calls it,
 * and the two share no source, header, table or helper.
 *
 * What it computes (one (batch, head) pair at a time, every quantity in double precision):
 *
 *   Neighbourhood.  The pages ("Backward pass is very slow towards much tokens and large
 *   kernels", NATTEN issue #161: the user's benchmark script and the maintainer's reply about
 *   the cubic receptive field of each query) use na2d/na3d(query, key, value, kernel_size, dilation) but never
 *   write the window down.  The reading taken here, per spatial axis of length L with odd kernel
 *   size k (r = k/2) and dilation d:
 *     query index i belongs to residue class c = i mod d, at class index j = i div d;
 *     the class holds Lc = ceil((L - c) / d) positions;
 *     the window starts at class index s = clamp(j - r, 0, Lc - k) (shifted, never truncated,
 *     at the borders), and the neighbours are c + d*(s + t), t = 0..k-1.
 *   The neighbour set of a multi-dimensional query is the Cartesian product over the axes, so
 *   every query sees exactly prod(k) keys.
 *
 *   Forward (the unfused decomposition in the user's script: na*_qk -> softmax -> na*_av):
 *     S_ij = scale * <q_i, k_j>  for j in N(i)
 *     m_i = max_j S_ij,  l_i = sum_j exp(S_ij - m_i),  P_ij = exp(S_ij - m_i) / l_i
 *     O_i = sum_j P_ij v_j,  LSE_i = m_i + ln(l_i)   (natural log)
 *
 *   Backward for an upstream gradient dO (the script's loss = output.sum() gives dO = 1):
 *     Delta_i = <dO_i, O_i>            (the "ComputeDelta" step of the maintainer's profile)
 *     dP_ij = <dO_i, v_j>,  dS_ij = P_ij (dP_ij - Delta_i)
 *     dQ_i = scale * sum_{j in N(i)} dS_ij k_j
 *     dK_j = scale * sum_{i : j in N(i)} dS_ij q_i,   dV_j = sum_{i : j in N(i)} P_ij dO_i
 *   The key-side sums visit every query of the same residue class within (k-1)*d positions per
 *   axis and keep those whose neighbour set contains the key (a direct membership test, no
 *   inverse-window formula).
 *
 * Tensors are contiguous [B, L1, .., Ln, heads, D]; a "row" is one (batch, token, head) triple,
 * numbered ((b * N + token) * heads + head) with token the row-major spatial index.
 * Inputs are read as float32, as bfloat16 bit patterns (widened exactly to float32, then to
 * double), or as float64 (finite-difference checks), so the oracle sees the very values the
 * device path sees.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NA_ORACLE_MAXDIM 3

typedef struct {
    int B, ndim, heads, D;
    int L[NA_ORACLE_MAXDIM], k[NA_ORACLE_MAXDIM], d[NA_ORACLE_MAXDIM];
    int64_t N;      /* tokens per batch entry */
    int64_t K;      /* keys per query */
    double scale;
    int in_kind;    /* 0: float32, 1: bfloat16 bit patterns, 2: float64 */
} geom_t;

/* ------------------------------------------------------------------------------------------ */
/* Input access                                                                                 */
/* ------------------------------------------------------------------------------------------ */

static double in_val(const void* base, int64_t idx, int in_kind) {
    if (in_kind == 2) return ((const double*)base)[idx];
    if (in_kind == 1) {
        uint32_t bits = (uint32_t)((const uint16_t*)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float*)base)[idx];
}

/* element offset of (row, channel 0) */
static int64_t row_off(const geom_t* g, int64_t row) { return row * (int64_t)g->D; }

static double dot_rows(const geom_t* g, const void* a, int64_t ra, const void* b, int64_t rb) {
    double acc = 0.0;
    int64_t oa = row_off(g, ra), ob = row_off(g, rb);
    for (int c = 0; c < g->D; ++c) acc += in_val(a, oa + c, g->in_kind) * in_val(b, ob + c, g->in_kind);
    return acc;
}

/* ------------------------------------------------------------------------------------------ */
/* Neighbourhood                                                                                */
/* ------------------------------------------------------------------------------------------ */

/* Spatial index of the first neighbour of spatial index i on one axis. */
static int first_neighbour(int i, int L, int k, int d) {
    int c = i % d, j = i / d;
    int Lc = (L - c + d - 1) / d;
    int s = j - k / 2;
    if (s > Lc - k) s = Lc - k;
    if (s < 0) s = 0;
    return c + d * s;
}

/* Does the window of spatial index i (one axis) contain spatial index p? */
static int axis_contains(int i, int p, int L, int k, int d) {
    if (p % d != i % d) return 0;
    int f = first_neighbour(i, L, k, d);
    return p >= f && p <= f + d * (k - 1);
}

static void token_coords(const geom_t* g, int64_t tok, int* x) {
    for (int a = g->ndim - 1; a >= 0; --a) { x[a] = (int)(tok % g->L[a]); tok /= g->L[a]; }
}

static int64_t token_index(const geom_t* g, const int* x) {
    int64_t t = 0;
    for (int a = 0; a < g->ndim; ++a) t = t * g->L[a] + x[a];
    return t;
}

/* List the K neighbour rows of query row `row` (Cartesian product, axis 1 slowest). */
static void neighbour_rows(const geom_t* g, int64_t row, int64_t* out) {
    int64_t h = row % g->heads, bt = row / g->heads;
    int64_t b = bt / g->N, tok = bt % g->N;
    int x[NA_ORACLE_MAXDIM], f[NA_ORACLE_MAXDIM], t[NA_ORACLE_MAXDIM], p[NA_ORACLE_MAXDIM];
    token_coords(g, tok, x);
    for (int a = 0; a < g->ndim; ++a) { f[a] = first_neighbour(x[a], g->L[a], g->k[a], g->d[a]); t[a] = 0; }
    for (int64_t n = 0; n < g->K; ++n) {
        for (int a = 0; a < g->ndim; ++a) p[a] = f[a] + g->d[a] * t[a];
        out[n] = ((b * g->N) + token_index(g, p)) * g->heads + h;
        for (int a = g->ndim - 1; a >= 0; --a) {       /* odometer step over the window */
            if (++t[a] < g->k[a]) break;
            t[a] = 0;
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Forward of one query row                                                                     */
/* ------------------------------------------------------------------------------------------ */

typedef struct { double lse, delta; } qstats_t;

/* O (D values), LSE of one query row.  `nb` and `s` are caller scratch of K entries. */
static void forward_row(const geom_t* g, const void* q, const void* k, const void* v, int64_t row,
                        int64_t* nb, double* s, double* o, double* lse) {
    neighbour_rows(g, row, nb);
    double m = -INFINITY;
    for (int64_t n = 0; n < g->K; ++n) {
        s[n] = g->scale * dot_rows(g, q, row, k, nb[n]);
        if (s[n] > m) m = s[n];
    }
    double l = 0.0;
    for (int64_t n = 0; n < g->K; ++n) l += exp(s[n] - m);
    for (int c = 0; c < g->D; ++c) o[c] = 0.0;
    for (int64_t n = 0; n < g->K; ++n) {
        double p = exp(s[n] - m) / l;
        int64_t ov = row_off(g, nb[n]);
        for (int c = 0; c < g->D; ++c) o[c] += p * in_val(v, ov + c, g->in_kind);
    }
    *lse = m + log(l);
}

/* ------------------------------------------------------------------------------------------ */
/* Validation                                                                                   */
/* ------------------------------------------------------------------------------------------ */

static int make_geom(geom_t* g, int B, int ndim, const int* L, int heads, int D, const int* ks,
                     const int* dil, double scale, int in_kind) {
    if (in_kind < 0 || in_kind > 2) return -1;
    if (ndim < 1 || ndim > NA_ORACLE_MAXDIM || B < 1 || heads < 1 || D < 1) return -1;
    memset(g, 0, sizeof *g);
    g->B = B; g->ndim = ndim; g->heads = heads; g->D = D; g->scale = scale; g->in_kind = in_kind;
    g->N = 1; g->K = 1;
    for (int a = 0; a < ndim; ++a) {
        if (L[a] < 1 || ks[a] < 1 || ks[a] % 2 == 0 || dil[a] < 1) return -1;
        if (L[a] / dil[a] < ks[a]) return -1;   /* every residue class needs k positions */
        g->L[a] = L[a]; g->k[a] = ks[a]; g->d[a] = dil[a];
        g->N *= L[a]; g->K *= ks[a];
    }
    return 0;
}

static int cmp_i64(const void* a, const void* b) {
    int64_t x = *(const int64_t*)a, y = *(const int64_t*)b;
    return (x > y) - (x < y);
}

static int64_t find_row(const int64_t* list, int64_t n, int64_t row) {
    int64_t lo = 0, hi = n - 1;
    while (lo <= hi) {
        int64_t mid = (lo + hi) / 2;
        if (list[mid] == row) return mid;
        if (list[mid] < row) lo = mid + 1; else hi = mid - 1;
    }
    return -1;
}

/* ------------------------------------------------------------------------------------------ */
/* Exported API                                                                                 */
/* ------------------------------------------------------------------------------------------ */

/* Spatial index of the first neighbour of i on one axis (exposed for the neighbourhood pins). */
int na_oracle_first_neighbour(int i, int L, int k, int d) {
    if (L < 1 || k < 1 || k % 2 == 0 || d < 1 || L / d < k || i < 0 || i >= L) return -1;
    return first_neighbour(i, L, k, d);
}

/*
 * Forward for the listed rows (rows == NULL: every row, nrows = B*N*heads).
 * o: nrows*D doubles, lse: nrows doubles.  Returns 0, or -1 on invalid arguments.
 */
int na_oracle_fwd(const void* q, const void* k, const void* v, int in_kind,
                  int B, int ndim, const int* L, int heads, int D,
                  const int* ks, const int* dil, double scale,
                  const int64_t* rows, int64_t nrows, double* o, double* lse, int nthreads) {
    geom_t g;
    if (make_geom(&g, B, ndim, L, heads, D, ks, dil, scale, in_kind)) return -1;
    int64_t total = (int64_t)B * g.N * heads;
    if (!rows && nrows != total) return -1;
    if (nthreads <= 0) nthreads = 1;
    int bad = 0;
#pragma omp parallel num_threads(nthreads)
    {
        int64_t* nb = (int64_t*)malloc(sizeof(int64_t) * g.K);
        double* s = (double*)malloc(sizeof(double) * g.K);
        if (!nb || !s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 64)
            for (int64_t n = 0; n < nrows; ++n) {
                int64_t row = rows ? rows[n] : n;
                if (row < 0 || row >= total) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                forward_row(&g, q, k, v, row, nb, s, o + n * D, lse + n);
            }
        }
        free(nb);
        free(s);
    }
    return bad ? -1 : 0;
}

/*
 * Backward.  dQ for the rows in qrows (nq of them; qrows == NULL: all rows) into dq (nq*D),
 * dK and dV for the rows in krows (nk; krows == NULL: all rows) into dk, dv (nk*D each).
 * Any of dq / dk,dv may be skipped by passing nq = 0 / nk = 0.
 */
int na_oracle_bwd(const void* q, const void* k, const void* v, const void* dO, int in_kind,
                  int B, int ndim, const int* L, int heads, int D,
                  const int* ks, const int* dil, double scale,
                  const int64_t* qrows, int64_t nq, double* dq,
                  const int64_t* krows, int64_t nk, double* dk, double* dv, int nthreads) {
    geom_t g;
    if (make_geom(&g, B, ndim, L, heads, D, ks, dil, scale, in_kind)) return -1;
    int64_t total = (int64_t)B * g.N * heads;
    if ((!qrows && nq != 0 && nq != total) || (!krows && nk != 0 && nk != total)) return -1;
    if (nthreads <= 0) nthreads = 1;

    /* Queries whose softmax statistics are needed: the dQ rows, and every query that attends a
       dK/dV row.  Collected with duplicates, then sorted and made unique. */
    int64_t span = 1;                         /* candidate queries per key */
    for (int a = 0; a < ndim; ++a) span *= 2 * g.k[a] - 1;
    int all_q = (!qrows && nq == total) || (!krows && nk == total);
    int64_t nneed = 0;
    int64_t* need = NULL;
    if (all_q) {
        need = (int64_t*)malloc(sizeof(int64_t) * (total > 0 ? total : 1));
        if (!need) return -1;
        for (int64_t r = 0; r < total; ++r) need[r] = r;
        nneed = total;
    } else {
        int64_t cap = nq + nk * span;
        need = (int64_t*)malloc(sizeof(int64_t) * (cap > 0 ? cap : 1));
        if (!need) return -1;
        for (int64_t n = 0; n < nq; ++n) {
            if (qrows[n] < 0 || qrows[n] >= total) { free(need); return -1; }
            need[nneed++] = qrows[n];
        }
        for (int64_t n = 0; n < nk; ++n) {
            int64_t kr = krows[n];
            if (kr < 0 || kr >= total) { free(need); return -1; }
            int64_t h = kr % heads, bt = kr / heads, b = bt / g.N;
            int x[NA_ORACLE_MAXDIM], off[NA_ORACLE_MAXDIM], p[NA_ORACLE_MAXDIM];
            token_coords(&g, bt % g.N, x);
            for (int a = 0; a < ndim; ++a) off[a] = -(g.k[a] - 1);
            for (int64_t c = 0; c < span; ++c) {
                int inside = 1;
                for (int a = 0; a < ndim; ++a) {
                    p[a] = x[a] + off[a] * g.d[a];
                    if (p[a] < 0 || p[a] >= g.L[a]) inside = 0;
                }
                if (inside) need[nneed++] = ((b * g.N) + token_index(&g, p)) * heads + h;
                for (int a = ndim - 1; a >= 0; --a) {
                    if (++off[a] <= g.k[a] - 1) break;
                    off[a] = -(g.k[a] - 1);
                }
            }
        }
        qsort(need, (size_t)nneed, sizeof(int64_t), cmp_i64);
        int64_t u = 0;
        for (int64_t n = 0; n < nneed; ++n)
            if (u == 0 || need[n] != need[u - 1]) need[u++] = need[n];
        nneed = u;
    }

    qstats_t* st = (qstats_t*)malloc(sizeof(qstats_t) * (nneed > 0 ? nneed : 1));
    if (!st) { free(need); return -1; }
    int bad = 0;

#pragma omp parallel num_threads(nthreads)
    {
        int64_t* nb = (int64_t*)malloc(sizeof(int64_t) * g.K);
        double* s = (double*)malloc(sizeof(double) * g.K);
        double* o = (double*)malloc(sizeof(double) * D);
        if (!nb || !s || !o) {
#pragma omp atomic write
            bad = 1;
        }
        /* 1. LSE and Delta = <dO, O> of every needed query */
#pragma omp for schedule(dynamic, 64)
        for (int64_t n = 0; n < nneed; ++n) {
            if (!nb || !s || !o) continue;
            double lse;
            forward_row(&g, q, k, v, need[n], nb, s, o, &lse);
            double delta = 0.0;
            int64_t od = row_off(&g, need[n]);
            for (int c = 0; c < D; ++c) delta += in_val(dO, od + c, in_kind) * o[c];
            st[n].lse = lse;
            st[n].delta = delta;
        }
        /* 2. dQ: gather over the query's own window */
#pragma omp for schedule(dynamic, 64)
        for (int64_t n = 0; n < nq; ++n) {
            if (!nb || !s || !o) continue;
            int64_t row = qrows ? qrows[n] : n;
            int64_t si = find_row(need, nneed, row);
            double* out = dq + n * D;
            for (int c = 0; c < D; ++c) out[c] = 0.0;
            if (si < 0) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            neighbour_rows(&g, row, nb);
            for (int64_t m = 0; m < g.K; ++m) {
                double p = exp(scale * dot_rows(&g, q, row, k, nb[m]) - st[si].lse);
                double dp = dot_rows(&g, dO, row, v, nb[m]);
                double ds = p * (dp - st[si].delta);
                int64_t ok = row_off(&g, nb[m]);
                for (int c = 0; c < D; ++c) out[c] += ds * in_val(k, ok + c, in_kind);
            }
            for (int c = 0; c < D; ++c) out[c] *= scale;
        }
        /* 3. dK, dV: gather over every query whose window holds the key */
#pragma omp for schedule(dynamic, 64)
        for (int64_t n = 0; n < nk; ++n) {
            int64_t kr = krows ? krows[n] : n;
            double* ok_ = dk + n * D;
            double* ov_ = dv + n * D;
            for (int c = 0; c < D; ++c) { ok_[c] = 0.0; ov_[c] = 0.0; }
            int64_t h = kr % heads, bt = kr / heads, b = bt / g.N;
            int x[NA_ORACLE_MAXDIM], off[NA_ORACLE_MAXDIM], p[NA_ORACLE_MAXDIM];
            token_coords(&g, bt % g.N, x);
            for (int a = 0; a < ndim; ++a) off[a] = -(g.k[a] - 1);
            for (int64_t c = 0; c < span; ++c) {
                int inside = 1;
                for (int a = 0; a < ndim; ++a) {
                    p[a] = x[a] + off[a] * g.d[a];
                    if (p[a] < 0 || p[a] >= g.L[a]) inside = 0;
                }
                if (inside) {
                    int member = 1;
                    for (int a = 0; a < ndim; ++a)
                        if (!axis_contains(p[a], x[a], g.L[a], g.k[a], g.d[a])) member = 0;
                    if (member) {
                        int64_t qr = ((b * g.N) + token_index(&g, p)) * heads + h;
                        int64_t si = find_row(need, nneed, qr);
                        if (si < 0) {
#pragma omp atomic write
                            bad = 1;
                        } else {
                            double pij = exp(scale * dot_rows(&g, q, qr, k, kr) - st[si].lse);
                            double dp = dot_rows(&g, dO, qr, v, kr);
                            double ds = pij * (dp - st[si].delta);
                            int64_t oq = row_off(&g, qr);
                            for (int e = 0; e < D; ++e) {
                                ov_[e] += pij * in_val(dO, oq + e, in_kind);
                                ok_[e] += ds * in_val(q, oq + e, in_kind);
                            }
                        }
                    }
                }
                for (int a = ndim - 1; a >= 0; --a) {
                    if (++off[a] <= g.k[a] - 1) break;
                    off[a] = -(g.k[a] - 1);
                }
            }
            for (int e = 0; e < D; ++e) ok_[e] *= scale;
        }
        free(nb);
        free(s);
        free(o);
    }
    free(st);
    free(need);
    return bad ? -1 : 0;
}

int na_oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
