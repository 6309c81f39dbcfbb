/*
 * oracle.c - plain, slow, obviously correct CPU reference for one partition's
 * GCN / GraphSAGE layer, forward and backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this code.  The CUDA library shares no
 * code, header, table or helper with it.
 *
 * All floating-point work is done in double precision (inputs are widened from
 * their stored fp32 / bf16 values by the Python wrapper).  Loops follow the
 * definitions in the order the pages state them; there is no blocking, fusion
 * or reordering beyond that.  Parallelism, where present, is an OpenMP loop
 * over independent output rows; each output row is summed in a fixed order
 * (CSR order), so results do not depend on the thread count.
 *
 * Notation (CAGNET page, "Reducing Communication in Graph Neural Network
 * Training", GNN background section): A is the n x n adjacency with self loops,
 * normalised as D^-1/2 (A + I) D^-1/2 with D the modified (self-loop) degrees;
 * a layer computes H^(l) = sigma(A^T H^(l-1) W^l).  One partition holds the
 * block of rows of its local vertices; its columns are the local vertices
 * followed by the HALO vertices (Sylvie page, "Graph Engine" and Fig. 3).  Row
 * v of the block lists the vertices u whose features v aggregates.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

#define OK 0
#define ERR_INDEX 5

/* ------------------------------------------------------------------------ */
/* stale-representation table: pull and push                                 */
/* DIGEST page, "Distributed Graph Neural Network Training with Periodic     */
/* Stale Representation Synchronization", system design (Fig. 1c):           */
/* pull   H_out <- H~_out  (halo rows are read from the table),              */
/* push   H_in  -> H~_in   (fresh local rows are written to the table).      */
/* ------------------------------------------------------------------------ */

/* H[n_local + i, 0:f] = T[halo_ids[i], 0:f] for i < n_halo (element size es
 * bytes).  Rows whose id lies outside [0, n_table) are not written and the
 * call returns ERR_INDEX. */
int oracle_halo_pull(const void *table, int64_t ld_t, int64_t n_table, const int64_t *halo_ids, int64_t n_halo,
                     void *H, int64_t ld_h, int64_t n_local, int64_t f, int es) {
    int status = OK;
    for (int64_t i = 0; i < n_halo; ++i) {
        int64_t id = halo_ids[i];
        if (id < 0 || id >= n_table) { status = ERR_INDEX; continue; }
        const char *src = (const char *)table + (size_t)id * (size_t)ld_t * (size_t)es;
        char *dst = (char *)H + (size_t)(n_local + i) * (size_t)ld_h * (size_t)es;
        for (int64_t j = 0; j < f * es; ++j) dst[j] = src[j];
    }
    return status;
}

/* T[local_ids[v], 0:f] = H[v, 0:f] for v < n_local.  The partition's vertex
 * sets do not overlap (DIGEST page, complexity analysis), so an id that occurs
 * twice is an error: every row carrying a repeated id is left unwritten, as is
 * every row whose id lies outside [0, n_table); the call then returns ERR_INDEX. */
int oracle_halo_push(const void *H, int64_t ld_h, int64_t n_local, int64_t f, const int64_t *local_ids, void *table,
                     int64_t ld_t, int64_t n_table, int es) {
    int status = OK;
    int32_t *count = (int32_t *)calloc((size_t)(n_table > 0 ? n_table : 1), sizeof(int32_t));
    if (!count) return -1;
    for (int64_t v = 0; v < n_local; ++v) {
        int64_t id = local_ids[v];
        if (id >= 0 && id < n_table) count[id]++;
    }
    for (int64_t v = 0; v < n_local; ++v) {
        int64_t id = local_ids[v];
        if (id < 0 || id >= n_table || count[id] != 1) { status = ERR_INDEX; continue; }
        const char *src = (const char *)H + (size_t)v * (size_t)ld_h * (size_t)es;
        char *dst = (char *)table + (size_t)id * (size_t)ld_t * (size_t)es;
        for (int64_t j = 0; j < f * es; ++j) dst[j] = src[j];
    }
    free(count);
    return status;
}

/* ------------------------------------------------------------------------ */
/* degrees                                                                   */
/* ------------------------------------------------------------------------ */

/* dinv[x] = deg[x]^-1/2 for the n_local + n_halo columns.  When deg is NULL the
 * partition can only see its own block: a local vertex's degree is its row
 * length (the self loop included) and a halo vertex's degree is one (its own
 * self loop) plus the number of times its column occurs in the block.  A
 * degree of zero gives dinv = 0. */
void oracle_gcn_dinv(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo, const float *deg,
                     double *dinv) {
    int64_t nT = n_local + n_halo;
    if (deg) {
        for (int64_t x = 0; x < nT; ++x) dinv[x] = deg[x] > 0.0f ? 1.0 / sqrt((double)deg[x]) : 0.0;
        return;
    }
    double *d = (double *)calloc((size_t)(nT > 0 ? nT : 1), sizeof(double));
    for (int64_t v = 0; v < n_local; ++v) d[v] = (double)(rowptr[v + 1] - rowptr[v]);
    for (int64_t u = n_local; u < nT; ++u) d[u] = 1.0;
    for (int64_t e = 0; e < rowptr[n_local]; ++e)
        if (colidx[e] >= n_local) d[colidx[e]] += 1.0;
    for (int64_t x = 0; x < nT; ++x) dinv[x] = d[x] > 0.0 ? 1.0 / sqrt(d[x]) : 0.0;
    free(d);
}

/* GraphSAGE mean weights: inv_cnt[v] = 1 / |N(v) \ {v}| over the entries of row
 * v whose column is not v itself; 0 when the row has no such entry. */
void oracle_sage_invcnt(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, double *inv_cnt) {
    for (int64_t v = 0; v < n_local; ++v) {
        int64_t c = 0;
        for (int64_t e = rowptr[v]; e < rowptr[v + 1]; ++e)
            if (colidx[e] != v) ++c;
        inv_cnt[v] = c > 0 ? 1.0 / (double)c : 0.0;
    }
}

/* ------------------------------------------------------------------------ */
/* forward aggregation                                                       */
/* ------------------------------------------------------------------------ */

/* Rows to compute: rows[k] for k < n_rows, or all local rows when rows == NULL.
 * Input rows: H[hmap[c]] for column c (hmap == NULL: H[c]).  Output row k of Z
 * (ld_z) belongs to rows[k]. */
static inline int64_t row_at(const int64_t *rows, int64_t k) { return rows ? rows[k] : k; }
static inline int64_t map_at(const int64_t *hmap, int64_t c) { return hmap ? hmap[c] : c; }

/* GCN (symmetric normalisation, Sylvie Alg. 1 matrix form; CAGNET GNN section):
 * Z[v] = sum over entries u of row v of dinv[v] * dinv[u] * H[u]. */
void oracle_gcn_aggregate(const int32_t *rowptr, const int32_t *colidx, const double *dinv, const double *H,
                          int64_t ld_h, const int64_t *hmap, int64_t f, const int64_t *rows, int64_t n_rows, double *Z,
                          int64_t ld_z) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t k = 0; k < n_rows; ++k) {
        int64_t v = row_at(rows, k);
        double *z = Z + (size_t)k * (size_t)ld_z;
        for (int64_t j = 0; j < f; ++j) z[j] = 0.0;
        for (int64_t e = rowptr[v]; e < rowptr[v + 1]; ++e) {
            int64_t u = colidx[e];
            double w = dinv[v] * dinv[u];
            const double *h = H + (size_t)map_at(hmap, u) * (size_t)ld_h;
            for (int64_t j = 0; j < f; ++j) z[j] += w * h[j];
        }
    }
}

/* GraphSAGE mean with self concatenation (Sylvie page names GraphSAGE; its
 * formula is not in the text, so this is the textbook mean + concat form):
 * Z[v] = [ H[v] , inv_cnt[v] * sum over entries u != v of row v of H[u] ].
 * The second half starts at column half_off of Z. */
void oracle_sage_aggregate(const int32_t *rowptr, const int32_t *colidx, const double *inv_cnt, const double *H,
                           int64_t ld_h, const int64_t *hmap, int64_t f, const int64_t *rows, int64_t n_rows, double *Z,
                           int64_t ld_z, int64_t half_off) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t k = 0; k < n_rows; ++k) {
        int64_t v = row_at(rows, k);
        double *z = Z + (size_t)k * (size_t)ld_z;
        const double *hv = H + (size_t)map_at(hmap, v) * (size_t)ld_h;
        for (int64_t j = 0; j < f; ++j) z[j] = hv[j];
        double *m = z + half_off;
        for (int64_t j = 0; j < f; ++j) m[j] = 0.0;
        for (int64_t e = rowptr[v]; e < rowptr[v + 1]; ++e) {
            int64_t u = colidx[e];
            if (u == v) continue;
            const double *h = H + (size_t)map_at(hmap, u) * (size_t)ld_h;
            for (int64_t j = 0; j < f; ++j) m[j] += h[j];
        }
        for (int64_t j = 0; j < f; ++j) m[j] *= inv_cnt[v];
    }
}

/* ------------------------------------------------------------------------ */
/* dense update (CAGNET GNN section: H^(l) = sigma(A^T H^(l-1) W^l))         */
/* ------------------------------------------------------------------------ */

/* Y = Z W (Z: n x K, W: K x N row-major); Hout = relu ? max(Y, 0) : Y. */
void oracle_update(const double *Z, int64_t ld_z, int64_t n, int64_t K, const double *W, int64_t N, int relu,
                   double *Hout, int64_t ld_o) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k) acc += Z[(size_t)i * ld_z + k] * W[(size_t)k * N + j];
            Hout[(size_t)i * ld_o + j] = (relu && !(acc > 0.0)) ? 0.0 : acc;
        }
    }
}

/* Backward of the update by the chain rule (the CAGNET page's own derivation
 * is not in the text).  dY = G * 1[Hout > 0] when relu (ReLU'(0) = 0), else G;
 * dZ = dY W^T (n x K) when dZ != NULL. */
void oracle_update_backward_dz(const double *G, int64_t ld_g, const double *Hout, int64_t ld_h, int64_t n, int64_t N,
                               int relu, const double *W, int64_t K, double *dZ, int64_t ld_dz) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        for (int64_t k = 0; k < K; ++k) {
            double acc = 0.0;
            for (int64_t j = 0; j < N; ++j) {
                double g = G[(size_t)i * ld_g + j];
                if (relu && !(Hout[(size_t)i * ld_h + j] > 0.0)) g = 0.0;
                acc += g * W[(size_t)k * N + j];
            }
            dZ[(size_t)i * ld_dz + k] = acc;
        }
    }
}

/* dW = Z^T dY (K x N), summed over rows i in increasing order. */
void oracle_update_backward_dw(const double *G, int64_t ld_g, const double *Hout, int64_t ld_h, const double *Z,
                               int64_t ld_z, int64_t n, int64_t K, int64_t N, int relu, double *dW) {
#pragma omp parallel for schedule(static)
    for (int64_t k = 0; k < K; ++k) {
        for (int64_t j = 0; j < N; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i < n; ++i) {
                double g = G[(size_t)i * ld_g + j];
                if (relu && !(Hout[(size_t)i * ld_h + j] > 0.0)) g = 0.0;
                acc += Z[(size_t)i * ld_z + k] * g;
            }
            dW[(size_t)k * N + j] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* graph attention (GAT): the Sylvie page names GAT among the models it       */
/* trains and the DIGEST page benchmarks it; neither prints its formula, so   */
/* this is the textbook single-head layer (Velickovic et al., ICLR 2018)      */
/* ------------------------------------------------------------------------ */

/* For every row v and entry u of row v (the self loop is an entry of A + I):
 *   z_vu = s_dst[v] + s_src[u],  e_vu = z_vu if z_vu > 0 else slope * z_vu,
 *   alpha_vu = exp(e_vu) / sum over the row's entries u' of exp(e_vu'),
 *   Y[v] = sum_u alpha_vu T[u].
 * alpha is written per entry (CSR order), Y for the n_local rows. */
void oracle_gat_attend(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, const double *s_src,
                       const double *s_dst, const double *T, int64_t ld_t, int64_t f, double slope, double *alpha,
                       double *Y, int64_t ld_y) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t v = 0; v < n_local; ++v) {
        double *y = Y + (size_t)v * (size_t)ld_y;
        for (int64_t j = 0; j < f; ++j) y[j] = 0.0;
        const int32_t b = rowptr[v], e = rowptr[v + 1];
        if (e == b) continue;
        double mx = -HUGE_VAL;
        for (int32_t k = b; k < e; ++k) {
            double z = s_dst[v] + s_src[colidx[k]];
            double a = z > 0.0 ? z : slope * z;
            alpha[k] = a;
            if (a > mx) mx = a;
        }
        double sum = 0.0;
        for (int32_t k = b; k < e; ++k) {
            alpha[k] = exp(alpha[k] - mx);
            sum += alpha[k];
        }
        for (int32_t k = b; k < e; ++k) {
            alpha[k] /= sum;
            const double *t = T + (size_t)colidx[k] * (size_t)ld_t;
            for (int64_t j = 0; j < f; ++j) y[j] += alpha[k] * t[j];
        }
    }
}

/* Backward of oracle_gat_attend by the chain rule, given dY (n_local rows):
 *   dT[u]     = sum over entries (v, u) of alpha_vu dY[v]
 *   dalpha_vu = dY[v] . T[u]
 *   de_vu     = alpha_vu (dalpha_vu - sum over the row's u' of alpha_vu' dalpha_vu')
 *   dz_vu     = de_vu (z_vu > 0 ? 1 : slope)
 *   ds_dst[v] = sum_u dz_vu,   ds_src[u] = sum over entries (v, u) of dz_vu
 * dT (n_total rows) and ds_src (n_total), ds_dst (n_local) are overwritten.
 * Rows are taken one after another (the scatter into dT and ds_src is a plain
 * loop, no parallelism). */
void oracle_gat_attend_backward(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_total,
                                const double *s_src, const double *s_dst, const double *T, int64_t ld_t, int64_t f,
                                double slope, const double *alpha, const double *dY, int64_t ld_dy, double *dT,
                                int64_t ld_dt, double *ds_src, double *ds_dst) {
    for (int64_t u = 0; u < n_total; ++u) {
        double *d = dT + (size_t)u * (size_t)ld_dt;
        for (int64_t j = 0; j < f; ++j) d[j] = 0.0;
        ds_src[u] = 0.0;
    }
    for (int64_t v = 0; v < n_local; ++v) {
        const double *dy = dY + (size_t)v * (size_t)ld_dy;
        const int32_t b = rowptr[v], e = rowptr[v + 1];
        double dot_sum = 0.0;
        for (int32_t k = b; k < e; ++k) {
            const double *t = T + (size_t)colidx[k] * (size_t)ld_t;
            double da = 0.0;
            for (int64_t j = 0; j < f; ++j) da += dy[j] * t[j];
            dot_sum += alpha[k] * da;
        }
        double sd = 0.0;
        for (int32_t k = b; k < e; ++k) {
            const int64_t u = colidx[k];
            const double *t = T + (size_t)u * (size_t)ld_t;
            double da = 0.0;
            for (int64_t j = 0; j < f; ++j) da += dy[j] * t[j];
            const double de = alpha[k] * (da - dot_sum);
            const double z = s_dst[v] + s_src[u];
            const double dz = de * (z > 0.0 ? 1.0 : slope);
            sd += dz;
            ds_src[u] += dz;
            double *d = dT + (size_t)u * (size_t)ld_dt;
            for (int64_t j = 0; j < f; ++j) d[j] += alpha[k] * dy[j];
        }
        ds_dst[v] = sd;
    }
}

/* ------------------------------------------------------------------------ */
/* transpose of the block (CAGNET: A and A^T are kept apart explicitly)      */
/* ------------------------------------------------------------------------ */

typedef struct {
    int32_t col, row, e;
} trip_t;

static int cmp_trip(const void *x, const void *y) {
    const trip_t *a = (const trip_t *)x, *b = (const trip_t *)y;
    if (a->col != b->col) return a->col < b->col ? -1 : 1;
    if (a->row != b->row) return a->row < b->row ? -1 : 1;
    if (a->e != b->e) return a->e < b->e ? -1 : 1;
    return 0;
}

/* Transpose of the n_local x n_total block: row c of the transpose lists the
 * block rows v that hold column c, ascending (ties by original entry order);
 * permT[k] is the block entry that transpose entry k came from.  Computed by
 * sorting (col, row, entry) triples. */
int oracle_transpose(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_total,
                     int32_t *rowptrT, int32_t *colidxT, int32_t *permT) {
    int64_t nnz = rowptr[n_local];
    trip_t *t = (trip_t *)malloc((size_t)(nnz > 0 ? nnz : 1) * sizeof(trip_t));
    if (!t) return -1;
    for (int64_t v = 0; v < n_local; ++v)
        for (int64_t e = rowptr[v]; e < rowptr[v + 1]; ++e) {
            t[e].col = colidx[e];
            t[e].row = (int32_t)v;
            t[e].e = (int32_t)e;
        }
    qsort(t, (size_t)nnz, sizeof(trip_t), cmp_trip);
    for (int64_t c = 0; c <= n_total; ++c) rowptrT[c] = 0;
    for (int64_t k = 0; k < nnz; ++k) rowptrT[t[k].col + 1]++;
    for (int64_t c = 0; c < n_total; ++c) rowptrT[c + 1] += rowptrT[c];
    for (int64_t k = 0; k < nnz; ++k) {
        colidxT[k] = t[k].row;
        permT[k] = t[k].e;
    }
    free(t);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* backward aggregation over the transpose                                   */
/* ------------------------------------------------------------------------ */

/* GCN: dH[u] = sum over entries v of transpose row u of dinv[v] * dinv[u] * dZ[v]
 * for the output rows rows[k] (u in [0, n_total); rows == NULL: all n_rows
 * rows from 0).  dZ row v is dZ[dmap[v]] (dmap == NULL: dZ[v]). */
void oracle_gcn_aggregate_backward(const int32_t *rowptrT, const int32_t *colidxT, const double *dinv,
                                   const double *dZ, int64_t ld_dz, const int64_t *dmap, int64_t f,
                                   const int64_t *rows, int64_t n_rows, double *dH, int64_t ld_dh) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t k = 0; k < n_rows; ++k) {
        int64_t u = row_at(rows, k);
        double *o = dH + (size_t)k * (size_t)ld_dh;
        for (int64_t j = 0; j < f; ++j) o[j] = 0.0;
        for (int64_t e = rowptrT[u]; e < rowptrT[u + 1]; ++e) {
            int64_t v = colidxT[e];
            double w = dinv[v] * dinv[u];
            const double *g = dZ + (size_t)map_at(dmap, v) * (size_t)ld_dz;
            for (int64_t j = 0; j < f; ++j) o[j] += w * g[j];
        }
    }
}

/* GraphSAGE: dZ = [dZ_self | dZ_mean] (the mean half at column half_off).
 * dH[u] = (u < n_local ? dZ_self[u] : 0)
 *       + sum over entries v != u of transpose row u of inv_cnt[v] * dZ_mean[v]. */
void oracle_sage_aggregate_backward(const int32_t *rowptrT, const int32_t *colidxT, const double *inv_cnt,
                                    int64_t n_local, const double *dZ, int64_t ld_dz, const int64_t *dmap, int64_t f,
                                    int64_t half_off, const int64_t *rows, int64_t n_rows, double *dH, int64_t ld_dh) {
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t k = 0; k < n_rows; ++k) {
        int64_t u = row_at(rows, k);
        double *o = dH + (size_t)k * (size_t)ld_dh;
        for (int64_t j = 0; j < f; ++j) o[j] = 0.0;
        if (u < n_local) {
            const double *s = dZ + (size_t)map_at(dmap, u) * (size_t)ld_dz;
            for (int64_t j = 0; j < f; ++j) o[j] = s[j];
        }
        for (int64_t e = rowptrT[u]; e < rowptrT[u + 1]; ++e) {
            int64_t v = colidxT[e];
            if (v == u) continue;
            const double *g = dZ + (size_t)map_at(dmap, v) * (size_t)ld_dz + half_off;
            for (int64_t j = 0; j < f; ++j) o[j] += inv_cnt[v] * g[j];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* loss (training harness, not a layer step)                                 */
/* ------------------------------------------------------------------------ */

/* Mean softmax cross-entropy over n rows of logits (C classes); returns the
 * loss and writes G = (softmax - onehot(label)) / n. */
double oracle_softmax_ce(const double *logits, int64_t ld_l, int64_t n, int64_t C, const int32_t *labels, double *G,
                         int64_t ld_g) {
    double total = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        const double *x = logits + (size_t)i * ld_l;
        double mx = x[0];
        for (int64_t c = 1; c < C; ++c)
            if (x[c] > mx) mx = x[c];
        double s = 0.0;
        for (int64_t c = 0; c < C; ++c) s += exp(x[c] - mx);
        double lse = mx + log(s);
        total += lse - x[labels[i]];
        for (int64_t c = 0; c < C; ++c) {
            double p = exp(x[c] - lse);
            G[(size_t)i * ld_g + c] = (p - (c == labels[i] ? 1.0 : 0.0)) / (double)n;
        }
    }
    return n > 0 ? total / (double)n : 0.0;
}

/* ------------------------------------------------------------------------ */
/* Sylvie low-bit halo codec ("Sylvie: 3D-Adaptive and Universal System for  */
/* Large-Scale Graph Neural Network Training" page, Quantizer and            */
/* Dequantizer, Eq. 3-5 as described in the text around them).              */
/* Per row h (f values): B = 2^b - 1 bins, zero point z = min(h),           */
/* scale s = (max(h) - min(h)) / B; the code of h[c] is the stochastic       */
/* rounding of (h[c] - z) / s, i.e. floor((h[c] - z) / s + u) with u         */
/* uniform in [0, 1), kept in [0, B]; the recovered value is q * s + z.      */
/* A constant row (s = 0) gets code 0 everywhere and is recovered exactly.  */
/* The arithmetic is IEEE single precision, one rounding per operation      */
/* (no fused multiply-add), so the codes are a pure function of the inputs; */
/* the division by s is taken as a multiplication by the rounded           */
/* reciprocal 1 / s of the row (t = (h[c] - z) * (1 / s)), and a value whose */
/* t + u is not a number (h[c] = z with an infinite reciprocal) gets 0.     */
/* ------------------------------------------------------------------------ */

/* SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom number  */
/* generators", OOPSLA 2014): the k-th output of the stream seeded with     */
/* `seed` mixes seed + k * 0x9E3779B97F4A7C15.                               */
uint64_t oracle_splitmix64(uint64_t seed, uint64_t k) {
    uint64_t z = seed + k * 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

/* the uniform u of element c of table row r: output k = r * 2^14 + c / 4 + 1 */
/* serves elements 4j .. 4j + 3, through its bits 48..63, 32..47, 16..31    */
/* and 0..15; 16 bits scaled to [0, 1)                                       */
static float codec_uniform(uint64_t seed, int64_t r, int64_t c) {
    const uint64_t k = ((uint64_t)r << 14) + (uint64_t)(c >> 2) + 1u;
    const uint64_t z = oracle_splitmix64(seed, k);
    const uint32_t u16 = (uint32_t)(z >> (48 - 16 * (c & 3))) & 0xFFFFu;
    return (float)u16 * (1.0f / 65536.0f);
}

/* Quantise n rows of f fp32 values (row i at x + i * ld_x, table id ids[i]) */
/* to b-bit codes packed little-endian (code c in bits [c*b, c*b + b) of the */
/* row's bytes, row i at codes + i * ld_codes) and per-row (scale, zero).    */
void oracle_codec_quantize(const float *x, int64_t ld_x, int64_t n, int64_t f, const int64_t *ids, int bits,
                           uint64_t seed, uint8_t *codes, int64_t ld_codes, float *scale_zero) {
    const int B = (1 << bits) - 1;
    for (int64_t i = 0; i < n; ++i) {
        const float *h = x + i * ld_x;
        uint8_t *row = codes + i * ld_codes;
        float mn = h[0], mx = h[0];
        for (int64_t c = 1; c < f; ++c) {
            if (h[c] < mn) mn = h[c];
            if (h[c] > mx) mx = h[c];
        }
        const float range = mx - mn;
        const float s = range / (float)B;
        const float inv = s > 0.0f ? 1.0f / s : 0.0f;
        memset(row, 0, (size_t)ld_codes);
        for (int64_t c = 0; c < f; ++c) {
            int q = 0;
            if (s > 0.0f) {
                const float t = (h[c] - mn) * inv;
                const float v = t + codec_uniform(seed, ids[i], c);
                q = !(v >= 0.0f) ? 0 : (v >= (float)B ? B : (int)floorf(v));
            }
            const int64_t bit = c * bits;
            row[bit >> 3] |= (uint8_t)(q << (bit & 7));
        }
        scale_zero[2 * i] = s;
        scale_zero[2 * i + 1] = mn;
    }
}

/* y[i, c] = q * scale_i + zero_i for c < f */
void oracle_codec_dequantize(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n, int64_t f,
                             int bits, float *y, int64_t ld_y) {
    const int B = (1 << bits) - 1;
    for (int64_t i = 0; i < n; ++i) {
        const uint8_t *row = codes + i * ld_codes;
        const float s = scale_zero[2 * i], z = scale_zero[2 * i + 1];
        for (int64_t c = 0; c < f; ++c) {
            const int64_t bit = c * bits;
            const int q = (row[bit >> 3] >> (bit & 7)) & B;
            const float qs = (float)q * s;
            y[i * ld_y + c] = qs + z;
        }
    }
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
