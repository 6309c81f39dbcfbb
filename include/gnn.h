/*
 * gnn.h - C ABI of libgnn: one graph partition's full-graph GCN / GraphSAGE
 * layer, forward and backward, on one GB300 GPU (sm_103a).
 *
 * The method (sources named by page title):
 *  - "Reducing Communication in Graph Neural Network Training" (CAGNET), GNN
 *    section: a layer computes H^(l) = sigma(A^T H^(l-1) W^l) where A holds the
 *    graph with self loops, normalised as D^-1/2 (A + I) D^-1/2 with D the
 *    modified degrees; the hot operations are the SpMM and the dense GEMM, and
 *    the backward uses the same primitives.
 *  - Sylvie (arxiv 2303.01277), Graph Engine and Alg. 1 / Alg. 2: each GPU
 *    holds one partition; its HALO vertices (neighbours owned by another
 *    partition) are received every layer; the feature gradients of HALO
 *    vertices (J) are sent back in the backward pass.
 *  - "Distributed Graph Neural Network Training with Periodic Stale
 *    Representation Synchronization" (DIGEST), system design, Fig. 1(c): halo
 *    rows are pulled from a table of stale representations (H_out <- H~_out)
 *    and the fresh local rows are pushed back (H_in -> H~_in).
 *
 * Conventions shared by every call
 *  - Pointers named as device pointers must point to device memory of the
 *    current CUDA device; host pointers are named as such.  The caller owns
 *    every buffer it passes; a gnn_graph owns what it allocated.
 *  - Matrices are row-major with a leading dimension `ld` in ELEMENTS.  Each
 *    row must start on a 16-byte boundary: base pointers 16-byte aligned and
 *    ld a multiple of 4 (fp32) or 8 (bf16).  A call writes columns [0, f) of
 *    the rows it produces; for the aggregation outputs (Z, dH) the columns up
 *    to the next 16-byte boundary are written as zeros too.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every call except gnn_graph_create, gnn_graph_destroy and
 *    gnn_get_error is asynchronous on that stream.
 *  - Host-checkable argument errors (NULL pointers, negative or inconsistent
 *    sizes, bad leading dimensions or alignment, unsupported widths) are
 *    returned synchronously and nothing is launched.  Data errors found on the
 *    device (an id outside the table, a repeated push id) set the graph's
 *    device error word; the offending row is not written and no out-of-bounds
 *    access happens; gnn_get_error reports them.
 *  - Floating point: fp32 data accumulates in fp32; bf16 data (activations,
 *    aggregations, activation gradients) accumulates in fp32 and is stored
 *    rounded to nearest even.  dW is always fp32.  No float atomics are used:
 *    every result is bitwise reproducible run to run.
 */
#ifndef GNN_H
#define GNN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gnn_graph gnn_graph; /* opaque, owned by the library */

typedef enum {
    GNN_OK = 0,
    GNN_EINVAL = 1,       /* bad argument (checked on the host) */
    GNN_ENOMEM = 2,       /* device allocation failed */
    GNN_ECUDA = 3,        /* a CUDA runtime call failed */
    GNN_EUNSUPPORTED = 4, /* valid but unsupported shape / dtype */
    GNN_EINDEX = 5,       /* bad index data found on the device */
    GNN_ETIMEOUT = 6      /* a kernel's bounded wait ran out: it gave up, and
                             the outputs of that call are incomplete */
} gnn_status;

typedef enum { GNN_F32 = 0, GNN_BF16 = 1 } gnn_dtype;

typedef enum {
    GNN_AGG_GCN_SYM = 0,  /* Z[v] = sum_u dinv[v] dinv[u] H[u]  (A_hat = D^-1/2 (A+I) D^-1/2) */
    GNN_AGG_SAGE_MEAN = 1, /* Z[v] = [ H[v] | mean of H[u] over u in N(v), u != v ] */
    GNN_AGG_GAT = 2        /* graph attention: gnn_gat_forward / gnn_gat_backward */
} gnn_agg;

/* Create the partition's graph (CAGNET GNN section: A with self loops and its
 * transpose kept apart; Sylvie Graph Engine: block rows of the local vertices,
 * columns = local vertices then HALO vertices).
 *   rowptr  device int32[n_local + 1], rowptr[0] = 0, non-decreasing, rowptr[n_local] = nnz
 *   colidx  device int32[nnz], every entry in [0, n_local + n_halo); row v lists
 *           the vertices whose rows v aggregates; self loops are stored by the
 *           caller (they are part of A + I).  Order within a row is free.
 *   deg     device float[n_local + n_halo] degrees of A + I (global), or NULL:
 *           then a local vertex's degree is its row length and a halo
 *           vertex's degree is 1 + the number of times its column occurs.
 *           Degree 0 gives a normalisation factor of 0.  (GCN only; ignored
 *           for GraphSAGE, whose mean counts the entries u != v of row v, and
 *           for attention graphs, whose weights are computed per call.)
 *   agg     the layer kind the graph serves: GCN and GraphSAGE graphs take
 *           gnn_layer_forward / backward, GNN_AGG_GAT graphs gnn_gat_forward /
 *           backward (they keep 4 bytes per entry more: where each transpose
 *           entry's attention sits in the block).
 * The graph copies the CSR, validates it on the device, computes the
 * normalisation, builds the transpose (entries of a transpose row ordered by
 * ascending source row) and the load-balance schedules.  For the aggregation
 * it also keeps, for both directions, each row's entries ordered by how often
 * their column is gathered (most first), so the order in which a row's terms
 * are summed is the library's, not the caller's; the exported transpose
 * (gnn_graph_copy_transpose) is the stable one above.  Device memory held:
 * about 24 bytes per entry and 12 bytes per vertex, plus the schedules and a
 * workspace that later calls grow as they need; up to 16 bytes per entry more
 * while the transpose is built.  Synchronous: returns after the stream's work
 * is done.  Errors: GNN_EINVAL (sizes, NULL),
 * GNN_EINDEX (CSR fails validation), GNN_ENOMEM, GNN_ECUDA.  On error *out is
 * set to NULL. */
gnn_status gnn_graph_create(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo,
                            int64_t nnz, const float *deg, gnn_agg agg, void *stream, gnn_graph **out);

/* Free everything the graph owns.  Synchronises the device first.  NULL
 * returns GNN_EINVAL. */
gnn_status gnn_graph_destroy(gnn_graph *g);

/* Pull (DIGEST Fig. 1c, H_out <- H~_out; Sylvie Alg. 1 halo receive):
 *   H[n_local + i, 0:f] = table[halo_ids[i], 0:f]   for i < n_halo.
 *   table     device, n_table x ld_table, dtype
 *   halo_ids  device int64[n_halo]; repeats allowed; an id outside
 *             [0, n_table) sets GNN_EINDEX on the device and leaves that row.
 *   H         device, (n_local + n_halo) x ld_h, dtype; only halo rows written.
 * Bit-exact copy. */
gnn_status gnn_halo_pull(gnn_graph *g, const void *table, int64_t ld_table, int64_t n_table,
                         const int64_t *halo_ids, void *H, int64_t ld_h, int64_t f, gnn_dtype dtype,
                         void *stream);

/* Push (DIGEST Fig. 1c, H_in -> H~_in):
 *   table[local_ids[v], 0:f] = H[v, 0:f]   for v < n_local.
 *   H         device, n_local x ld_h (rows beyond n_local are not read)
 *   local_ids device int64[n_local]; the partition's vertex sets do not
 *             overlap (DIGEST complexity analysis), so a repeated id is an
 *             error: every row carrying it is left unwritten and GNN_EINDEX is
 *             set on the device; likewise for ids outside [0, n_table).
 * Bit-exact copy.  Uses a graph-owned claim array of n_table words (grown on
 * first use with a larger table; that call synchronises). */
gnn_status gnn_halo_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t f, const int64_t *local_ids,
                         void *table, int64_t ld_table, int64_t n_table, gnn_dtype dtype, void *stream);

/* Low-bit halo codec (Sylvie page, "Quantizer" / "Dequantizer"; its Eq. 3-5
 * are stripped from the page text, this is the plainest reading of the prose
 * around them): rows cross the table as b-bit codes plus a per-row scale and
 * zero point, b = 1, 2, 4 or 8, B = 2^b - 1.
 *
 * Push with quantisation: for v < n_local, row h = H[v, 0:f] is stored at
 * table row r = local_ids[v] as
 *   scale_zero[2r] = s = (max h - min h) / B,  scale_zero[2r + 1] = min h,
 *   code c = min(B, floor((h[c] - min h) * (1 / s) + u)),  c < f,
 * with u uniform in [0, 1) (stochastic rounding), or code 0 where s = 0 (or
 * where the sum is not a number).  u of element c of row r is 16 bits of
 * output k = r * 2^14 + floor(c/4) + 1 of a SplitMix64 stream seeded with
 * `seed` (bits 48..63, 32..47, 16..31, 0..15 for c % 4 = 0, 1, 2, 3), so the
 * codes are reproducible.  Arithmetic is IEEE fp32, one rounding per
 * operation (1 / s is the row's rounded reciprocal).
 *   codes      device, n_table x ld_codes bytes; ld_codes a multiple of 16 and
 *              at least b * ceil(f / 8); code c of a row sits in bits
 *              [c b, c b + b) (little-endian); the row's remaining bytes are
 *              written as 0
 *   scale_zero device float[2 n_table]
 * Ids are checked as in gnn_halo_push (repeated or out-of-range ids set
 * GNN_EINDEX on the device; their rows are not written).  Uses the push claim
 * array.  Returns GNN_EINVAL for another b or a bad ld_codes. */
gnn_status gnn_halo_push_quantized(gnn_graph *g, const void *H, int64_t ld_h, int64_t f, const int64_t *local_ids,
                                   uint8_t *codes, int64_t ld_codes, float *scale_zero, int64_t n_table, int bits,
                                   uint64_t seed, gnn_dtype dtype, void *stream);

/* Pull with dequantisation: for i < n_halo, with r = halo_ids[i],
 *   H[n_local + i, c] = code(r, c) * scale_zero[2r] + scale_zero[2r + 1],
 * fp32 multiply then add, rounded to dtype (bf16: round to nearest even);
 * columns c >= f are not written.  An id outside [0, n_table) sets GNN_EINDEX
 * on the device and leaves its row. */
gnn_status gnn_halo_pull_quantized(gnn_graph *g, const uint8_t *codes, int64_t ld_codes, const float *scale_zero,
                                   int64_t n_table, int bits, const int64_t *halo_ids, void *H, int64_t ld_h,
                                   int64_t f, gnn_dtype dtype, void *stream);

/* Column where the mean half of a GraphSAGE aggregation starts:
 * f rounded up to 4 (fp32) or 8 (bf16) elements.  The aggregation width K' of
 * a layer is f_in (GCN) or 2 * gnn_sage_half_offset(f_in) (GraphSAGE). */
int64_t gnn_sage_half_offset(int64_t f, gnn_dtype dtype);

/* Forward layer (CAGNET GNN section; aggregation first, then the update):
 *   Z     = A_hat_block H           (GCN)   or [H_local | mean] (GraphSAGE)
 *   H_out = relu ? max(Z W, 0) : Z W
 *   H      device (n_local + n_halo) x ld_h, dtype: local rows then halo rows
 *   W      device float[K x f_out] row-major, K = f_in (GCN) or 2 f_in
 *          (GraphSAGE: rows 0..f_in-1 multiply the self half, f_in..2f_in-1 the
 *          mean half).  The bf16 path rounds W to bf16 for the tensor cores.
 *   Z      device n_local x ld_z, dtype (written; kept for the backward).
 *          GraphSAGE: self half at column 0, mean half at
 *          gnn_sage_half_offset(f_in), padding columns zero.  ld_z >= K'.
 *   H_out  device n_local x ld_out, dtype.
 * No bias (none in sigma(A^T H W)).  The aggregated rows may be up to 4096
 * bytes (f_in x element size); wider returns GNN_EUNSUPPORTED.  bf16 layers
 * whose shapes the tensor-core kernel takes run on it, the rest (and all
 * fp32 layers) on a CUDA-core kernel with the same results up to rounding. */
gnn_status gnn_layer_forward(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W,
                             int64_t f_out, int relu, void *Z, int64_t ld_z, void *H_out, int64_t ld_out,
                             gnn_dtype dtype, void *stream);

/* Backward layer, by the chain rule of the forward above:
 *   dY = relu ? G * 1[H_out > 0] : G      (ReLU'(0) = 0)
 *   dW = Z^T dY                           device float[K x f_out], overwritten
 *   dZ = dY W^T                           device n_local x ld_dz, grad_dtype
 *                                         (work buffer, same layout as Z);
 *                                         needed only when dH != NULL
 *   dH = A_hat_block^T dZ                 (GCN)
 *   dH[u] = [u local] dZ_self[u] + sum over v with u in N(v), u != v of
 *           dZ_mean[v] / |N(v) \ {v}|     (GraphSAGE)
 *   G      device n_local x ld_g, grad_dtype
 *   H_out  device n_local x ld_out, dtype (read only when relu)
 *   Z      device n_local x ld_z, dtype (as written by gnn_layer_forward)
 *   dH     device (n_local or n_local + n_halo) x ld_dh, grad_dtype, or NULL to
 *          skip the transposed aggregation (first layer).  want_halo_grad != 0
 *          also writes the n_halo halo rows (Sylvie Alg. 2: the HALO gradients
 *          J that are sent back to their owners).
 * Precision: `dtype` is that of the activations (H_out, Z), `grad_dtype` that
 * of the activation gradients (G, dZ, dH).  Accepted pairs: (F32, F32),
 * (BF16, BF16) and (BF16, F32) - bf16 activations with fp32 gradients; another
 * pair returns GNN_EINVAL.  With bf16 activations every operand of the
 * update's products is bf16: Z, W (rounded as in the forward) and dY, which in
 * the (BF16, F32) pair is rounded to bf16 from the fp32 G; the products
 * accumulate in fp32 and dZ and dH are stored in fp32, so the transposed
 * aggregation gathers fp32 rows.  On the tensor cores this pair stages dY in
 * the graph's workspace (n_local x f_out bf16).
 * dW is summed over rows in a fixed order (deterministic).  Same width limit
 * as gnn_layer_forward, in bytes of grad_dtype for the aggregation. */
gnn_status gnn_layer_backward(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                              const void *Z, int64_t ld_z, const float *W, int64_t f_in, int64_t f_out, int relu,
                              float *dW, void *dZ, int64_t ld_dz, void *dH, int64_t ld_dh, int want_halo_grad,
                              gnn_dtype dtype, gnn_dtype grad_dtype, void *stream);

/* The backward of a GCN layer (gnn_layer_forward's) with the products in the
 * other order: dH = (A_hat_block^T dY) W^T instead of A_hat_block^T (dY W^T)
 * (associativity; the chain rule of the CAGNET page's H = sigma(A^T H W)).
 * The transposed aggregation then gathers the bf16 rows of dY (f_out values)
 * instead of the fp32 rows of dZ (f_in values).
 *   dY = G * 1[H_out > 0] (or G) rounded to bf16, as in gnn_layer_backward
 *   dW = Z^T dY                  device float[f_in x f_out], overwritten
 *   P  = A_hat_block^T dY        device (n_local or n_local + n_halo) x ld_p,
 *                                bf16 (fp32 sums, rounded once: it is the
 *                                operand of the next product)
 *   dH = P W^T                   device (as P's rows) x ld_dh, fp32
 * want_halo_grad != 0 computes P and dH for the halo rows too (Sylvie's J).
 * The results agree with gnn_layer_backward up to the rounding of P.  Only the
 * GCN aggregation with bf16 activations and fp32 gradients, on the tensor
 * cores, is taken: a GraphSAGE graph, another precision pair or widths past
 * the tensor-core limits return GNN_EUNSUPPORTED before anything runs; an
 * attention graph (as for every layer call), bad pointers or sizes
 * GNN_EINVAL. */
gnn_status gnn_layer_backward_reordered(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                                        const void *Z, int64_t ld_z, const float *W, int64_t f_in, int64_t f_out,
                                        int relu, float *dW, void *P, int64_t ld_p, void *dH, int64_t ld_dh,
                                        int want_halo_grad, gnn_dtype dtype, gnn_dtype grad_dtype, void *stream);

/* The same GCN layer with the multiplication first, for layers whose output
 * is narrower than their input (f_out < f_in): A_hat (H W) = (A_hat H) W, so
 * the aggregations run at width f_out instead of f_in (fewer bytes gathered);
 * the results agree with gnn_layer_forward / gnn_layer_backward up to
 * rounding (bf16 storage rounds T and P instead of Z and dZ).  GCN only
 * (GraphSAGE: GNN_EUNSUPPORTED).
 * Forward:
 *   T     = H W                          device (n_local + n_halo) x ld_t, dtype
 *                                        (work; every row, local and halo)
 *   H_out = relu ? max(A_hat_block T, 0) : A_hat_block T    (n_local rows)
 * Backward (T is not needed; the layer input H is):
 *   dY = relu ? G * 1[H_out > 0] : G
 *   P  = A_hat_block^T dY               device (n_local + n_halo) x ld_p, dtype
 *                                        (work; every row)
 *   dW = H^T P                           device float[f_in x f_out], overwritten
 *   dH = P W^T                           device (n_local + n_halo) x ld_dh, dtype,
 *                                        every row (the halo rows are Sylvie's
 *                                        J), or NULL to skip
 * The other arguments are as for gnn_layer_forward / gnn_layer_backward; here
 * the aggregated rows are f_out wide (at most 4096 bytes), and every operand,
 * gradients included, is stored in the one `dtype`. */
gnn_status gnn_layer_forward_narrow(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W,
                                    int64_t f_out, int relu, void *T, int64_t ld_t, void *H_out, int64_t ld_out,
                                    gnn_dtype dtype, void *stream);
gnn_status gnn_layer_backward_narrow(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                                     const void *H, int64_t ld_h, const float *W, int64_t f_in, int64_t f_out,
                                     int relu, float *dW, void *P, int64_t ld_p, void *dH, int64_t ld_dh,
                                     gnn_dtype dtype, void *stream);

/* Training-harness helper (not a layer step): mean softmax cross-entropy over
 * n rows of C logits with integer labels.
 *   logits  device n x ld, dtype;  labels device int32[n] in [0, C)
 *   G       device n x ld_g, grad_dtype: (softmax - onehot) / n (computed in
 *           fp32, rounded to grad_dtype); columns past C are not written
 *   row_loss device float[n] work buffer;  loss device float[1]: the mean,
 *   summed in a fixed order.  A label outside [0, C) yields a NaN loss (the
 *   labels live on the device and are not checked on the host).
 * ld and ld_g are multiples of the 16-byte element counts of their dtypes
 * for the vectorised kernel; other leading dimensions take a slower one. */
gnn_status gnn_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                          int64_t ld_g, float *row_loss, float *loss, gnn_dtype dtype, gnn_dtype grad_dtype,
                          void *stream);

/* As gnn_softmax_ce, but the mean (and the gradient's 1/n) divides by n_mean
 * >= n instead of n: the share of these n rows in the mean over n_mean rows
 * spread over several partitions (summing the partitions' losses gives the
 * whole mean, and their G together are the gradient of it). */
gnn_status gnn_softmax_ce_partial(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels,
                                  void *G, int64_t ld_g, float *row_loss, float *loss, int64_t n_mean,
                                  gnn_dtype dtype, gnn_dtype grad_dtype, void *stream);

/* Halo-gradient return (Sylvie page, backward propagation and Alg. 2: the
 * feature gradients J of a partition's HALO vertices go back to the owning
 * partitions and are added to their gradients), through an fp32 gradient table
 * indexed by global vertex id (gtable device float, n_table x ld_gt, ld_gt a
 * multiple of 4; the caller zeroes it before the first send of a layer).
 * Send:    gtable[halo_ids[i], 0:f] += dH[n_local + i, 0:f]   for i < n_halo
 *          (dH as written by gnn_layer_backward with want_halo_grad).  The halo
 *          ids of one graph are distinct: a repeated id sets GNN_EINDEX on the
 *          device and its rows are not sent; an id outside [0, n_table) too.
 *          Uses the push claim array.
 * Receive: dH[v, 0:f] += gtable[local_ids[v], 0:f]            for v < n_local
 *          (fp32 sum, rounded to dtype).
 * Sends of several graphs into one table, issued in order on one stream, add
 * in that order: the sums are reproducible bit for bit. */
gnn_status gnn_halo_grad_send(gnn_graph *g, const void *dH, int64_t ld_dh, int64_t f, const int64_t *halo_ids,
                              float *gtable, int64_t ld_gt, int64_t n_table, gnn_dtype dtype, void *stream);
gnn_status gnn_halo_grad_recv(gnn_graph *g, const float *gtable, int64_t ld_gt, int64_t n_table,
                              const int64_t *local_ids, void *dH, int64_t ld_dh, int64_t f, gnn_dtype dtype,
                              void *stream);

/* Graph attention layer (GAT) on a graph created with GNN_AGG_GAT.  The
 * Sylvie page names GAT among the models it trains and the DIGEST page
 * benchmarks it; neither prints the layer, so this is the textbook
 * single-head form (no normalisation by degrees):
 *   T        = H W over every row, local and halo      device (n_local + n_halo) x ld_t, dtype
 *   s_src[u] = T[u] . a_src (every row),  s_dst[v] = T[v] . a_dst (local rows)
 *              scores: device float[2 n_local + n_halo] = s_src then s_dst
 *   alpha_vu = softmax over the entries u of row v of LeakyReLU_0.2(s_dst[v] + s_src[u])
 *              alpha: device float[nnz], in the library's entry order, with the
 *              sign bit of each row's last entry set (kept for the backward)
 *   H_out[v] = relu ? max(sum_u alpha_vu T[u], 0) : sum_u alpha_vu T[u]
 *              device n_local x ld_out, dtype
 * W device float[f_in x f_out] (rounded to bf16 for the bf16 path);
 * a_src, a_dst device float[f_out].  The aggregated rows T are at most 4096
 * bytes wide.  GNN_EINVAL for a graph of another kind. */
gnn_status gnn_gat_forward(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W,
                           const float *a_src, const float *a_dst, int64_t f_out, int relu, void *T, int64_t ld_t,
                           float *scores, float *alpha, void *H_out, int64_t ld_out, gnn_dtype dtype, void *stream);

/* Backward of gnn_gat_forward, by the chain rule:
 *   dY        = relu ? G * 1[H_out > 0] : G
 *   de_vu     = alpha_vu (dY[v] . T[u] - sum_u' alpha_vu' dY[v] . T[u'])
 *   dz_vu     = de_vu (s_dst[v] + s_src[u] > 0 ? 1 : 0.2)
 *   ds_dst[v] = sum_u dz_vu,   ds_src[u] = sum over entries (v, u) of dz_vu
 *   dT[u]     = sum over entries (v, u) of alpha_vu dY[v] + ds_src[u] a_src
 *               + [u local] ds_dst[u] a_dst          device (n_local + n_halo) x ld_dt, grad_dtype (written)
 *   da_src    = sum_u ds_src[u] T[u],  da_dst = sum_v ds_dst[v] T[v]   device float[f_out]
 *   dW        = H^T dT                                device float[f_in x f_out]
 *   dH        = dT W^T over every row (the halo rows are Sylvie's J)
 *               device (n_local + n_halo) x ld_dh, grad_dtype, or NULL to skip
 * G device n_local x ld_g, grad_dtype; H_out, H, T, scores and alpha as the
 * forward used or wrote them.  Precision pairs as for gnn_layer_backward; with
 * bf16 activations dT enters the products as bf16.  Every sum is formed in a
 * fixed order (reproducible bits).  The workspace grows by about 8 bytes per
 * entry plus the staging of dY (and of dT in bf16). */
gnn_status gnn_gat_backward(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                            const void *H, int64_t ld_h, int64_t f_in, const float *W, const float *a_src,
                            const float *a_dst, int64_t f_out, int relu, const void *T, int64_t ld_t,
                            const float *scores, const float *alpha, float *dW, float *da_src, float *da_dst,
                            void *dT, int64_t ld_dt, void *dH, int64_t ld_dh, gnn_dtype dtype, gnn_dtype grad_dtype,
                            void *stream);

/* Rows of the halo exchange between processes (Sylvie page, Graph Engine and
 * Alg. 1 / Alg. 2: each partition sends the rows of its vertices that other
 * partitions hold as HALO vertices, and in the backward pass receives the
 * gradients J of those rows back).  No graph is involved: these are the
 * packing and unpacking steps around a collective (all-to-all) that moves the
 * rows between partitions.
 * Gather: dst[i, 0:f] = src[ids[i], 0:f] for i < n (bit-exact copy).
 *   src  device n_src x ld_src, dtype;  ids device int64[n];  dst device n x ld_dst.
 * Scatter-add: dst[ids[i], 0:f] += src[i, 0:f] for i < n, summed in fp32 and
 *   stored as dtype.  The ids of one call must be distinct (rows added by one
 *   call must not collide; several calls on one stream add in call order, so
 *   sums are reproducible).  src device n x ld_src; dst device n_dst x ld_dst.
 * An id outside the rows of its matrix leaves that row alone and, when err
 * (device int, nullable) is given, sets bit 0 of *err.  Host-checkable
 * argument errors return GNN_EINVAL. */
gnn_status gnn_gather_rows(const void *src, int64_t ld_src, int64_t n_src, const int64_t *ids, int64_t n, void *dst,
                           int64_t ld_dst, int64_t f, gnn_dtype dtype, int *err, void *stream);
gnn_status gnn_scatter_add_rows(const void *src, int64_t ld_src, const int64_t *ids, int64_t n, void *dst,
                                int64_t ld_dst, int64_t n_dst, int64_t f, gnn_dtype dtype, int *err, void *stream);

/* The low-bit codec on rows that travel as a message between processes
 * (Sylvie page, Quantizer / Dequantizer: halo rows in the forward pass and
 * the feature gradients J in the backward pass cross the network as b-bit
 * codes).  Same code and draw layout as gnn_halo_push_quantized, with row i of
 * the message in place of table row r:
 * Quantise: codes row i and scale_zero[2i], [2i + 1] from X[i, 0:f], the
 *   draws keyed by keys[i] (e.g. the vertex's global id) and seed.
 *   X device n x ld_x, dtype; keys device int64[n]; codes device n x ld_codes.
 * Dequantise: dst[ids[i], 0:f] = (add ? dst[ids[i], 0:f] : 0) + code * scale +
 *   zero (fp32 multiply, add, add, each rounded once, stored as dtype); ids
 *   NULL means row i.  The ids of one call are distinct.  An id outside
 *   [0, n_dst) leaves its row alone and sets bit 0 of *err (nullable).
 * GNN_EINVAL for another b, a bad ld_codes or other host-checkable errors. */
gnn_status gnn_quantize_rows(const void *X, int64_t ld_x, int64_t n, int64_t f, const int64_t *keys, int bits,
                             uint64_t seed, uint8_t *codes, int64_t ld_codes, float *scale_zero, gnn_dtype dtype,
                             void *stream);
gnn_status gnn_dequantize_rows(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n, int64_t f,
                               int bits, const int64_t *ids, void *dst, int64_t ld_dst, int64_t n_dst, int add,
                               gnn_dtype dtype, int *err, void *stream);

/* Synchronise the device, then return and clear the graph's device error word:
 * GNN_OK, GNN_ETIMEOUT (a kernel of one of the graph's calls gave up on a
 * bounded wait - every wait on the device gives up after about 2 s, records
 * this and returns instead of spinning), or GNN_EINDEX (bad index data);
 * GNN_ECUDA if the synchronisation itself failed. */
gnn_status gnn_get_error(gnn_graph *g);

/* Failure-detection test hook (not a step of the method): arms a one-shot
 * fault in the next aggregation launched by this process, on any graph.  The
 * first batch of that launch's first producer / consumer warp pair is never
 * issued, so its consumer's bounded wait runs out after wait_ns nanoseconds
 * (> 0): the kernel raises its abort flag, the other warps of the block stop,
 * every gather already issued is waited for, and the launch returns; the
 * call's graph then reports GNN_ETIMEOUT through gnn_get_error.  Nothing faults
 * and the context stays usable.  wait_ns <= 0 disarms the hook. */
gnn_status gnn_debug_expire_next_wait(int64_t wait_ns);

/* Sizes of a graph (host outputs, any may be NULL). */
gnn_status gnn_graph_sizes(const gnn_graph *g, int64_t *n_local, int64_t *n_halo, int64_t *nnz);

/* Copy the transpose built by gnn_graph_create into caller device buffers
 * (asynchronous on stream): rowptrT int32[n_local + n_halo + 1],
 * colidxT int32[nnz] (source rows, ascending within each row) and
 * permT int32[nnz] (the block entry each transpose entry came from).  Any of
 * the three may be NULL to skip it. */
gnn_status gnn_graph_copy_transpose(const gnn_graph *g, int32_t *rowptrT, int32_t *colidxT, int32_t *permT,
                                    void *stream);

/* Event timing of the library's kernel groups, for profiling (off by default).
 * When enabled on a graph, every call on it records a CUDA event pair around
 * each group it launches, on the call's stream:
 *   GNN_PROF_AGG_FWD   the forward aggregation (SpMM kernel and its heavy-row fix-up)
 *   GNN_PROF_AGG_BWD   the backward aggregation over the transpose
 *   GNN_PROF_UPD_FWD   the forward dense update (GEMM + ReLU)
 *   GNN_PROF_UPD_BWD   the backward dense update (dZ and dW)
 *   GNN_PROF_PULL, GNN_PROF_PUSH  the table copies
 * gnn_profile_read synchronises the device, writes the summed milliseconds and
 * the number of recorded groups per kind (arrays of GNN_PROF_COUNT entries,
 * host memory) and clears the records. */
typedef enum {
    GNN_PROF_AGG_FWD = 0,
    GNN_PROF_AGG_BWD = 1,
    GNN_PROF_UPD_FWD = 2,
    GNN_PROF_UPD_BWD = 3,
    GNN_PROF_PULL = 4,
    GNN_PROF_PUSH = 5,
    GNN_PROF_COUNT = 6
} gnn_prof_kind;
gnn_status gnn_profile_enable(gnn_graph *g, int on);
gnn_status gnn_profile_read(gnn_graph *g, double *ms, int64_t *count);

/* Forward aggregation that allocates no device memory.  No counterpart in the
 * method's sources: this entry point exists for callers that cannot call
 * cudaMalloc at the point where they aggregate - e.g. a serving or training
 * loop whose device memory is all reserved up front by another allocator (a
 * framework's caching pool), or code that must not pay for the device-wide
 * synchronisation that cudaMalloc / cudaFree can cause.
 *   Computes exactly the Z of gnn_layer_forward (GCN: A_hat_block H; GraphSAGE:
 *   the self / mean halves), with the same arguments, layout and errors:
 *   H  device (n_local + n_halo) x ld_h, dtype;  Z  device n_local x ld_z.
 * It runs the same kernels, but keeps the fp32 partial sums of the heavy-row
 * chunks in a fixed 16 MiB array that is part of the library (held on every
 * GPU that loads libgnn until the process exits) instead of the graph's
 * workspace.  A graph and width whose partials would not fit (chunks of rows
 * longer than 512 entries x f rounded up to 8 x 4 bytes > 16 MiB) are rejected
 * with GNN_EUNSUPPORTED before anything is launched; so are widths above 4096
 * bytes.  The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) once for that device.  All calls share the array:
 * calls that overlap on the GPU (other streams, other threads) race, so
 * serialise them.  Nothing in the array needs to start at zero: every call
 * overwrites the partials it reads.  The graph must have been created before
 * (gnn_graph_create allocates). */
gnn_status gnn_aggregate_forward_noalloc(const gnn_graph *g, const void *H, int64_t ld_h, int64_t f, void *Z,
                                         int64_t ld_z, gnn_dtype dtype, void *stream);

/* Number of kernels libgnn has launched in this process so far (all graphs). */
int64_t gnn_launch_count(void);

/* Static text for a status code. */
const char *gnn_status_string(gnn_status s);

/* Static text of the last CUDA runtime error behind a GNN_ECUDA (or
 * GNN_ENOMEM) status returned by any call in this process, e.g. "an illegal
 * memory access was encountered"; "no error" if there was none.  Process-wide,
 * not per thread or per graph: read it right after the failing call. */
const char *gnn_last_cuda_error(void);

#ifdef __cplusplus
}
#endif

#endif /* GNN_H */
