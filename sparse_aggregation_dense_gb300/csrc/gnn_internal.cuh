// gnn_internal.cuh - internal declarations shared by the libgnn translation units.
#pragma once

#include <cuda_bf16.h>
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <vector>

#include "../../include/gnn.h"

namespace gnn {

constexpr int kWarp = 32;

// bits of a graph's device error word
constexpr int kErrIndex = 1;    // bad index data (a row was skipped)
constexpr int kErrWaitTc = 2;   // a tensor-core kernel's bounded wait ran out
constexpr int kErrWaitAgg = 4;  // an aggregation's bounded wait ran out

// A row of the block (or of its transpose) with more than kHeavyNnz entries is
// split into chunks of kChunkNnz entries, each summed by its own warp into an
// fp32 partial; a fix-up pass adds the partials of a row in chunk order.
constexpr int kHeavyNnz = 512;
constexpr int kChunkNnz = 512;
constexpr int kGroupNnz = 512;   // entry window of a row group
constexpr int kGroupRows = 256;  // rows of a row group at most
// rows wider than this are aggregated in column slices of this many bytes (0: never)
constexpr int64_t kAggSliceBytes = 0;
// pipeline shape of the aggregation (see agg_pipe in aggregate.cu)
constexpr int kAggPipe = 0;

// Column ids of the graph's CSR copies carry a 5-bit "hotness tier" in bits
// 27..31 (when the column count is below 2^27): tier t holds the columns of
// access-count rank below about 1024 * 2^(t/2).  An aggregation keeps the rows of
// the hottest tiers that fit a share of L2 resident (evict_last) and streams the
// rest (evict_first).
constexpr int kTierShift = 27;
constexpr uint32_t kColMask = (1u << kTierShift) - 1u;
constexpr int kTiers = 32;

// Schedule of one CSR (block rows or transpose rows) for the aggregation.
// Work items: chunks of heavy rows and groups of light rows.  The fix-up rows
// are the heavy rows (partials added in chunk order) and the empty rows (no
// chunk: only their zero or self term is written).
struct Schedule {
    bool tagged = false;           // column ids carry tiers
    int64_t tier_rows[kTiers] = {};  // columns per tier
    int64_t n_rows = 0;        // rows of the CSR
    int64_t n_heavy = 0;       // fix-up rows: rows split into chunks, and empty rows
    int64_t n_chunks = 0;      // total chunks
    int32_t *heavy_rows = nullptr;   // [n_heavy] row ids, ascending
    int32_t *heavy_choff = nullptr;  // [n_heavy + 1] first chunk of each heavy row
    int32_t *chunk_row = nullptr;    // [n_chunks]
    int32_t *chunk_begin = nullptr;  // [n_chunks] entry range of the chunk
    int32_t *chunk_end = nullptr;    // [n_chunks]
    // row groups: runs of consecutive light rows (1 to kHeavyNnz entries)
    // whose first entries fall in one kGroupNnz-entry window (at most
    // kGroupRows rows); the aggregation streams a group's entries as one range
    int64_t n_groups = 0;
    int32_t *group_r0 = nullptr;     // [n_groups] first row of the group
    int32_t *group_r1 = nullptr;     // [n_groups] one past its last row
};

}  // namespace gnn

struct gnn_graph {
    int device = 0;
    int64_t n_local = 0, n_halo = 0, nnz = 0;
    gnn_agg agg = GNN_AGG_GCN_SYM;
    // block CSR (graph-owned copy)
    int32_t *rowptr = nullptr, *colidx = nullptr;
    // transpose of the block: n_local + n_halo rows
    int32_t *rowptrT = nullptr, *colidxT = nullptr, *permT = nullptr;
    // GCN: dinv over n_local + n_halo columns; GraphSAGE: inverse neighbour counts of local rows
    float *colw = nullptr;
    // the transpose's tagged column ids in the aggregation's order (each row
    // hottest tier first); null when untagged, and colidxT is used instead
    int32_t *colidxTa = nullptr;
    // graph attention graphs: for each entry of the transpose in the
    // aggregation's order, the block entry (in the block's aggregation order)
    // it came from
    int32_t *t2b = nullptr;
    int32_t *erow = nullptr;  // graph attention: the row of every block entry
    // per-entry weights of the block (forward) and of its transpose (backward),
    // in the aggregation's order
    float *wfwd = nullptr, *wbwd = nullptr;
    gnn::Schedule fwd, bwd;
    int *err = nullptr;  // device error word
    // workspace (heavy-row partials, dW split partials, packed W)
    void *ws = nullptr;
    size_t ws_bytes = 0;
    // push claim array
    uint32_t *claim = nullptr;
    int64_t claim_n = 0;
    uint32_t claim_gen = 0;
    uint8_t *push_ok = nullptr;  // per pushed row: its id may be written (after the claim pass)
    int64_t push_ok_n = 0;
    // event timing (gnn_profile_enable)
    struct ProfRec {
        int kind;
        cudaEvent_t a, b;
    };
    bool prof_on = false;
    std::vector<ProfRec> prof;
};

namespace gnn {

// ---- common helpers -------------------------------------------------------
#define GNN_CUDA_TRY(expr)                                  \
    do {                                                    \
        cudaError_t e_ = (expr);                            \
        if (e_ != cudaSuccess) return gnn::cuda_status(e_); \
    } while (0)

gnn_status cuda_status(cudaError_t e);
// text of the last CUDA runtime error cuda_status saw (gnn_last_cuda_error)
const char *last_cuda_error_text();
// process-wide count of kernel launches (gnn_launch_count)
void count_launches(int64_t n);
#define GNN_LAUNCHED(n) gnn::count_launches(n)
gnn_status ensure_workspace(gnn_graph *g, size_t bytes, cudaStream_t s);

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }
inline int elem_size(gnn_dtype t) { return t == GNN_BF16 ? 2 : 4; }
inline int64_t elems_per_16b(gnn_dtype t) { return 16 / elem_size(t); }

// ---- scan / sort / schedule (graph set-up) --------------------------------
// Exclusive prefix sum of int32 values: out[i] = sum_{j<i} in[i]; out[n] = total
// when out has n + 1 entries (write_total).  in and out may alias.
gnn_status exclusive_scan_i32(const int32_t *in, int32_t *out, int64_t n, bool write_total, cudaStream_t s);
// Transpose of an n_rows x n_cols CSR: stable by source row.
gnn_status csr_transpose(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, int64_t n_cols, int64_t nnz,
                         int32_t *rowptrT, int32_t *colidxT, int32_t *permT, cudaStream_t s);
gnn_status build_schedule(const int32_t *rowptr, int64_t n_rows, Schedule *sc, cudaStream_t s);
// Tag colidx entries with the tier of their column's access count, where the
// count of column c is ptr[c + 1] - ptr[c] (ptr: n_cols + 1 entries).
gnn_status tag_tiers(int32_t *colidx, int64_t nnz, const int32_t *ptr, int64_t n_cols, Schedule *sc, cudaStream_t s);
// Largest tier whose rows (row_bytes each, tiers 0..t together) fit the L2 share.
int hot_tier_for(const Schedule &sc, int64_t row_bytes);
// Copy column ids without their tier bits.
gnn_status copy_untagged(const int32_t *src, int32_t *dst, int64_t n, uint32_t mask, cudaStream_t s);
// every row's entries (tagged column ids and weights), out of place, in a
// stable order by tier, hottest first
gnn_status sort_rows_by_tier(const int32_t *rowptr, int64_t n_rows, const int32_t *col_in, const float *w_in,
                             int32_t *col_out, float *w_out, cudaStream_t s);
void free_schedule(Schedule *sc);

// ---- graph attention (GAT) steps -------------------------------------------
gnn_status launch_iota(int32_t *out, int64_t n, cudaStream_t s);
// t2b[k] = block position (sorted order) of transpose entry k (sorted order):
// fperm[e_sorted] = e_original (null: not sorted), tperm[k_sorted] = k_stable
// (null: not sorted), permT[k_stable] = e_original; scratch: int32[nnz]
gnn_status launch_gat_entry_map(const int32_t *fperm, const int32_t *tperm, const int32_t *permT, int64_t nnz,
                                int32_t *t2b, int32_t *scratch, cudaStream_t s);
// erow[k] = the row holding entry k of a CSR (rowptr of n_rows rows)
gnn_status launch_entry_rows(const int32_t *rowptr, int64_t n_rows, int32_t *erow, cudaStream_t s);
gnn_status launch_gat_scores(const void *T, int64_t ld, int64_t n_total, int64_t n_local, int64_t f,
                             const float *a_src, const float *a_dst, float *s_src, float *s_dst, gnn_dtype dt,
                             cudaStream_t s);
gnn_status launch_gat_softmax(const gnn_graph *g, const float *s_src, const float *s_dst, float *alpha,
                              cudaStream_t s);
gnn_status launch_gat_mask(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int64_t n, int64_t f,
                           void *Y, int64_t ld_y, gnn_dtype dt, gnn_dtype gdt, cudaStream_t s);
gnn_status launch_gat_edge_backward(const gnn_graph *g, const float *s_src, const float *s_dst, const float *alpha,
                                    const void *dY, int64_t ld_y, const void *T, int64_t ld_t, int64_t f, float *dz,
                                    float *ds_dst, gnn_dtype dt, gnn_dtype gdt, cudaStream_t s);
gnn_status launch_gat_transpose(const gnn_graph *g, const float *dz, const float *alpha, float *ds_src,
                                float *alphaT, cudaStream_t s);
gnn_status launch_gat_rank1(void *dT, int64_t ld, int64_t n_total, int64_t n_local, int64_t f, const float *ds_src,
                            const float *ds_dst, const float *a_src, const float *a_dst, gnn_dtype gdt,
                            cudaStream_t s);
size_t gat_colsum_ws_floats(int64_t n_rows, int64_t f);
gnn_status launch_gat_colsum(const void *T, int64_t ld, int64_t n_rows, int64_t f, const float *w, float *out,
                             float *ws, gnn_dtype dt, cudaStream_t s);

// ---- kernels launched by the API ------------------------------------------
gnn_status launch_validate_csr(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, int64_t n_cols,
                               int64_t nnz, int *err, cudaStream_t s);
gnn_status launch_gcn_dinv(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo,
                           int64_t nnz, const float *deg, float *dinv, cudaStream_t s);
gnn_status launch_sage_invcnt(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, float *out,
                              cudaStream_t s);
// per-entry weights: w[e] = colw[col_e] (or 1 when colw is null), 0 when
// skip_self and col_e equals the entry's row
gnn_status launch_entry_weights(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, const float *colw,
                                bool skip_self, float *w, cudaStream_t s);
// set the sign bit of the weight of each row's last entry (in the aggregation's
// entry order): the aggregation reads it as the row's end; weights are >= 0
gnn_status launch_mark_row_ends(const int32_t *rowptr, int64_t n_rows, float *w, cudaStream_t s);

gnn_status launch_pull(const void *table, int64_t ld_t, int64_t n_table, const int64_t *ids, int64_t n_ids,
                       void *H, int64_t ld_h, int64_t row0, int64_t f, int es, int *err, cudaStream_t s);
gnn_status ensure_claim(gnn_graph *g, int64_t n_table);
// claim pass of a push: marks each table id with a generation-stamped count
// (ids seen more than once are reported and skipped by the copy)
gnn_status launch_push_claim(gnn_graph *g, const int64_t *ids, int64_t n_rows, int64_t n_table, uint32_t *gen_out,
                             cudaStream_t s);
// the checks of a push: the claim pass, then g->push_ok[v] = 1 for every row
// whose id is in range and claimed once (repeated ids set the error word)
gnn_status launch_push_checks(gnn_graph *g, const int64_t *ids, int64_t n_rows, int64_t n_table, cudaStream_t s);
// halo-gradient return: send J rows into an fp32 gradient table, receive the sums
gnn_status launch_grad_send(gnn_graph *g, const void *dH, int64_t ld_dh, int64_t f, const int64_t *halo_ids,
                            float *gtable, int64_t ld_gt, int64_t n_table, gnn_dtype dt, cudaStream_t s);
gnn_status launch_grad_recv(gnn_graph *g, const float *gtable, int64_t ld_gt, int64_t n_table,
                            const int64_t *local_ids, void *dH, int64_t ld_dh, int64_t f, gnn_dtype dt,
                            cudaStream_t s);
// rows for the exchange between processes: an indexed gather and an ordered scatter-add
gnn_status launch_gather_rows(const void *src, int64_t ld_src, int64_t n_src, const int64_t *ids, int64_t n,
                              void *dst, int64_t ld_dst, int64_t f, gnn_dtype dt, int *err, cudaStream_t s);
gnn_status launch_scatter_add_rows(const void *src, int64_t ld_src, const int64_t *ids, int64_t n, void *dst,
                                   int64_t ld_dst, int64_t n_dst, int64_t f, gnn_dtype dt, int *err, cudaStream_t s);
// low-bit halo codec (quantise on push, dequantise on pull)
gnn_status launch_codec_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                             uint8_t *codes, int64_t ld_codes, float *scale_zero, int64_t n_table, int bits,
                             uint64_t seed, gnn_dtype dt, cudaStream_t s);
gnn_status launch_quantize_rows(const void *X, int64_t ld_x, int64_t n, int64_t f, const int64_t *keys, int bits,
                                uint64_t seed, uint8_t *codes, int64_t ld_codes, float *scale_zero, gnn_dtype dt,
                                cudaStream_t s);
gnn_status launch_dequantize_rows(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n,
                                  int64_t f, int bits, const int64_t *ids, void *dst, int64_t ld_dst, int64_t n_dst,
                                  int add, gnn_dtype dt, int *err, cudaStream_t s);
gnn_status launch_codec_pull(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n_table,
                             int bits, const int64_t *ids, int64_t n_ids, void *H, int64_t ld_h, int64_t row0,
                             int64_t f, gnn_dtype dt, int *err, cudaStream_t s);
gnn_status launch_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                       void *table, int64_t ld_t, int64_t n_table, int es, cudaStream_t s);

// Aggregation over a CSR with its heavy-row schedule:
//   out[r, off : off + f] = rowscale[r] * sum_{e in row r} wts[e] * X[col_e, 0:f]   (+ the self term)
// The per-entry weights hold the column factor (GCN: dinv[c]; GraphSAGE: 1 or
// inv_cnt[c], and 0 on the diagonal entry the mean leaves out).
enum SelfMode {
    SELF_NONE = 0,
    SELF_COPY = 1,  // out[r, 0:f] = X[r, 0:f]                      (GraphSAGE forward)
    SELF_ADD = 2,   // result += self[r, 0:f] for r < n_self          (GraphSAGE backward)
};
struct AggParams {
    const int32_t *rowptr;
    const uint32_t *colidx;  // column ids, tier bits above colmask
    const float *wts;        // per-entry weights
    const float *rowscale;   // per-row scale, nullptr for 1
    int64_t n_rows;          // output rows computed: [0, n_rows)
    uint32_t colmask;
    int hot_tier;            // entries with tier <= hot_tier are gathered with evict_last
    const void *X;
    int64_t ldx;
    int64_t n_x;             // rows of X: every column id is below it
    int64_t f;
    int self_mode;
    void *out;
    int64_t ldo;
    int64_t out_off;         // column of out where the aggregate is written
    int64_t self_off;        // column of out where SELF_COPY writes the copied row (0)
    const void *self;        // SELF_ADD source (row stride ld_self)
    int64_t ld_self;
    int64_t n_self;
    int relu;                // 1: the aggregated values are written as max(x, 0)
    int *err;                // device error word
    // set by launch_aggregate: the bound of every wait, and the failure-test
    // switch (first batch of the first pair not issued)
    uint64_t wait_ns;
    int starve;
};
gnn_status launch_aggregate(const AggParams &p, const Schedule &sc, gnn_dtype dt, float *partial, cudaStream_t s);
size_t aggregate_partial_bytes(const Schedule &sc, int64_t f);

// Dense update, forward: out = act(Zp Wp), Zp n x Kp (dtype, ld_z), Wp Kp x N fp32 packed (ld_w)
gnn_status launch_update_fwd(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w,
                             int64_t N, int relu, void *out, int64_t ld_o, gnn_dtype dt, cudaStream_t s);
// Dense update, forward, on the tensor cores (bf16): W^T is packed into wt_ws
// (update_tc_wt_bytes); err receives an abort code if a bounded wait expires.
bool update_fwd_tc_supported(int64_t Kp, int64_t N);
size_t update_tc_wt_bytes(int64_t Kp, int64_t N);
gnn_status launch_update_fwd_tc(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w,
                                int64_t N, int relu, void *out, int64_t ld_o, void *wt_ws, int *err, cudaStream_t s);
// 2-D bf16 tensor map with 128-byte swizzle (box_inner x box_outer elements)
bool make_map_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                      uint32_t box_inner, uint32_t box_outer);
// 2-D tensor map over rows of `inner` elements (bf16 or fp32), a box one row
// high and box_inner elements wide, no swizzle, zero fill past the edges: the
// map of the matrix the aggregation gathers rows from (TMA gather of 4 rows)
bool make_map_rows(CUtensorMap *m, bool bf16, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner);
int num_sms();
// Dense update, backward, on the tensor cores (bf16): dZ = dY W^T and the dW
// partials of each CTA (ws: update_bwd_tc_ws_bytes), then dWp = their sum.
bool update_bwd_tc_supported(int64_t Kp, int64_t N);
size_t update_bwd_tc_ws_bytes(int64_t n, int64_t Kp, int64_t N);
// dz_f32: dZ is stored in fp32 (G, H_out and Z are bf16 either way).
gnn_status launch_update_bwd_tc(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                                int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                                float *dWp, void *dZ, int64_t ld_dz, bool dz_f32, void *ws, int *err, cudaStream_t s);
// dY = bf16(relu ? G * 1[H_out > 0] : G) for an fp32 G and a bf16 H_out (H_out may
// be null without ReLU): the tensor-core operand of the (bf16, fp32) backward.
// Y: n x ld_y bf16, ld_y a multiple of 8; columns [N, ld_y) are written as 0.
gnn_status launch_grad_to_bf16(const float *G, int64_t ld_g, const void *Hout, int64_t ld_h, int64_t n, int64_t N,
                               void *Y, int64_t ld_y, cudaStream_t s);
// 2-D fp32 tensor map with 128-byte swizzle (box_inner x box_outer elements)
bool make_map_f32_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                     uint32_t box_inner, uint32_t box_outer);
// GNN_UPDATE_SIMT=1 in the environment selects the CUDA-core update for bf16 too
bool force_simt_update();
// Dense update, backward: dZ = dY Wp^T (n x Kp) when dZ != NULL; dWp partials then dW.
// dt: the activations (Z, Hout); gdt: the gradients (G, dZ); (F32, BF16) is not taken.
gnn_status launch_update_bwd(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                             int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                             float *dWp, void *dZ, int64_t ld_dz, gnn_dtype dt, gnn_dtype gdt, float *ws,
                             size_t ws_bytes, cudaStream_t s);
size_t update_bwd_ws_bytes(int64_t n, int64_t Kp, int64_t N, gnn_dtype dt);

gnn_status launch_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                             int64_t ld_g, float *row_loss, float *loss, int64_t n_mean, gnn_dtype dt, gnn_dtype gdt,
                             cudaStream_t s);

}  // namespace gnn
