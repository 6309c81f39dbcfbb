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

// A row of the block (or of its transpose) with more than kHeavyNnz entries is
// split into chunks of kChunkNnz entries, each summed by its own warp into an
// fp32 partial; a fix-up pass adds the partials of a row in chunk order.
constexpr int kHeavyNnz = 512;
constexpr int kChunkNnz = 512;
constexpr int kGroupNnz = 512;   // entry window of a row group
constexpr int kGroupRows = 256;  // rows of a row group at most

// Column ids of the graph's CSR copies carry a 5-bit "hotness tier" in bits
// 27..31 (when the column count is below 2^27): tier t holds the columns of
// access-count rank below about 1024 * 2^(t/2).  An aggregation keeps the rows of
// the hottest tiers that fit a share of L2 resident (evict_last) and streams the
// rest (evict_first).
constexpr int kTierShift = 27;
constexpr uint32_t kColMask = (1u << kTierShift) - 1u;
constexpr int kTiers = 32;

// Heavy-row schedule of one CSR (block rows or transpose rows).
struct Schedule {
    bool tagged = false;           // column ids carry tiers
    int64_t tier_rows[kTiers] = {};  // columns per tier
    int64_t n_rows = 0;        // rows of the CSR
    int64_t n_heavy = 0;       // rows split into chunks
    int64_t n_chunks = 0;      // total chunks
    int32_t *heavy_rows = nullptr;   // [n_heavy] row ids, ascending
    int32_t *heavy_choff = nullptr;  // [n_heavy + 1] first chunk of each heavy row
    int32_t *chunk_row = nullptr;    // [n_chunks]
    int32_t *chunk_begin = nullptr;  // [n_chunks] entry range of the chunk
    int32_t *chunk_end = nullptr;    // [n_chunks]
    // row groups: runs of consecutive light rows whose first entries fall in
    // one kGroupNnz-entry window (at most kGroupRows rows); the aggregation
    // streams a group's entries as one range
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

gnn_status launch_pull(const void *table, int64_t ld_t, int64_t n_table, const int64_t *ids, int64_t n_ids,
                       void *H, int64_t ld_h, int64_t row0, int64_t f, int es, int *err, cudaStream_t s);
gnn_status ensure_claim(gnn_graph *g, int64_t n_table);
// claim pass of a push: marks each table id with a generation-stamped count
// (ids seen more than once are reported and skipped by the copy)
gnn_status launch_push_claim(gnn_graph *g, const int64_t *ids, int64_t n_rows, int64_t n_table, uint32_t *gen_out,
                             cudaStream_t s);
// halo-gradient return: send J rows into an fp32 gradient table, receive the sums
gnn_status launch_grad_send(gnn_graph *g, const void *dH, int64_t ld_dh, int64_t f, const int64_t *halo_ids,
                            float *gtable, int64_t ld_gt, int64_t n_table, gnn_dtype dt, cudaStream_t s);
gnn_status launch_grad_recv(gnn_graph *g, const float *gtable, int64_t ld_gt, int64_t n_table,
                            const int64_t *local_ids, void *dH, int64_t ld_dh, int64_t f, gnn_dtype dt,
                            cudaStream_t s);
// low-bit halo codec (quantise on push, dequantise on pull)
gnn_status launch_codec_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                             uint8_t *codes, int64_t ld_codes, float *scale_zero, int64_t n_table, int bits,
                             uint64_t seed, gnn_dtype dt, cudaStream_t s);
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
    const void *self;        // SELF_ADD source (row stride ld_self)
    int64_t ld_self;
    int64_t n_self;
    int relu;                // 1: the aggregated values are written as max(x, 0)
    int *err;                // device error word
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
gnn_status launch_update_bwd_tc(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                                int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                                float *dWp, void *dZ, int64_t ld_dz, void *ws, int *err, cudaStream_t s);
// GNN_UPDATE_SIMT=1 in the environment selects the CUDA-core update for bf16 too
bool force_simt_update();
// Dense update, backward: dZ = dY Wp^T (n x Kp) when dZ != NULL; dWp partials then dW.
gnn_status launch_update_bwd(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                             int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                             float *dWp, void *dZ, int64_t ld_dz, gnn_dtype dt, float *ws, size_t ws_bytes,
                             cudaStream_t s);
size_t update_bwd_ws_bytes(int64_t n, int64_t Kp, int64_t N, gnn_dtype dt);

gnn_status launch_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                             int64_t ld_g, float *row_loss, float *loss, int64_t n_mean, gnn_dtype dt,
                             cudaStream_t s);

}  // namespace gnn
