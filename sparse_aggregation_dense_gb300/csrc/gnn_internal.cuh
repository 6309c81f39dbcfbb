// gnn_internal.cuh - internal declarations shared by the libgnn translation units.
#pragma once

#include <cuda_bf16.h>
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

// Heavy-row schedule of one CSR (block rows or transpose rows).
struct Schedule {
    int64_t n_rows = 0;        // rows of the CSR
    int64_t n_heavy = 0;       // rows split into chunks
    int64_t n_chunks = 0;      // total chunks
    int32_t *heavy_rows = nullptr;   // [n_heavy] row ids, ascending
    int32_t *heavy_choff = nullptr;  // [n_heavy + 1] first chunk of each heavy row
    int32_t *chunk_row = nullptr;    // [n_chunks]
    int32_t *chunk_begin = nullptr;  // [n_chunks] entry range of the chunk
    int32_t *chunk_end = nullptr;    // [n_chunks]
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
void free_schedule(Schedule *sc);

// ---- kernels launched by the API ------------------------------------------
gnn_status launch_validate_csr(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, int64_t n_cols,
                               int64_t nnz, int *err, cudaStream_t s);
gnn_status launch_gcn_dinv(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo,
                           int64_t nnz, const float *deg, float *dinv, cudaStream_t s);
gnn_status launch_sage_invcnt(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, float *out,
                              cudaStream_t s);

gnn_status launch_pull(const void *table, int64_t ld_t, int64_t n_table, const int64_t *ids, int64_t n_ids,
                       void *H, int64_t ld_h, int64_t row0, int64_t f, int es, int *err, cudaStream_t s);
gnn_status ensure_claim(gnn_graph *g, int64_t n_table);
gnn_status launch_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                       void *table, int64_t ld_t, int64_t n_table, int es, cudaStream_t s);

// Aggregation over a CSR with its heavy-row schedule.
//   out[r, off : off + f] = rowscale(r) * sum_{e in row r, keep(e)} colw(col_e) * X[col_e, 0:f]
// mode selects the weights and the self term:
enum AggMode {
    AGG_GCN = 0,        // rowscale = colw[r], weight = colw[c]                 (forward and backward)
    AGG_SAGE_FWD = 1,   // rowscale = colw[r], weight 1, skip c == r, out[r, 0:f] = X[r] copied
    AGG_SAGE_BWD = 2,   // rowscale 1, weight = colw[c], skip c == r, + self[r, 0:f] for r < n_self
};
struct AggParams {
    const int32_t *rowptr;
    const int32_t *colidx;
    int64_t n_rows;      // output rows computed: [0, n_rows)
    const void *X;
    int64_t ldx;
    int64_t f;
    const float *colw;
    int mode;
    void *out;
    int64_t ldo;
    int64_t out_off;     // column of out where the aggregate is written
    const void *self;    // AGG_SAGE_BWD: dZ (self half at column 0); AGG_SAGE_FWD: unused (X)
    int64_t ld_self;
    int64_t n_self;      // AGG_SAGE_BWD: rows r < n_self get the self term
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
// GNN_UPDATE_SIMT=1 in the environment selects the CUDA-core update for bf16 too
bool force_simt_update();
// Dense update, backward: dZ = dY Wp^T (n x Kp) when dZ != NULL; dWp partials then dW.
gnn_status launch_update_bwd(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                             int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                             float *dWp, void *dZ, int64_t ld_dz, gnn_dtype dt, float *ws, size_t ws_bytes,
                             cudaStream_t s);
size_t update_bwd_ws_bytes(int64_t n, int64_t Kp, int64_t N, gnn_dtype dt);

gnn_status launch_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                             int64_t ld_g, float *row_loss, float *loss, gnn_dtype dt, cudaStream_t s);

}  // namespace gnn
