// api.cu - the C ABI (include/gnn.h): argument checks, graph lifetime and the
// order of the kernels of each call.
#include <algorithm>
#include <atomic>
#include <cstdlib>
#include <new>

#include "gnn_internal.cuh"

using namespace gnn;

namespace {

constexpr size_t kAlign = 256;

inline size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool dtype_ok(gnn_dtype t) { return t == GNN_F32 || t == GNN_BF16; }

// a row-major operand of `rows` rows whose rows start on 16-byte boundaries
inline bool operand_ok(const void *p, int64_t rows, int64_t ld, int64_t f, gnn_dtype t) {
    if (rows == 0) return true;
    if (!p || !aligned16(p)) return false;
    if (ld < f || ld % elems_per_16b(t) != 0) return false;
    return true;
}

inline cudaStream_t as_stream(void *s) { return static_cast<cudaStream_t>(s); }

// Wp = W laid out on the rows of the aggregation (GraphSAGE padding rows zero);
// the bf16 path rounds W to bf16 (nearest even), the precision its products use.
__global__ void pack_w_kernel(const float *__restrict__ W, int64_t K, int64_t N, int64_t f_in, int64_t half, int sage,
                              int64_t Kp, float *__restrict__ Wp, int64_t ldw, int to_bf16) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= Kp * ldw) return;
    int64_t kp = x / ldw, j = x % ldw;
    int64_t k = -1;
    if (!sage) k = kp < K ? kp : -1;
    else if (kp < f_in) k = kp;
    else if (kp >= half && kp < half + f_in) k = f_in + (kp - half);
    float w = (k >= 0 && j < N) ? W[k * N + j] : 0.f;
    Wp[x] = to_bf16 ? __bfloat162float(__float2bfloat16_rn(w)) : w;
}

__global__ void unpack_dw_kernel(const float *__restrict__ dWp, int64_t N, int64_t f_in, int64_t half,
                                 float *__restrict__ dW) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= 2 * f_in * N) return;
    int64_t k = x / N, j = x % N;
    int64_t kp = k < f_in ? k : half + (k - f_in);
    dW[x] = dWp[kp * N + j];
}

// dY = G * 1[H_out > 0] (ReLU'(0) = 0), element by element
template <typename T>
__global__ void relu_mask_kernel(const T *__restrict__ G, int64_t ld_g, const T *__restrict__ Hout, int64_t ld_h,
                                 int64_t n, int64_t f, T *__restrict__ Y, int64_t ld_y) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n * f) return;
    const int64_t r = x / f, c = x % f;
    const T h = Hout[r * ld_h + c];
    Y[r * ld_y + c] = (float)h > 0.f ? G[r * ld_g + c] : T(0.f);
}

}  // namespace

namespace gnn {

static std::atomic<int64_t> g_launches{0};

bool force_simt_update() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("GNN_UPDATE_SIMT");
        v = (e && e[0] == '1') ? 1 : 0;
    }
    return v == 1;
}

void count_launches(int64_t n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

gnn_status ensure_workspace(gnn_graph *g, size_t bytes, cudaStream_t s) {
    if (bytes <= g->ws_bytes) return GNN_OK;
    if (g->ws) GNN_CUDA_TRY(cudaFreeAsync(g->ws, s));
    g->ws = nullptr;
    g->ws_bytes = 0;
    size_t want = bytes + bytes / 4;
    GNN_CUDA_TRY(cudaMallocAsync(&g->ws, want, s));
    g->ws_bytes = want;
    return GNN_OK;
}

}  // namespace gnn

namespace {

// Records an event pair around a group of launches when profiling is on.
struct ProfScope {
    gnn_graph *g;
    int kind;
    cudaStream_t s;
    cudaEvent_t a = nullptr, b = nullptr;
    ProfScope(gnn_graph *g_, int kind_, cudaStream_t s_) : g(g_), kind(kind_), s(s_) {
        if (!g->prof_on) return;
        if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) {
            a = b = nullptr;
            return;
        }
        cudaEventRecord(a, s);
    }
    ~ProfScope() {
        if (!a) return;
        cudaEventRecord(b, s);
        g->prof.push_back({kind, a, b});
    }
};

}  // namespace

extern "C" {

int64_t gnn_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

gnn_status gnn_profile_enable(gnn_graph *g, int on) {
    if (!g) return GNN_EINVAL;
    g->prof_on = on != 0;
    return GNN_OK;
}

gnn_status gnn_profile_read(gnn_graph *g, double *ms, int64_t *count) {
    if (!g || !ms || !count) return GNN_EINVAL;
    for (int k = 0; k < GNN_PROF_COUNT; ++k) {
        ms[k] = 0.0;
        count[k] = 0;
    }
    if (cudaDeviceSynchronize() != cudaSuccess) return GNN_ECUDA;
    for (auto &r : g->prof) {
        float t = 0.f;
        if (cudaEventElapsedTime(&t, r.a, r.b) == cudaSuccess && r.kind >= 0 && r.kind < GNN_PROF_COUNT) {
            ms[r.kind] += t;
            count[r.kind] += 1;
        }
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    g->prof.clear();
    return GNN_OK;
}

const char *gnn_status_string(gnn_status s) {
    switch (s) {
        case GNN_OK: return "ok";
        case GNN_EINVAL: return "invalid argument";
        case GNN_ENOMEM: return "out of device memory";
        case GNN_ECUDA: return "CUDA runtime error";
        case GNN_EUNSUPPORTED: return "unsupported shape or type";
        case GNN_EINDEX: return "bad index data on the device";
        case GNN_ETIMEOUT: return "a bounded wait on the device ran out";
    }
    return "unknown status";
}

const char *gnn_last_cuda_error(void) { return last_cuda_error_text(); }

int64_t gnn_sage_half_offset(int64_t f, gnn_dtype dtype) {
    return round_up(f, dtype == GNN_BF16 ? 8 : 4);
}

static void destroy_graph(gnn_graph *g) {
    if (!g) return;
    for (auto &r : g->prof) {
        cudaEventDestroy(r.a);
        cudaEventDestroy(r.b);
    }
    cudaFree(g->rowptr);
    cudaFree(g->colidx);
    cudaFree(g->rowptrT);
    cudaFree(g->colidxT);
    cudaFree(g->colidxTa);
    cudaFree(g->permT);
    cudaFree(g->colw);
    cudaFree(g->wfwd);
    cudaFree(g->wbwd);
    cudaFree(g->t2b);
    cudaFree(g->erow);
    cudaFree(g->err);
    cudaFree(g->ws);
    cudaFree(g->claim);
    cudaFree(g->push_ok);
    free_schedule(&g->fwd);
    free_schedule(&g->bwd);
    delete g;
}

gnn_status gnn_graph_create(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo,
                            int64_t nnz, const float *deg, gnn_agg agg, void *stream, gnn_graph **out) {
    if (!out) return GNN_EINVAL;
    *out = nullptr;
    if (n_local < 0 || n_halo < 0 || nnz < 0 || !rowptr) return GNN_EINVAL;
    if (nnz > 0 && !colidx) return GNN_EINVAL;
    if (agg != GNN_AGG_GCN_SYM && agg != GNN_AGG_SAGE_MEAN && agg != GNN_AGG_GAT) return GNN_EINVAL;
    if (n_local + n_halo >= ((int64_t)1 << 31) || nnz >= ((int64_t)1 << 31)) return GNN_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    gnn_graph *g = new (std::nothrow) gnn_graph();
    if (!g) return GNN_ENOMEM;
    cudaGetDevice(&g->device);
    g->n_local = n_local;
    g->n_halo = n_halo;
    g->nnz = nnz;
    g->agg = agg;
    const int64_t nT = n_local + n_halo;
    gnn_status st = GNN_OK;
    auto fail = [&](gnn_status e) {
        cudaStreamSynchronize(s);
        destroy_graph(g);
        return e;
    };
#define TRY_CUDA(x)                                          \
    do {                                                     \
        cudaError_t e_ = (x);                                \
        if (e_ != cudaSuccess) return fail(cuda_status(e_)); \
    } while (0)
#define TRY(x)                         \
    do {                               \
        st = (x);                      \
        if (st != GNN_OK) return fail(st); \
    } while (0)
    TRY_CUDA(cudaMalloc((void **)&g->err, sizeof(int)));
    TRY_CUDA(cudaMemsetAsync(g->err, 0, sizeof(int), s));
    TRY_CUDA(cudaMalloc((void **)&g->rowptr, (size_t)(n_local + 1) * sizeof(int32_t)));
    TRY_CUDA(cudaMalloc((void **)&g->colidx, (size_t)(nnz > 0 ? nnz : 1) * sizeof(int32_t)));
    TRY_CUDA(cudaMemcpyAsync(g->rowptr, rowptr, (size_t)(n_local + 1) * sizeof(int32_t), cudaMemcpyDefault, s));
    if (nnz > 0)
        TRY_CUDA(cudaMemcpyAsync(g->colidx, colidx, (size_t)nnz * sizeof(int32_t), cudaMemcpyDefault, s));
    TRY(launch_validate_csr(g->rowptr, g->colidx, n_local, nT, nnz, g->err, s));
    int bad = 0;
    TRY_CUDA(cudaMemcpyAsync(&bad, g->err, sizeof(int), cudaMemcpyDeviceToHost, s));
    TRY_CUDA(cudaStreamSynchronize(s));
    if (bad) return fail(GNN_EINDEX);
    const bool gat = agg == GNN_AGG_GAT;
    // normalisation (GraphSAGE: inverse neighbour counts; attention: computed per call)
    if (gat) {
    } else if (agg == GNN_AGG_GCN_SYM) {
        TRY_CUDA(cudaMalloc((void **)&g->colw, (size_t)(nT > 0 ? nT : 1) * sizeof(float)));
        TRY(launch_gcn_dinv(g->rowptr, g->colidx, n_local, n_halo, nnz, deg, g->colw, s));
    } else {
        TRY_CUDA(cudaMalloc((void **)&g->colw, (size_t)(n_local > 0 ? n_local : 1) * sizeof(float)));
        TRY(launch_sage_invcnt(g->rowptr, g->colidx, n_local, g->colw, s));
    }
    // transpose
    TRY_CUDA(cudaMalloc((void **)&g->rowptrT, (size_t)(nT + 1) * sizeof(int32_t)));
    TRY_CUDA(cudaMalloc((void **)&g->colidxT, (size_t)(nnz > 0 ? nnz : 1) * sizeof(int32_t)));
    TRY_CUDA(cudaMalloc((void **)&g->permT, (size_t)(nnz > 0 ? nnz : 1) * sizeof(int32_t)));
    TRY(csr_transpose(g->rowptr, g->colidx, n_local, nT, nnz, g->rowptrT, g->colidxT, g->permT, s));
    // schedules
    TRY(build_schedule(g->rowptr, n_local, &g->fwd, s));
    TRY(build_schedule(g->rowptrT, nT, &g->bwd, s));
    // per-entry weights: the column factor of each entry (forward over the
    // block, backward over the transpose), 0 on the diagonal for the mean
    const bool sage = agg == GNN_AGG_SAGE_MEAN;
    if (!gat) {
        TRY_CUDA(cudaMalloc((void **)&g->wfwd, (size_t)(nnz > 0 ? nnz : 1) * sizeof(float)));
        TRY_CUDA(cudaMalloc((void **)&g->wbwd, (size_t)(nnz > 0 ? nnz : 1) * sizeof(float)));
        TRY(launch_entry_weights(g->rowptr, g->colidx, n_local, sage ? nullptr : g->colw, sage, g->wfwd, s));
        TRY(launch_entry_weights(g->rowptrT, g->colidxT, nT, g->colw, sage, g->wbwd, s));
    }
    // hotness tiers: forward columns by how often they are gathered (their
    // transpose row length), backward columns (local rows) by their row length
    TRY(tag_tiers(g->colidx, nnz, g->rowptrT, nT, &g->fwd, s));
    TRY(tag_tiers(g->colidxT, nnz, g->rowptr, n_local, &g->bwd, s));
    // each row's entries hottest tier first (stable), so the four rows of a
    // gather mostly share one L2 policy; the block's own copy is reordered in
    // place, the transpose gets a second copy (colidxT stays the stable
    // transpose that gnn_graph_copy_transpose hands out)
    // graph attention: the weights are the attention, computed per call; what
    // the graph keeps is where each transpose entry's attention sits in the
    // block (the permutations of the two sorts below, composed with permT)
    int32_t *fperm = nullptr, *tperm = nullptr, *iota = nullptr;
    if (gat && nnz > 0) {
        TRY_CUDA(cudaMalloc((void **)&g->t2b, (size_t)nnz * sizeof(int32_t)));
        TRY_CUDA(cudaMallocAsync((void **)&iota, (size_t)nnz * sizeof(int32_t), s));
        TRY(launch_iota(iota, nnz, s));
        if (g->fwd.tagged) TRY_CUDA(cudaMallocAsync((void **)&fperm, (size_t)nnz * sizeof(int32_t), s));
        if (g->bwd.tagged) TRY_CUDA(cudaMallocAsync((void **)&tperm, (size_t)nnz * sizeof(int32_t), s));
    }
    if (gat && nnz > 0 && (g->fwd.tagged || g->bwd.tagged)) {
        // the sorts carry entry indices (moved bit for bit as the weight payload)
        int32_t *tc = nullptr;
        TRY_CUDA(cudaMallocAsync((void **)&tc, (size_t)nnz * sizeof(int32_t), s));
        if (g->fwd.tagged) {
            TRY_CUDA(cudaMemcpyAsync(tc, g->colidx, (size_t)nnz * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
            TRY(sort_rows_by_tier(g->rowptr, n_local, tc, reinterpret_cast<const float *>(iota), g->colidx,
                                  reinterpret_cast<float *>(fperm), s));
        }
        if (g->bwd.tagged) {
            TRY_CUDA(cudaMalloc((void **)&g->colidxTa, (size_t)nnz * sizeof(int32_t)));
            TRY(sort_rows_by_tier(g->rowptrT, nT, g->colidxT, reinterpret_cast<const float *>(iota), g->colidxTa,
                                  reinterpret_cast<float *>(tperm), s));
        }
        TRY_CUDA(cudaFreeAsync(tc, s));
    }
    if (gat && nnz > 0) {
        TRY_CUDA(cudaMalloc((void **)&g->erow, (size_t)nnz * sizeof(int32_t)));
        TRY(launch_entry_rows(g->rowptr, n_local, g->erow, s));
        TRY(launch_gat_entry_map(fperm, tperm, g->permT, nnz, g->t2b, iota, s));
        TRY_CUDA(cudaFreeAsync(iota, s));
        if (fperm) TRY_CUDA(cudaFreeAsync(fperm, s));
        if (tperm) TRY_CUDA(cudaFreeAsync(tperm, s));
    }
    if (!gat && nnz > 0 && (g->fwd.tagged || g->bwd.tagged)) {
        int32_t *tc = nullptr;
        float *tw = nullptr;
        TRY_CUDA(cudaMallocAsync((void **)&tc, (size_t)nnz * sizeof(int32_t), s));
        TRY_CUDA(cudaMallocAsync((void **)&tw, (size_t)nnz * sizeof(float), s));
        if (g->fwd.tagged) {
            TRY_CUDA(cudaMemcpyAsync(tc, g->colidx, (size_t)nnz * sizeof(int32_t), cudaMemcpyDeviceToDevice, s));
            TRY_CUDA(cudaMemcpyAsync(tw, g->wfwd, (size_t)nnz * sizeof(float), cudaMemcpyDeviceToDevice, s));
            TRY(sort_rows_by_tier(g->rowptr, n_local, tc, tw, g->colidx, g->wfwd, s));
        }
        if (g->bwd.tagged) {
            TRY_CUDA(cudaMalloc((void **)&g->colidxTa, (size_t)nnz * sizeof(int32_t)));
            TRY_CUDA(cudaMemcpyAsync(tw, g->wbwd, (size_t)nnz * sizeof(float), cudaMemcpyDeviceToDevice, s));
            TRY(sort_rows_by_tier(g->rowptrT, nT, g->colidxT, tw, g->colidxTa, g->wbwd, s));
        }
        TRY_CUDA(cudaFreeAsync(tc, s));
        TRY_CUDA(cudaFreeAsync(tw, s));
    }
    // row ends, on the entries in their final order (attention: set per call)
    if (!gat) {
        TRY(launch_mark_row_ends(g->rowptr, n_local, g->wfwd, s));
        TRY(launch_mark_row_ends(g->rowptrT, nT, g->wbwd, s));
    }
    TRY_CUDA(cudaStreamSynchronize(s));
    TRY_CUDA(cudaGetLastError());
#undef TRY
#undef TRY_CUDA
    *out = g;
    return GNN_OK;
}

gnn_status gnn_graph_destroy(gnn_graph *g) {
    if (!g) return GNN_EINVAL;
    cudaError_t e = cudaDeviceSynchronize();
    destroy_graph(g);
    return e == cudaSuccess ? GNN_OK : GNN_ECUDA;
}

gnn_status gnn_graph_sizes(const gnn_graph *g, int64_t *n_local, int64_t *n_halo, int64_t *nnz) {
    if (!g) return GNN_EINVAL;
    if (n_local) *n_local = g->n_local;
    if (n_halo) *n_halo = g->n_halo;
    if (nnz) *nnz = g->nnz;
    return GNN_OK;
}

gnn_status gnn_graph_copy_transpose(const gnn_graph *g, int32_t *rowptrT, int32_t *colidxT, int32_t *permT,
                                    void *stream) {
    if (!g) return GNN_EINVAL;
    cudaStream_t s = as_stream(stream);
    const size_t nT1 = (size_t)(g->n_local + g->n_halo + 1) * sizeof(int32_t);
    const size_t nz = (size_t)g->nnz * sizeof(int32_t);
    if (rowptrT) GNN_CUDA_TRY(cudaMemcpyAsync(rowptrT, g->rowptrT, nT1, cudaMemcpyDeviceToDevice, s));
    if (colidxT && nz) {
        gnn_status st = copy_untagged(g->colidxT, colidxT, g->nnz, g->bwd.tagged ? kColMask : 0xffffffffu, s);
        if (st != GNN_OK) return st;
    }
    if (permT && nz) GNN_CUDA_TRY(cudaMemcpyAsync(permT, g->permT, nz, cudaMemcpyDeviceToDevice, s));
    return GNN_OK;
}

gnn_status gnn_get_error(gnn_graph *g) {
    if (!g) return GNN_EINVAL;
    GNN_CUDA_TRY(cudaDeviceSynchronize());
    int v = 0;
    GNN_CUDA_TRY(cudaMemcpy(&v, g->err, sizeof(int), cudaMemcpyDeviceToHost));
    GNN_CUDA_TRY(cudaMemset(g->err, 0, sizeof(int)));
    if (v & (kErrWaitTc | kErrWaitAgg)) return GNN_ETIMEOUT;
    return v ? GNN_EINDEX : GNN_OK;
}

gnn_status gnn_halo_pull(gnn_graph *g, const void *table, int64_t ld_table, int64_t n_table, const int64_t *halo_ids,
                         void *H, int64_t ld_h, int64_t f, gnn_dtype dtype, void *stream) {
    if (!g || !dtype_ok(dtype) || f <= 0 || n_table < 0) return GNN_EINVAL;
    if (g->n_halo == 0) return GNN_OK;
    if (!halo_ids || !operand_ok(table, n_table > 0 ? 1 : 0, ld_table, f, dtype) ||
        !operand_ok(H, g->n_local + g->n_halo, ld_h, f, dtype))
        return GNN_EINVAL;
    ProfScope prof(g, GNN_PROF_PULL, as_stream(stream));
    return launch_pull(table, ld_table, n_table, halo_ids, g->n_halo, H, ld_h, g->n_local, f, elem_size(dtype), g->err,
                       as_stream(stream));
}

gnn_status gnn_halo_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t f, const int64_t *local_ids, void *table,
                         int64_t ld_table, int64_t n_table, gnn_dtype dtype, void *stream) {
    if (!g || !dtype_ok(dtype) || f <= 0 || n_table < 0) return GNN_EINVAL;
    if (g->n_local == 0) return GNN_OK;
    if (!local_ids || !operand_ok(H, g->n_local, ld_h, f, dtype) ||
        !operand_ok(table, n_table > 0 ? 1 : 0, ld_table, f, dtype))
        return GNN_EINVAL;
    gnn_status st = ensure_claim(g, n_table);  // a first push to a larger table allocates (synchronising)
    if (st != GNN_OK) return st;
    ProfScope prof(g, GNN_PROF_PUSH, as_stream(stream));
    return launch_push(g, H, ld_h, g->n_local, f, local_ids, table, ld_table, n_table, elem_size(dtype),
                       as_stream(stream));
}

namespace {
bool codec_args_ok(const void *codes, int64_t ld_codes, const float *scale_zero, int64_t n_table, int bits,
                   int64_t f) {
    if (bits != 1 && bits != 2 && bits != 4 && bits != 8) return false;
    if (n_table < 0 || f <= 0 || ld_codes % 16 != 0 || ld_codes < (f + 7) / 8 * bits) return false;
    if (n_table > 0 && (!codes || !scale_zero || (reinterpret_cast<uintptr_t>(codes) & 15u) ||
                        (reinterpret_cast<uintptr_t>(scale_zero) & 7u)))
        return false;
    return true;
}
}  // namespace

gnn_status gnn_halo_push_quantized(gnn_graph *g, const void *H, int64_t ld_h, int64_t f, const int64_t *local_ids,
                                   uint8_t *codes, int64_t ld_codes, float *scale_zero, int64_t n_table, int bits,
                                   uint64_t seed, gnn_dtype dtype, void *stream) {
    if (!g || !dtype_ok(dtype) || !codec_args_ok(codes, ld_codes, scale_zero, n_table, bits, f)) return GNN_EINVAL;
    if (g->n_local == 0) return GNN_OK;
    if (!local_ids || !operand_ok(H, g->n_local, ld_h, f, dtype)) return GNN_EINVAL;
    gnn_status st = ensure_claim(g, n_table);  // a first push to a larger table allocates (synchronising)
    if (st != GNN_OK) return st;
    ProfScope prof(g, GNN_PROF_PUSH, as_stream(stream));
    return launch_codec_push(g, H, ld_h, g->n_local, f, local_ids, codes, ld_codes, scale_zero, n_table, bits, seed,
                             dtype, as_stream(stream));
}

gnn_status gnn_halo_pull_quantized(gnn_graph *g, const uint8_t *codes, int64_t ld_codes, const float *scale_zero,
                                   int64_t n_table, int bits, const int64_t *halo_ids, void *H, int64_t ld_h,
                                   int64_t f, gnn_dtype dtype, void *stream) {
    if (!g || !dtype_ok(dtype) || !codec_args_ok(codes, ld_codes, scale_zero, n_table, bits, f)) return GNN_EINVAL;
    if (g->n_halo == 0) return GNN_OK;
    if (!halo_ids || !operand_ok(H, g->n_local + g->n_halo, ld_h, f, dtype)) return GNN_EINVAL;
    ProfScope prof(g, GNN_PROF_PULL, as_stream(stream));
    return launch_codec_pull(codes, ld_codes, scale_zero, n_table, bits, halo_ids, g->n_halo, H, ld_h, g->n_local, f,
                             dtype, g->err, as_stream(stream));
}

gnn_status gnn_layer_forward(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W, int64_t f_out,
                             int relu, void *Z, int64_t ld_z, void *H_out, int64_t ld_out, gnn_dtype dtype,
                             void *stream) {
    if (g && g->agg == GNN_AGG_GAT) return GNN_EINVAL;  // attention layers: gnn_gat_forward / backward
    if (!g || !dtype_ok(dtype) || f_in <= 0 || f_out <= 0 || !W) return GNN_EINVAL;
    const bool sage = g->agg == GNN_AGG_SAGE_MEAN;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    const int64_t half = gnn_sage_half_offset(f_in, dtype);
    const int64_t K = sage ? 2 * f_in : f_in;
    const int64_t Kp = sage ? 2 * half : f_in;
    if (!operand_ok(H, nT, ld_h, f_in, dtype) || !operand_ok(Z, nL, ld_z, Kp, dtype) ||
        !operand_ok(H_out, nL, ld_out, f_out, dtype))
        return GNN_EINVAL;
    if (f_in * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    if (nL == 0) return GNN_OK;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const bool use_tc = dtype == GNN_BF16 && update_fwd_tc_supported(Kp, f_out) && !force_simt_update();
    const size_t wp_bytes = align_up((size_t)Kp * ldw * sizeof(float));
    const size_t wt_bytes = use_tc ? align_up(update_tc_wt_bytes(Kp, f_out)) : 0;
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->fwd, f_in));
    gnn_status st = ensure_workspace(g, wp_bytes + wt_bytes + part_bytes, s);
    if (st != GNN_OK) return st;
    float *Wp = static_cast<float *>(g->ws);
    void *wt = static_cast<char *>(g->ws) + wp_bytes;
    float *partial = reinterpret_cast<float *>(static_cast<char *>(g->ws) + wp_bytes + wt_bytes);
    { pack_w_kernel<<<(unsigned)ceil_div(Kp * ldw, 256), 256, 0, s>>>(W, K, f_out, f_in, half, sage, Kp, Wp, ldw,
                                                                      dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    AggParams p{};
    p.err = g->err;
    p.rowptr = g->rowptr;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidx);
    p.wts = g->wfwd;
    p.rowscale = g->colw;
    p.n_rows = nL;
    p.colmask = g->fwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->fwd, round_up(f_in * elem_size(dtype), 32));
    p.X = H;
    p.ldx = ld_h;
    p.n_x = nT;
    p.f = f_in;
    p.self_mode = sage ? SELF_COPY : SELF_NONE;
    p.out = Z;
    p.ldo = ld_z;
    p.out_off = sage ? half : 0;
    {
        ProfScope prof(g, GNN_PROF_AGG_FWD, s);
        st = launch_aggregate(p, g->fwd, dtype, partial, s);
    }
    if (st != GNN_OK) return st;
    ProfScope prof(g, GNN_PROF_UPD_FWD, s);
    if (use_tc) return launch_update_fwd_tc(Z, ld_z, nL, Kp, Wp, ldw, f_out, relu, H_out, ld_out, wt, g->err, s);
    return launch_update_fwd(Z, ld_z, nL, Kp, Wp, ldw, f_out, relu, H_out, ld_out, dtype, s);
}

gnn_status gnn_layer_backward(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                              const void *Z, int64_t ld_z, const float *W, int64_t f_in, int64_t f_out, int relu,
                              float *dW, void *dZ, int64_t ld_dz, void *dH, int64_t ld_dh, int want_halo_grad,
                              gnn_dtype dtype, gnn_dtype grad_dtype, void *stream) {
    if (g && g->agg == GNN_AGG_GAT) return GNN_EINVAL;  // attention layers: gnn_gat_forward / backward
    if (!g || !dtype_ok(dtype) || !dtype_ok(grad_dtype) || f_in <= 0 || f_out <= 0 || !W || !dW) return GNN_EINVAL;
    if (dtype == GNN_F32 && grad_dtype != GNN_F32) return GNN_EINVAL;  // fp32 activations keep fp32 gradients
    const bool mixed = dtype != grad_dtype;                              // bf16 activations, fp32 gradients
    const bool sage = g->agg == GNN_AGG_SAGE_MEAN;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    // Z's layout is that of the activations; dZ shares it column for column
    const int64_t half = gnn_sage_half_offset(f_in, dtype);
    const int64_t K = sage ? 2 * f_in : f_in;
    const int64_t Kp = sage ? 2 * half : f_in;
    const int64_t out_rows = want_halo_grad ? nT : nL;
    if (!operand_ok(G, nL, ld_g, f_out, grad_dtype) || !operand_ok(Z, nL, ld_z, Kp, dtype)) return GNN_EINVAL;
    if (relu && !operand_ok(H_out, nL, ld_out, f_out, dtype)) return GNN_EINVAL;
    if (dH && (!operand_ok(dH, out_rows, ld_dh, f_in, grad_dtype) || !operand_ok(dZ, nL, ld_dz, Kp, grad_dtype)))
        return GNN_EINVAL;
    if (f_in * elem_size(grad_dtype) > 4096 || f_in * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const bool use_tc = dtype == GNN_BF16 && update_bwd_tc_supported(Kp, f_out) && !force_simt_update();
    // the tensor cores take dY in bf16: the fp32 gradient is masked and rounded into a staging buffer
    const int64_t ldy = round_up(f_out, 8);
    const size_t y_bytes = (use_tc && mixed) ? align_up((size_t)nL * ldy * 2) : 0;
    const size_t wp_bytes = align_up((size_t)Kp * ldw * sizeof(float));
    const size_t dwp_bytes = sage ? align_up((size_t)Kp * f_out * sizeof(float)) : 0;
    const size_t wg_bytes = align_up(use_tc ? update_bwd_tc_ws_bytes(nL, Kp, f_out)
                                            : update_bwd_ws_bytes(nL, Kp, f_out, dtype));
    const size_t part_bytes = dH ? align_up(aggregate_partial_bytes(g->bwd, f_in)) : 0;
    gnn_status st = ensure_workspace(g, wp_bytes + dwp_bytes + wg_bytes + part_bytes + y_bytes, s);
    if (st != GNN_OK) return st;
    char *base = static_cast<char *>(g->ws);
    float *Wp = reinterpret_cast<float *>(base);
    float *dWp = sage ? reinterpret_cast<float *>(base + wp_bytes) : dW;
    float *wg = reinterpret_cast<float *>(base + wp_bytes + dwp_bytes);
    float *partial = reinterpret_cast<float *>(base + wp_bytes + dwp_bytes + wg_bytes);
    void *Ystage = base + wp_bytes + dwp_bytes + wg_bytes + part_bytes;
    { pack_w_kernel<<<(unsigned)ceil_div(Kp * ldw, 256), 256, 0, s>>>(W, K, f_out, f_in, half, sage, Kp, Wp, ldw,
                                                                      dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    {
        ProfScope prof(g, GNN_PROF_UPD_BWD, s);
        if (use_tc && mixed) {
            st = launch_grad_to_bf16(static_cast<const float *>(G), ld_g, relu ? H_out : nullptr, ld_out, nL, f_out,
                                     Ystage, ldy, s);
            if (st == GNN_OK)
                st = launch_update_bwd_tc(Ystage, ldy, nullptr, 0, 0, Z, ld_z, nL, Kp, Wp, ldw, f_out, dWp,
                                          dH ? dZ : nullptr, ld_dz, true, wg, g->err, s);
        } else if (use_tc) {
            st = launch_update_bwd_tc(G, ld_g, H_out, ld_out, relu, Z, ld_z, nL, Kp, Wp, ldw, f_out, dWp,
                                      dH ? dZ : nullptr, ld_dz, false, wg, g->err, s);
        } else {
            st = launch_update_bwd(G, ld_g, H_out, ld_out, relu, Z, ld_z, nL, Kp, Wp, ldw, f_out, dWp,
                                   dH ? dZ : nullptr, ld_dz, dtype, grad_dtype, wg, wg_bytes, s);
        }
    }
    if (st != GNN_OK) return st;
    if (sage) {
        { unpack_dw_kernel<<<(unsigned)ceil_div(K * f_out, 256), 256, 0, s>>>(dWp, f_out, f_in, half, dW); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    if (!dH) return GNN_OK;
    AggParams p{};
    p.err = g->err;
    p.rowptr = g->rowptrT;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidxTa ? g->colidxTa : g->colidxT);
    p.wts = g->wbwd;
    p.rowscale = sage ? nullptr : g->colw;
    p.n_rows = out_rows;
    p.colmask = g->bwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->bwd, round_up(f_in * elem_size(grad_dtype), 32));
    p.f = f_in;
    p.out = dH;
    p.ldo = ld_dh;
    p.out_off = 0;
    p.ldx = ld_dz;
    p.n_x = nL;
    if (sage) {
        p.self_mode = SELF_ADD;
        p.X = static_cast<const char *>(dZ) + half * elem_size(grad_dtype);
        p.self = dZ;
        p.ld_self = ld_dz;
        p.n_self = nL;
    } else {
        p.self_mode = SELF_NONE;
        p.X = dZ;
    }
    ProfScope prof(g, GNN_PROF_AGG_BWD, s);
    return launch_aggregate(p, g->bwd, grad_dtype, partial, s);
}

gnn_status gnn_layer_backward_reordered(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                                        const void *Z, int64_t ld_z, const float *W, int64_t f_in, int64_t f_out,
                                        int relu, float *dW, void *P, int64_t ld_p, void *dH, int64_t ld_dh,
                                        int want_halo_grad, gnn_dtype dtype, gnn_dtype grad_dtype, void *stream) {
    if (g && g->agg == GNN_AGG_GAT) return GNN_EINVAL;  // attention layers: gnn_gat_forward / backward
    if (!g || !dtype_ok(dtype) || !dtype_ok(grad_dtype) || f_in <= 0 || f_out <= 0 || !W || !dW || !dH)
        return GNN_EINVAL;
    // the GCN layer, bf16 activations with fp32 gradients, on the tensor cores
    if (g->agg != GNN_AGG_GCN_SYM || dtype != GNN_BF16 || grad_dtype != GNN_F32) return GNN_EUNSUPPORTED;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    const int64_t out_rows = want_halo_grad ? nT : nL;
    if (!operand_ok(G, nL, ld_g, f_out, GNN_F32) || !operand_ok(Z, nL, ld_z, f_in, GNN_BF16) ||
        !operand_ok(P, out_rows, ld_p, f_out, GNN_BF16) || !operand_ok(dH, out_rows, ld_dh, f_in, GNN_F32))
        return GNN_EINVAL;
    if (relu && !operand_ok(H_out, nL, ld_out, f_out, GNN_BF16)) return GNN_EINVAL;
    if (f_out * 2 > 4096 || !update_bwd_tc_supported(f_in, f_out) || force_simt_update()) return GNN_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const int64_t ldy = round_up(f_out, 8);
    const size_t wp_bytes = align_up((size_t)f_in * ldw * sizeof(float));
    const size_t y_bytes = align_up((size_t)(nL > 0 ? nL : 1) * ldy * 2);
    const size_t wg_bytes = align_up(update_bwd_tc_ws_bytes(out_rows > nL ? out_rows : nL, f_in, f_out));
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->bwd, f_out));
    gnn_status st = ensure_workspace(g, wp_bytes + y_bytes + wg_bytes + part_bytes, s);
    if (st != GNN_OK) return st;
    char *base = static_cast<char *>(g->ws);
    float *Wp = reinterpret_cast<float *>(base);
    void *Y = base + wp_bytes;
    float *wg = reinterpret_cast<float *>(base + wp_bytes + y_bytes);
    float *partial = reinterpret_cast<float *>(base + wp_bytes + y_bytes + wg_bytes);
    { pack_w_kernel<<<(unsigned)ceil_div(f_in * ldw, 256), 256, 0, s>>>(W, f_in, f_out, f_in, f_in, 0, f_in, Wp, ldw,
                                                                        true); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    {
        // dY = G * 1[H_out > 0] rounded to bf16, and dW = Z^T dY
        ProfScope prof(g, GNN_PROF_UPD_BWD, s);
        st = launch_grad_to_bf16(static_cast<const float *>(G), ld_g, relu ? H_out : nullptr, ld_out, nL, f_out, Y,
                                 ldy, s);
        if (st == GNN_OK)
            st = launch_update_bwd_tc(Y, ldy, nullptr, 0, 0, Z, ld_z, nL, f_in, Wp, ldw, f_out, dW, nullptr, 0, true,
                                      wg, g->err, s);
    }
    if (st != GNN_OK) return st;
    {
        // P = A_hat^T dY over the output rows (gathering the bf16 dY rows), stored in bf16: the product's operand
        AggParams p{};
        p.err = g->err;
        p.rowptr = g->rowptrT;
        p.colidx = reinterpret_cast<const uint32_t *>(g->colidxTa ? g->colidxTa : g->colidxT);
        p.wts = g->wbwd;
        p.rowscale = g->colw;
        p.n_rows = out_rows;
        p.colmask = g->bwd.tagged ? kColMask : 0xffffffffu;
        p.hot_tier = hot_tier_for(g->bwd, round_up(f_out * 2, 32));
        p.X = Y;
        p.ldx = ldy;
        p.n_x = nL;
        p.f = f_out;
        p.self_mode = SELF_NONE;
        p.out = P;
        p.ldo = ld_p;
        p.out_off = 0;
        ProfScope prof(g, GNN_PROF_AGG_BWD, s);
        st = launch_aggregate(p, g->bwd, GNN_BF16, partial, s);
    }
    if (st != GNN_OK) return st;
    // dH = P W^T over the output rows, fp32
    ProfScope prof(g, GNN_PROF_UPD_BWD, s);
    return launch_update_bwd_tc(P, ld_p, nullptr, 0, 0, nullptr, 0, out_rows, f_in, Wp, ldw, f_out, nullptr, dH, ld_dh,
                                true, wg, g->err, s);
}

gnn_status gnn_layer_forward_narrow(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W,
                                    int64_t f_out, int relu, void *T, int64_t ld_t, void *H_out, int64_t ld_out,
                                    gnn_dtype dtype, void *stream) {
    if (g && g->agg == GNN_AGG_GAT) return GNN_EINVAL;  // attention layers: gnn_gat_forward / backward
    if (!g || !dtype_ok(dtype) || f_in <= 0 || f_out <= 0 || !W) return GNN_EINVAL;
    if (g->agg != GNN_AGG_GCN_SYM) return GNN_EUNSUPPORTED;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    if (!operand_ok(H, nT, ld_h, f_in, dtype) || !operand_ok(T, nT, ld_t, f_out, dtype) ||
        !operand_ok(H_out, nL, ld_out, f_out, dtype))
        return GNN_EINVAL;
    if (f_out * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    if (nL == 0) return GNN_OK;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const bool use_tc = dtype == GNN_BF16 && update_fwd_tc_supported(f_in, f_out) && !force_simt_update();
    const size_t wp_bytes = align_up((size_t)f_in * ldw * sizeof(float));
    const size_t wt_bytes = use_tc ? align_up(update_tc_wt_bytes(f_in, f_out)) : 0;
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->fwd, f_out));
    gnn_status st = ensure_workspace(g, wp_bytes + wt_bytes + part_bytes, s);
    if (st != GNN_OK) return st;
    float *Wp = static_cast<float *>(g->ws);
    void *wt = static_cast<char *>(g->ws) + wp_bytes;
    float *partial = reinterpret_cast<float *>(static_cast<char *>(g->ws) + wp_bytes + wt_bytes);
    { pack_w_kernel<<<(unsigned)ceil_div(f_in * ldw, 256), 256, 0, s>>>(W, f_in, f_out, f_in, f_in, 0, f_in, Wp, ldw,
                                                                        dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    {
        // T = H W over every row, local and halo (the multiplication first)
        ProfScope prof(g, GNN_PROF_UPD_FWD, s);
        st = use_tc ? launch_update_fwd_tc(H, ld_h, nT, f_in, Wp, ldw, f_out, 0, T, ld_t, wt, g->err, s)
                    : launch_update_fwd(H, ld_h, nT, f_in, Wp, ldw, f_out, 0, T, ld_t, dtype, s);
    }
    if (st != GNN_OK) return st;
    AggParams p{};
    p.err = g->err;
    p.rowptr = g->rowptr;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidx);
    p.wts = g->wfwd;
    p.rowscale = g->colw;
    p.n_rows = nL;
    p.colmask = g->fwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->fwd, round_up(f_out * elem_size(dtype), 32));
    p.X = T;
    p.ldx = ld_t;
    p.n_x = nT;
    p.f = f_out;
    p.self_mode = SELF_NONE;
    p.out = H_out;
    p.ldo = ld_out;
    p.out_off = 0;
    p.relu = relu;
    ProfScope prof(g, GNN_PROF_AGG_FWD, s);
    return launch_aggregate(p, g->fwd, dtype, partial, s);
}

gnn_status gnn_layer_backward_narrow(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                                     const void *H, int64_t ld_h, const float *W, int64_t f_in, int64_t f_out,
                                     int relu, float *dW, void *P, int64_t ld_p, void *dH, int64_t ld_dh,
                                     gnn_dtype dtype, void *stream) {
    if (g && g->agg == GNN_AGG_GAT) return GNN_EINVAL;  // attention layers: gnn_gat_forward / backward
    if (!g || !dtype_ok(dtype) || f_in <= 0 || f_out <= 0 || !W || !dW) return GNN_EINVAL;
    if (g->agg != GNN_AGG_GCN_SYM) return GNN_EUNSUPPORTED;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    if (!operand_ok(G, nL, ld_g, f_out, dtype) || !operand_ok(H, nT, ld_h, f_in, dtype) ||
        !operand_ok(P, nT, ld_p, f_out, dtype))
        return GNN_EINVAL;
    if (relu && !operand_ok(H_out, nL, ld_out, f_out, dtype)) return GNN_EINVAL;
    if (dH && !operand_ok(dH, nT, ld_dh, f_in, dtype)) return GNN_EINVAL;
    if (f_out * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const int64_t ldy = round_up(f_out, elems_per_16b(dtype));
    const bool use_tc = dtype == GNN_BF16 && update_bwd_tc_supported(f_in, f_out) && !force_simt_update();
    const size_t wp_bytes = align_up((size_t)f_in * ldw * sizeof(float));
    const size_t y_bytes = relu ? align_up((size_t)nL * ldy * elem_size(dtype)) : 0;
    const size_t wg_bytes = align_up(use_tc ? update_bwd_tc_ws_bytes(nT, f_in, f_out)
                                            : update_bwd_ws_bytes(nT, f_in, f_out, dtype));
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->bwd, f_out));
    gnn_status st = ensure_workspace(g, wp_bytes + y_bytes + wg_bytes + part_bytes, s);
    if (st != GNN_OK) return st;
    char *base = static_cast<char *>(g->ws);
    float *Wp = reinterpret_cast<float *>(base);
    void *Y = base + wp_bytes;
    float *wg = reinterpret_cast<float *>(base + wp_bytes + y_bytes);
    float *partial = reinterpret_cast<float *>(base + wp_bytes + y_bytes + wg_bytes);
    { pack_w_kernel<<<(unsigned)ceil_div(f_in * ldw, 256), 256, 0, s>>>(W, f_in, f_out, f_in, f_in, 0, f_in, Wp, ldw,
                                                                        dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    // dY = G (masked by the ReLU), then P = A_hat^T dY over every row, local and halo
    const void *dY = G;
    int64_t ld_y = ld_g;
    if (relu && nL > 0) {
        const unsigned blocks = (unsigned)ceil_div(nL * f_out, 256);
        if (dtype == GNN_BF16)
            { relu_mask_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(G), ld_g,
                                                                     static_cast<const __nv_bfloat16 *>(H_out), ld_out,
                                                                     nL, f_out, static_cast<__nv_bfloat16 *>(Y), ldy); GNN_LAUNCHED(1); }
        else
            { relu_mask_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(G), ld_g,
                                                             static_cast<const float *>(H_out), ld_out, nL, f_out,
                                                             static_cast<float *>(Y), ldy); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        dY = Y;
        ld_y = ldy;
    }
    {
        AggParams p{};
        p.err = g->err;
        p.rowptr = g->rowptrT;
        p.colidx = reinterpret_cast<const uint32_t *>(g->colidxTa ? g->colidxTa : g->colidxT);
        p.wts = g->wbwd;
        p.rowscale = g->colw;
        p.n_rows = nT;
        p.colmask = g->bwd.tagged ? kColMask : 0xffffffffu;
        p.hot_tier = hot_tier_for(g->bwd, round_up(f_out * elem_size(dtype), 32));
        p.X = dY;
        p.ldx = ld_y;
        p.n_x = nL;
        p.f = f_out;
        p.self_mode = SELF_NONE;
        p.out = P;
        p.ldo = ld_p;
        p.out_off = 0;
        ProfScope prof(g, GNN_PROF_AGG_BWD, s);
        st = launch_aggregate(p, g->bwd, dtype, partial, s);
    }
    if (st != GNN_OK) return st;
    // dW = H^T P and dH = P W^T over every row
    ProfScope prof(g, GNN_PROF_UPD_BWD, s);
    if (use_tc)
        return launch_update_bwd_tc(P, ld_p, nullptr, 0, 0, H, ld_h, nT, f_in, Wp, ldw, f_out, dW, dH, ld_dh, false,
                                    wg, g->err, s);
    return launch_update_bwd(P, ld_p, nullptr, 0, 0, H, ld_h, nT, f_in, Wp, ldw, f_out, dW, dH, ld_dh, dtype, dtype,
                             wg, wg_bytes, s);
}

gnn_status gnn_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                          int64_t ld_g, float *row_loss, float *loss, gnn_dtype dtype, gnn_dtype grad_dtype,
                          void *stream) {
    if (!dtype_ok(dtype) || !dtype_ok(grad_dtype) || n < 0 || C <= 0 || !loss) return GNN_EINVAL;
    if (n > 0 && (!logits || !labels || !G || !row_loss || ld < C || ld_g < C)) return GNN_EINVAL;
    return launch_softmax_ce(logits, ld, n, C, labels, G, ld_g, row_loss, loss, n, dtype, grad_dtype,
                             as_stream(stream));
}

gnn_status gnn_softmax_ce_partial(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels,
                                  void *G, int64_t ld_g, float *row_loss, float *loss, int64_t n_mean,
                                  gnn_dtype dtype, gnn_dtype grad_dtype, void *stream) {
    if (!dtype_ok(dtype) || !dtype_ok(grad_dtype) || n < 0 || C <= 0 || !loss || n_mean < n || n_mean <= 0)
        return GNN_EINVAL;
    if (n > 0 && (!logits || !labels || !G || !row_loss || ld < C || ld_g < C)) return GNN_EINVAL;
    return launch_softmax_ce(logits, ld, n, C, labels, G, ld_g, row_loss, loss, n_mean, dtype, grad_dtype,
                             as_stream(stream));
}

gnn_status gnn_halo_grad_send(gnn_graph *g, const void *dH, int64_t ld_dh, int64_t f, const int64_t *halo_ids,
                              float *gtable, int64_t ld_gt, int64_t n_table, gnn_dtype dtype, void *stream) {
    if (!g || !dtype_ok(dtype) || f <= 0 || n_table < 0) return GNN_EINVAL;
    if (g->n_halo == 0) return GNN_OK;
    if (!halo_ids || !operand_ok(dH, g->n_local + g->n_halo, ld_dh, f, dtype) ||
        !operand_ok(gtable, n_table > 0 ? 1 : 0, ld_gt, f, GNN_F32))
        return GNN_EINVAL;
    gnn_status st = ensure_claim(g, n_table);
    if (st != GNN_OK) return st;
    return launch_grad_send(g, dH, ld_dh, f, halo_ids, gtable, ld_gt, n_table, dtype, as_stream(stream));
}

gnn_status gnn_halo_grad_recv(gnn_graph *g, const float *gtable, int64_t ld_gt, int64_t n_table,
                              const int64_t *local_ids, void *dH, int64_t ld_dh, int64_t f, gnn_dtype dtype,
                              void *stream) {
    if (!g || !dtype_ok(dtype) || f <= 0 || n_table < 0) return GNN_EINVAL;
    if (g->n_local == 0) return GNN_OK;
    if (!local_ids || !operand_ok(dH, g->n_local, ld_dh, f, dtype) ||
        !operand_ok(gtable, n_table > 0 ? 1 : 0, ld_gt, f, GNN_F32))
        return GNN_EINVAL;
    return launch_grad_recv(g, gtable, ld_gt, n_table, local_ids, dH, ld_dh, f, dtype, as_stream(stream));
}

gnn_status gnn_gat_forward(gnn_graph *g, const void *H, int64_t ld_h, int64_t f_in, const float *W,
                           const float *a_src, const float *a_dst, int64_t f_out, int relu, void *T, int64_t ld_t,
                           float *scores, float *alpha, void *H_out, int64_t ld_out, gnn_dtype dtype, void *stream) {
    if (!g || g->agg != GNN_AGG_GAT || !dtype_ok(dtype) || f_in <= 0 || f_out <= 0 || !W || !a_src || !a_dst)
        return GNN_EINVAL;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    if (!operand_ok(H, nT, ld_h, f_in, dtype) || !operand_ok(T, nT, ld_t, f_out, dtype) ||
        !operand_ok(H_out, nL, ld_out, f_out, dtype) || (nT > 0 && !scores) || (g->nnz > 0 && !alpha))
        return GNN_EINVAL;
    if (f_out * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    if (nL == 0) return GNN_OK;
    cudaStream_t s = as_stream(stream);
    const int64_t ldw = round_up(f_out, 4);
    const bool use_tc = dtype == GNN_BF16 && update_fwd_tc_supported(f_in, f_out) && !force_simt_update();
    const size_t wp_bytes = align_up((size_t)f_in * ldw * sizeof(float));
    const size_t wt_bytes = use_tc ? align_up(update_tc_wt_bytes(f_in, f_out)) : 0;
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->fwd, f_out));
    gnn_status st = ensure_workspace(g, wp_bytes + wt_bytes + part_bytes, s);
    if (st != GNN_OK) return st;
    float *Wp = static_cast<float *>(g->ws);
    void *wt = static_cast<char *>(g->ws) + wp_bytes;
    float *partial = reinterpret_cast<float *>(static_cast<char *>(g->ws) + wp_bytes + wt_bytes);
    { pack_w_kernel<<<(unsigned)ceil_div(f_in * ldw, 256), 256, 0, s>>>(W, f_in, f_out, f_in, f_in, 0, f_in, Wp, ldw,
                                                                        dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    {
        // T = H W over every row, local and halo
        ProfScope prof(g, GNN_PROF_UPD_FWD, s);
        st = use_tc ? launch_update_fwd_tc(H, ld_h, nT, f_in, Wp, ldw, f_out, 0, T, ld_t, wt, g->err, s)
                    : launch_update_fwd(H, ld_h, nT, f_in, Wp, ldw, f_out, 0, T, ld_t, dtype, s);
    }
    if (st != GNN_OK) return st;
    float *s_src = scores, *s_dst = scores + nT;
    st = launch_gat_scores(T, ld_t, nT, nL, f_out, a_src, a_dst, s_src, s_dst, dtype, s);
    if (st != GNN_OK) return st;
    st = launch_gat_softmax(g, s_src, s_dst, alpha, s);
    if (st != GNN_OK) return st;
    AggParams p{};
    p.err = g->err;
    p.rowptr = g->rowptr;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidx);
    p.wts = alpha;
    p.rowscale = nullptr;
    p.n_rows = nL;
    p.colmask = g->fwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->fwd, round_up(f_out * elem_size(dtype), 32));
    p.X = T;
    p.ldx = ld_t;
    p.n_x = nT;
    p.f = f_out;
    p.self_mode = SELF_NONE;
    p.out = H_out;
    p.ldo = ld_out;
    p.relu = relu;
    ProfScope prof(g, GNN_PROF_AGG_FWD, s);
    return launch_aggregate(p, g->fwd, dtype, partial, s);
}

gnn_status gnn_gat_backward(gnn_graph *g, const void *G, int64_t ld_g, const void *H_out, int64_t ld_out,
                            const void *H, int64_t ld_h, int64_t f_in, const float *W, const float *a_src,
                            const float *a_dst, int64_t f_out, int relu, const void *T, int64_t ld_t,
                            const float *scores, const float *alpha, float *dW, float *da_src, float *da_dst,
                            void *dT, int64_t ld_dt, void *dH, int64_t ld_dh, gnn_dtype dtype, gnn_dtype grad_dtype,
                            void *stream) {
    if (!g || g->agg != GNN_AGG_GAT || !dtype_ok(dtype) || !dtype_ok(grad_dtype) || f_in <= 0 || f_out <= 0 || !W ||
        !a_src || !a_dst || !dW || !da_src || !da_dst)
        return GNN_EINVAL;
    if (dtype == GNN_F32 && grad_dtype != GNN_F32) return GNN_EINVAL;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    if (!operand_ok(G, nL, ld_g, f_out, grad_dtype) || !operand_ok(H, nT, ld_h, f_in, dtype) ||
        !operand_ok(T, nT, ld_t, f_out, dtype) || !operand_ok(dT, nT, ld_dt, f_out, grad_dtype) ||
        (relu && !operand_ok(H_out, nL, ld_out, f_out, dtype)) || (dH && !operand_ok(dH, nT, ld_dh, f_in, grad_dtype)) ||
        (nT > 0 && !scores) || (g->nnz > 0 && !alpha))
        return GNN_EINVAL;
    if (f_out * elem_size(grad_dtype) > 4096) return GNN_EUNSUPPORTED;
    cudaStream_t s = as_stream(stream);
    const bool mixed = dtype != grad_dtype;
    const int64_t ldw = round_up(f_out, 4);
    const int64_t ldy = round_up(f_out, elems_per_16b(grad_dtype));
    const int64_t ldb = round_up(f_out, 8);
    const bool use_tc = dtype == GNN_BF16 && update_bwd_tc_supported(f_in, f_out) && !force_simt_update();
    const size_t wp_bytes = align_up((size_t)f_in * ldw * sizeof(float));
    const size_t y_bytes = align_up((size_t)(nL > 0 ? nL : 1) * ldy * elem_size(grad_dtype));
    const size_t e_bytes = align_up((size_t)(g->nnz > 0 ? g->nnz : 1) * sizeof(float));  // dz, then alphaT
    const size_t v_bytes = align_up((size_t)(nT + nL + 1) * sizeof(float));                // ds_src, ds_dst
    const size_t c_bytes = align_up(std::max(gat_colsum_ws_floats(nT, f_out), (size_t)1) * sizeof(float));
    const size_t b_bytes = (use_tc && mixed) ? align_up((size_t)(nT > 0 ? nT : 1) * ldb * 2) : 0;
    const size_t wg_bytes = align_up(use_tc ? update_bwd_tc_ws_bytes(nT, f_in, f_out)
                                            : update_bwd_ws_bytes(nT, f_in, f_out, dtype));
    const size_t part_bytes = align_up(aggregate_partial_bytes(g->bwd, f_out));
    gnn_status st = ensure_workspace(g, wp_bytes + y_bytes + 2 * e_bytes + v_bytes + c_bytes + b_bytes + wg_bytes +
                                            part_bytes, s);
    if (st != GNN_OK) return st;
    char *base = static_cast<char *>(g->ws);
    float *Wp = reinterpret_cast<float *>(base);
    char *q = base + wp_bytes;
    void *Y = q;
    q += y_bytes;
    float *dz = reinterpret_cast<float *>(q);
    q += e_bytes;
    float *alphaT = reinterpret_cast<float *>(q);
    q += e_bytes;
    float *ds_src = reinterpret_cast<float *>(q), *ds_dst = ds_src + nT;
    q += v_bytes;
    float *cws = reinterpret_cast<float *>(q);
    q += c_bytes;
    void *dTb = q;
    q += b_bytes;
    float *wg = reinterpret_cast<float *>(q);
    q += wg_bytes;
    float *partial = reinterpret_cast<float *>(q);
    const float *s_src = scores, *s_dst = scores + nT;
    { pack_w_kernel<<<(unsigned)ceil_div(f_in * ldw, 256), 256, 0, s>>>(W, f_in, f_out, f_in, f_in, 0, f_in, Wp, ldw,
                                                                        dtype == GNN_BF16); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    // dY, the attention's backward per entry (dz) and per row (ds_dst), then over the transpose (ds_src, alphaT)
    st = launch_gat_mask(G, ld_g, relu ? H_out : nullptr, ld_out, nL, f_out, Y, ldy, dtype, grad_dtype, s);
    if (st == GNN_OK)
        st = launch_gat_edge_backward(g, s_src, s_dst, alpha, Y, ldy, T, ld_t, f_out, dz, ds_dst, dtype, grad_dtype, s);
    if (st == GNN_OK) st = launch_gat_transpose(g, dz, alpha, ds_src, alphaT, s);
    if (st != GNN_OK) return st;
    {
        // dT = sum over the transpose of alpha dY, then the rank-1 terms of the scores
        AggParams p{};
        p.err = g->err;
        p.rowptr = g->rowptrT;
        p.colidx = reinterpret_cast<const uint32_t *>(g->colidxTa ? g->colidxTa : g->colidxT);
        p.wts = alphaT;
        p.rowscale = nullptr;
        p.n_rows = nT;
        p.colmask = g->bwd.tagged ? kColMask : 0xffffffffu;
        p.hot_tier = hot_tier_for(g->bwd, round_up(f_out * elem_size(grad_dtype), 32));
        p.X = Y;
        p.ldx = ldy;
        p.n_x = nL;
        p.f = f_out;
        p.self_mode = SELF_NONE;
        p.out = dT;
        p.ldo = ld_dt;
        ProfScope prof(g, GNN_PROF_AGG_BWD, s);
        st = launch_aggregate(p, g->bwd, grad_dtype, partial, s);
    }
    if (st == GNN_OK) st = launch_gat_rank1(dT, ld_dt, nT, nL, f_out, ds_src, ds_dst, a_src, a_dst, grad_dtype, s);
    if (st == GNN_OK) st = launch_gat_colsum(T, ld_t, nT, f_out, ds_src, da_src, cws, dtype, s);
    if (st == GNN_OK) st = launch_gat_colsum(T, ld_t, nL, f_out, ds_dst, da_dst, cws, dtype, s);
    if (st != GNN_OK) return st;
    // dW = H^T dT and dH = dT W^T over every row (bf16 activations: dT is a bf16 operand)
    ProfScope prof(g, GNN_PROF_UPD_BWD, s);
    if (use_tc && mixed) {
        st = launch_grad_to_bf16(static_cast<const float *>(dT), ld_dt, nullptr, 0, nT, f_out, dTb, ldb, s);
        if (st != GNN_OK) return st;
        return launch_update_bwd_tc(dTb, ldb, nullptr, 0, 0, H, ld_h, nT, f_in, Wp, ldw, f_out, dW, dH, ld_dh, true,
                                    wg, g->err, s);
    }
    if (use_tc)
        return launch_update_bwd_tc(dT, ld_dt, nullptr, 0, 0, H, ld_h, nT, f_in, Wp, ldw, f_out, dW, dH, ld_dh, false,
                                    wg, g->err, s);
    return launch_update_bwd(dT, ld_dt, nullptr, 0, 0, H, ld_h, nT, f_in, Wp, ldw, f_out, dW, dH, ld_dh, dtype,
                             grad_dtype, wg, wg_bytes, s);
}

gnn_status gnn_quantize_rows(const void *X, int64_t ld_x, int64_t n, int64_t f, const int64_t *keys, int bits,
                             uint64_t seed, uint8_t *codes, int64_t ld_codes, float *scale_zero, gnn_dtype dtype,
                             void *stream) {
    if (!dtype_ok(dtype) || n < 0 || !codec_args_ok(codes, ld_codes, scale_zero, n, bits, f)) return GNN_EINVAL;
    if (n == 0) return GNN_OK;
    if (!keys || !operand_ok(X, n, ld_x, f, dtype)) return GNN_EINVAL;
    return launch_quantize_rows(X, ld_x, n, f, keys, bits, seed, codes, ld_codes, scale_zero, dtype,
                                as_stream(stream));
}

gnn_status gnn_dequantize_rows(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n, int64_t f,
                               int bits, const int64_t *ids, void *dst, int64_t ld_dst, int64_t n_dst, int add,
                               gnn_dtype dtype, int *err, void *stream) {
    if (!dtype_ok(dtype) || n < 0 || n_dst < 0 || !codec_args_ok(codes, ld_codes, scale_zero, n, bits, f))
        return GNN_EINVAL;
    if (n == 0) return GNN_OK;
    if (!operand_ok(dst, n_dst > 0 ? 1 : 0, ld_dst, f, dtype) || (!ids && n_dst < n)) return GNN_EINVAL;
    return launch_dequantize_rows(codes, ld_codes, scale_zero, n, f, bits, ids, dst, ld_dst, n_dst, add, dtype, err,
                                  as_stream(stream));
}

gnn_status gnn_gather_rows(const void *src, int64_t ld_src, int64_t n_src, const int64_t *ids, int64_t n, void *dst,
                           int64_t ld_dst, int64_t f, gnn_dtype dtype, int *err, void *stream) {
    if (!dtype_ok(dtype) || n < 0 || n_src < 0 || f <= 0) return GNN_EINVAL;
    if (n == 0) return GNN_OK;
    if (!ids || !operand_ok(src, n_src > 0 ? 1 : 0, ld_src, f, dtype) || !operand_ok(dst, n, ld_dst, f, dtype))
        return GNN_EINVAL;
    return launch_gather_rows(src, ld_src, n_src, ids, n, dst, ld_dst, f, dtype, err, as_stream(stream));
}

gnn_status gnn_scatter_add_rows(const void *src, int64_t ld_src, const int64_t *ids, int64_t n, void *dst,
                                int64_t ld_dst, int64_t n_dst, int64_t f, gnn_dtype dtype, int *err, void *stream) {
    if (!dtype_ok(dtype) || n < 0 || n_dst < 0 || f <= 0) return GNN_EINVAL;
    if (n == 0) return GNN_OK;
    if (!ids || !operand_ok(src, n, ld_src, f, dtype) || !operand_ok(dst, n_dst > 0 ? 1 : 0, ld_dst, f, dtype))
        return GNN_EINVAL;
    return launch_scatter_add_rows(src, ld_src, ids, n, dst, ld_dst, n_dst, f, dtype, err, as_stream(stream));
}

}  // extern "C"
