// halo.cu - pull and push between the partition and its table of stale
// representations (DIGEST page, system design, Fig. 1(c): pull H_out <- H~_out,
// push H_in -> H~_in).  The pages note that rows are independent, so the I/O
// parallelises at the granularity of a vertex; here a group of lanes moves one
// row with 16-byte vector copies.  Both are bit-exact copies.
#include <type_traits>

#include "gnn_internal.cuh"

namespace gnn {

namespace {

constexpr uint32_t kCountMask = 3u;  // low bits of a claim word: 0, 1 or 2 (= repeated)

constexpr int kRowsPerGroup = 8;  // rows a lane group moves at once (their loads are all in flight)

// Copy kRowsPerGroup rows of a lane group: row k goes from src + sidx(k) *
// sbytes to dst + didx(k) * dbytes.  One of the two indices is computed from
// the group's first row, the other comes from an id array (held as int64 in
// `ix`, -1 = skip the row).  Full 16-byte vectors first, every row's load
// issued before the stores, then (when nbytes is not a multiple of 16) the
// element tail.  GATHER: the ids index the source (pull); else the
// destination (push).  The vectors copied are q0, q0 + LPR, ... of each row
// (q0 = sub unless the caller moved the first one itself).
template <int LPR, bool GATHER>
__device__ __forceinline__ void copy_rows(const char *__restrict__ src, int64_t sbytes, char *__restrict__ dst,
                                          int64_t dbytes, int64_t first, const int64_t (&ix)[kRowsPerGroup],
                                          int64_t nbytes, int es, int sub, int64_t q0) {
    const int64_t nvec = nbytes / 16;
    for (int64_t q = q0; q < nvec; q += LPR) {
        uint4 v[kRowsPerGroup];
#pragma unroll
        for (int k = 0; k < kRowsPerGroup; ++k) {
            const int64_t si = GATHER ? ix[k] : first + k;
            if (ix[k] >= 0) v[k] = __ldg(reinterpret_cast<const uint4 *>(src + si * sbytes) + q);
        }
#pragma unroll
        for (int k = 0; k < kRowsPerGroup; ++k) {
            const int64_t di = GATHER ? first + k : ix[k];
            if (ix[k] >= 0) reinterpret_cast<uint4 *>(dst + di * dbytes)[q] = v[k];
        }
    }
    if (sub == 0 && nvec * 16 < nbytes) {
        const int64_t tail0 = nvec * 16;
#pragma unroll
        for (int k = 0; k < kRowsPerGroup; ++k) {
            if (ix[k] < 0) continue;
            const char *s = src + (GATHER ? ix[k] : first + k) * sbytes;
            char *d = dst + (GATHER ? first + k : ix[k]) * dbytes;
            if (es == 4) {
                for (int64_t b = tail0; b < nbytes; b += 4)
                    *reinterpret_cast<uint32_t *>(d + b) = *reinterpret_cast<const uint32_t *>(s + b);
            } else {
                for (int64_t b = tail0; b < nbytes; b += 2)
                    *reinterpret_cast<uint16_t *>(d + b) = *reinterpret_cast<const uint16_t *>(s + b);
            }
        }
    }
}

template <int LPR>
__global__ void __launch_bounds__(256, 3) pull_kernel(const char *__restrict__ table, int64_t row_bytes_t, int64_t n_table,
                                                   const int64_t *__restrict__ ids, int64_t n_ids,
                                                   char *__restrict__ H, int64_t row_bytes_h, int64_t row0,
                                                   int64_t nbytes, int es, int *err) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t i0 = (t / LPR) * kRowsPerGroup;
    const int sub = (int)(t % LPR);
    if (i0 >= n_ids) return;
    int64_t ix[kRowsPerGroup];
#pragma unroll
    for (int k = 0; k < kRowsPerGroup; ++k) {
        ix[k] = -1;
        const int64_t i = i0 + k;
        if (i < n_ids) {
            const int64_t id = __ldg(ids + i);
            if (id < 0 || id >= n_table) {
                if (sub == 0) atomicOr(err, 1);
            } else {
                ix[k] = id;
            }
        }
    }
    copy_rows<LPR, true>(table, row_bytes_t, H, row_bytes_h, row0 + i0, ix, nbytes, es, sub, sub);
}

// claim word = (generation << 2) | min(count, 2)
__global__ void push_claim_kernel(const int64_t *__restrict__ ids, int64_t n, int64_t n_table, uint32_t *claim,
                                  uint32_t gen, int *err) {
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= n) return;
    const int64_t id = ids[v];
    if (id < 0 || id >= n_table) {
        atomicOr(err, 1);
        return;
    }
    uint32_t old = claim[id];
    for (;;) {
        uint32_t cnt = (old >> 2) == gen ? (old & kCountMask) : 0u;
        uint32_t want = (gen << 2) | (cnt >= 2u ? 2u : cnt + 1u);
        if (want == old) break;
        uint32_t seen = atomicCAS(claim + id, old, want);
        if (seen == old) break;
        old = seen;
    }
}

// after the claim pass: ok[v] = 1 when row v's id is in range and was claimed
// once (a repeated id sets the error word and its rows are not copied).  The
// copy then reads one byte per row in row order instead of a claim word at a
// random place behind the id's load.
__global__ void push_ok_kernel(const int64_t *__restrict__ ids, int64_t n, int64_t n_table,
                               const uint32_t *__restrict__ claim, uint32_t gen, uint8_t *__restrict__ ok, int *err) {
    const int64_t v = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (v >= n) return;
    const int64_t id = ids[v];
    uint8_t good = 0;
    if (id >= 0 && id < n_table) {  // out-of-range ids are reported by the claim pass
        if (claim[id] == ((gen << 2) | 1u)) good = 1;
        else atomicOr(err, 1);  // repeated id: no copy of it is written
    }
    ok[v] = good;
}

template <int LPR>
__global__ void __launch_bounds__(256, 3) push_copy_kernel(const char *__restrict__ H, int64_t row_bytes_h,
                                                        const int64_t *__restrict__ ids, int64_t n,
                                                        const uint8_t *__restrict__ ok, char *__restrict__ table,
                                                        int64_t row_bytes_t, int64_t nbytes, int es) {
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t v0 = (t / LPR) * kRowsPerGroup;
    const int sub = (int)(t % LPR);
    if (v0 >= n) return;
    // The source rows are consecutive: the first vector of each is loaded
    // before the ids and claim words, so those loads are in flight together
    // instead of one after the other; only the stores wait for the ids.
    const int nsrc = n - v0 < kRowsPerGroup ? (int)(n - v0) : kRowsPerGroup;
    const bool lead = sub < nbytes / 16;
    uint4 head[kRowsPerGroup];
#pragma unroll
    for (int k = 0; k < kRowsPerGroup; ++k)
        if (lead && k < nsrc) head[k] = __ldg(reinterpret_cast<const uint4 *>(H + (v0 + k) * row_bytes_h) + sub);
    int64_t ix[kRowsPerGroup];
#pragma unroll
    for (int k = 0; k < kRowsPerGroup; ++k) {
        const int64_t v = v0 + k;
        ix[k] = (v < n && __ldg(ok + v)) ? __ldg(ids + v) : -1;
    }
#pragma unroll
    for (int k = 0; k < kRowsPerGroup; ++k)
        if (lead && ix[k] >= 0) reinterpret_cast<uint4 *>(table + ix[k] * row_bytes_t)[sub] = head[k];
    copy_rows<LPR, false>(H, row_bytes_h, table, row_bytes_t, v0, ix, nbytes, es, sub, sub + LPR);
}

int lanes_per_row(int64_t nbytes) {
    int64_t nvec = ceil_div(nbytes, 16);
    int l = 1;
    while (l < 32 && l < nvec) l <<= 1;
    return l;
}

template <typename F>
gnn_status dispatch_lpr(int lpr, F &&f) {
    switch (lpr) {
        case 1: return f(std::integral_constant<int, 1>());
        case 2: return f(std::integral_constant<int, 2>());
        case 4: return f(std::integral_constant<int, 4>());
        case 8: return f(std::integral_constant<int, 8>());
        case 16: return f(std::integral_constant<int, 16>());
        default: return f(std::integral_constant<int, 32>());
    }
}

}  // namespace

gnn_status launch_pull(const void *table, int64_t ld_t, int64_t n_table, const int64_t *ids, int64_t n_ids, void *H,
                       int64_t ld_h, int64_t row0, int64_t f, int es, int *err, cudaStream_t s) {
    if (n_ids == 0) return GNN_OK;
    const int64_t nbytes = f * es;
    const int lpr = lanes_per_row(nbytes);
    return dispatch_lpr(lpr, [&](auto L) -> gnn_status {
        constexpr int LPR = decltype(L)::value;
        const int64_t blocks = ceil_div(ceil_div(n_ids, kRowsPerGroup) * LPR, 256);
        { pull_kernel<LPR><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const char *>(table), ld_t * es, n_table, ids,
                                                          n_ids, static_cast<char *>(H), ld_h * es, row0, nbytes, es,
                                                          err); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

gnn_status ensure_claim(gnn_graph *g, int64_t n_table) {
    if (g->claim_n >= n_table) return GNN_OK;
    // grow the claim array; ordered after earlier work on the device
    GNN_CUDA_TRY(cudaDeviceSynchronize());
    if (g->claim) GNN_CUDA_TRY(cudaFree(g->claim));
    g->claim = nullptr;
    g->claim_n = 0;
    GNN_CUDA_TRY(cudaMalloc((void **)&g->claim, (size_t)n_table * sizeof(uint32_t)));
    GNN_CUDA_TRY(cudaMemset(g->claim, 0, (size_t)n_table * sizeof(uint32_t)));
    g->claim_n = n_table;
    g->claim_gen = 0;
    return GNN_OK;
}

gnn_status launch_push_claim(gnn_graph *g, const int64_t *ids, int64_t n_rows, int64_t n_table, uint32_t *gen_out,
                             cudaStream_t s) {
    gnn_status st = ensure_claim(g, n_table);
    if (st != GNN_OK) return st;
    g->claim_gen += 1;
    if (g->claim_gen >= (1u << 30)) {
        GNN_CUDA_TRY(cudaMemsetAsync(g->claim, 0, (size_t)g->claim_n * sizeof(uint32_t), s));
        g->claim_gen = 1;
    }
    const uint32_t gen = g->claim_gen;
    { push_claim_kernel<<<(unsigned)ceil_div(n_rows, 256), 256, 0, s>>>(ids, n_rows, n_table, g->claim, gen, g->err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    *gen_out = gen;
    return GNN_OK;
}

gnn_status ensure_push_ok(gnn_graph *g, int64_t n_rows) {
    if (g->push_ok_n >= n_rows) return GNN_OK;
    // grow the per-row flags; ordered after earlier work on the device
    GNN_CUDA_TRY(cudaDeviceSynchronize());
    if (g->push_ok) GNN_CUDA_TRY(cudaFree(g->push_ok));
    g->push_ok = nullptr;
    g->push_ok_n = 0;
    GNN_CUDA_TRY(cudaMalloc((void **)&g->push_ok, (size_t)n_rows));
    g->push_ok_n = n_rows;
    return GNN_OK;
}

gnn_status launch_push_checks(gnn_graph *g, const int64_t *ids, int64_t n_rows, int64_t n_table, cudaStream_t s) {
    uint32_t gen = 0;
    gnn_status st = ensure_push_ok(g, n_rows);
    if (st != GNN_OK) return st;
    st = launch_push_claim(g, ids, n_rows, n_table, &gen, s);
    if (st != GNN_OK) return st;
    { push_ok_kernel<<<(unsigned)ceil_div(n_rows, 256), 256, 0, s>>>(ids, n_rows, n_table, g->claim, gen, g->push_ok,
                                                                     g->err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                       void *table, int64_t ld_t, int64_t n_table, int es, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    gnn_status st = launch_push_checks(g, ids, n_rows, n_table, s);
    if (st != GNN_OK) return st;
    const int64_t nbytes = f * es;
    const int lpr = lanes_per_row(nbytes);
    return dispatch_lpr(lpr, [&](auto L) -> gnn_status {
        constexpr int LPR = decltype(L)::value;
        const int64_t blocks = ceil_div(ceil_div(n_rows, kRowsPerGroup) * LPR, 256);
        { push_copy_kernel<LPR><<<(unsigned)blocks, 256, 0, s>>>(static_cast<const char *>(H), ld_h * es, ids, n_rows,
                                                               g->push_ok, static_cast<char *>(table), ld_t * es,
                                                               nbytes, es); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

}  // namespace gnn
