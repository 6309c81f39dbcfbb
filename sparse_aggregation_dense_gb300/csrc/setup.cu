// setup.cu - graph set-up on the device: CSR validation, degree normalisation,
// the stable CSR transpose (LSD radix sort of column ids) and the heavy-row
// schedules of the aggregation.
//
// The transpose keeps A and A^T apart explicitly, as the CAGNET page ("Reducing
// Communication in Graph Neural Network Training", GNN section) prescribes for a
// training algorithm that works on directed graphs; entries of a transpose row
// are ordered by ascending source row, so every later pass is deterministic.
#include <algorithm>
#include <atomic>
#include <cstdlib>

#include "gnn_internal.cuh"

namespace gnn {

namespace {
std::atomic<int> g_last_cuda_error{0};  // cudaError_t of the last failed runtime call
}

gnn_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return GNN_OK;
    g_last_cuda_error.store((int)e, std::memory_order_relaxed);
    if (e == cudaErrorMemoryAllocation) return GNN_ENOMEM;
    return GNN_ECUDA;
}

const char *last_cuda_error_text() {
    const int e = g_last_cuda_error.load(std::memory_order_relaxed);
    return e ? cudaGetErrorString((cudaError_t)e) : "no error";
}

// ---------------------------------------------------------------------------
// exclusive scan of int32 (three phases: block sums, scan of the sums, block
// scans plus offsets); used only at set-up and by the push claim logic
// ---------------------------------------------------------------------------
constexpr int kScanThreads = 1024;
constexpr int kScanItems = 4;
constexpr int kScanTile = kScanThreads * kScanItems;

__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t *warp_tot, int32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t t = lane < (int)(blockDim.x >> 5) ? warp_tot[lane] : 0;
        int32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_tot[lane] = s - t;  // exclusive prefix of warp totals
        if (lane == 31) *total = s;
    }
    __syncthreads();
    return x - v + warp_tot[warp];
}

__global__ void scan_block_sums(const int32_t *__restrict__ in, int64_t n, int32_t *__restrict__ sums) {
    __shared__ int32_t red[32];
    int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int32_t s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k)
        if (base + k < n) s += in[base + k];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = s;
    __syncthreads();
    if (threadIdx.x < 32) {
        int32_t t = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (threadIdx.x == 0) sums[blockIdx.x] = t;
    }
}

__global__ void scan_block_apply(const int32_t *in, int32_t *out, int64_t n, const int32_t *__restrict__ offsets,
                                 bool write_total) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t total;
    int64_t base = (int64_t)blockIdx.x * kScanTile + (int64_t)threadIdx.x * kScanItems;
    int32_t v[kScanItems];
    int32_t s = 0;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        v[k] = base + k < n ? in[base + k] : 0;
        s += v[k];
    }
    int32_t pre = block_exclusive_scan(s, warp_tot, &total);
    int32_t off = offsets ? offsets[blockIdx.x] : 0;
    int32_t run = off + pre;
#pragma unroll
    for (int k = 0; k < kScanItems; ++k) {
        if (base + k < n) out[base + k] = run;
        run += v[k];
    }
    if (write_total && blockIdx.x == gridDim.x - 1 && threadIdx.x == 0) out[n] = off + total;
}

gnn_status exclusive_scan_i32(const int32_t *in, int32_t *out, int64_t n, bool write_total, cudaStream_t s) {
    if (n <= 0) {
        if (write_total) GNN_CUDA_TRY(cudaMemsetAsync(out, 0, sizeof(int32_t), s));
        return GNN_OK;
    }
    int64_t nb = ceil_div(n, kScanTile);
    int32_t *sums = nullptr;
    if (nb > 1) {
        GNN_CUDA_TRY(cudaMallocAsync((void **)&sums, (size_t)nb * sizeof(int32_t), s));
        { scan_block_sums<<<(unsigned)nb, kScanThreads, 0, s>>>(in, n, sums); GNN_LAUNCHED(1); }
        gnn_status st = exclusive_scan_i32(sums, sums, nb, false, s);
        if (st != GNN_OK) return st;
    }
    { scan_block_apply<<<(unsigned)nb, kScanThreads, 0, s>>>(in, out, n, sums, write_total); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    if (sums) GNN_CUDA_TRY(cudaFreeAsync(sums, s));
    return GNN_OK;
}

// ---------------------------------------------------------------------------
// validation and degrees
// ---------------------------------------------------------------------------
__global__ void validate_csr_kernel(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ colidx,
                                    int64_t n_rows, int64_t n_cols, int64_t nnz, int *err) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int bad = 0;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_rows + 1 || i < nnz; i += stride) {
        if (i <= n_rows) {
            int32_t a = rowptr[i];
            if (i == 0 && a != 0) bad = 1;
            if (i == n_rows && (int64_t)a != nnz) bad = 1;
            if (i < n_rows && rowptr[i + 1] < a) bad = 1;
        }
        if (i < nnz) {
            int32_t c = colidx[i];
            if (c < 0 || (int64_t)c >= n_cols) bad = 1;
        }
    }
    if (bad) atomicOr(err, 1);
}

gnn_status launch_validate_csr(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, int64_t n_cols,
                               int64_t nnz, int *err, cudaStream_t s) {
    int64_t work = (n_rows + 1 > nnz ? n_rows + 1 : nnz);
    int64_t blocks = ceil_div(work, 256);
    if (blocks > 152 * 32) blocks = 152 * 32;
    { validate_csr_kernel<<<(unsigned)blocks, 256, 0, s>>>(rowptr, colidx, n_rows, n_cols, nnz, err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

__global__ void init_degree_counts(const int32_t *__restrict__ rowptr, int64_t n_local, int64_t n_total,
                                   int32_t *cnt) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n_total) return;
    cnt[x] = x < n_local ? rowptr[x + 1] - rowptr[x] : 1;
}

__global__ void count_halo_columns(const int32_t *__restrict__ colidx, int64_t nnz, int64_t n_local, int32_t *cnt) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) {
        int32_t c = colidx[e];
        if (c >= n_local) atomicAdd(&cnt[c], 1);
    }
}

__global__ void dinv_from_counts(const int32_t *__restrict__ cnt, int64_t n, float *dinv) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n) return;
    float d = (float)cnt[x];
    dinv[x] = d > 0.0f ? 1.0f / sqrtf(d) : 0.0f;
}

__global__ void dinv_from_deg(const float *__restrict__ deg, int64_t n, float *dinv) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n) return;
    float d = deg[x];
    dinv[x] = d > 0.0f ? 1.0f / sqrtf(d) : 0.0f;
}

gnn_status launch_gcn_dinv(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, int64_t n_halo,
                           int64_t nnz, const float *deg, float *dinv, cudaStream_t s) {
    int64_t nT = n_local + n_halo;
    if (nT == 0) return GNN_OK;
    unsigned b = (unsigned)ceil_div(nT, 256);
    if (deg) {
        { dinv_from_deg<<<b, 256, 0, s>>>(deg, nT, dinv); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    }
    int32_t *cnt = nullptr;
    GNN_CUDA_TRY(cudaMallocAsync((void **)&cnt, (size_t)nT * sizeof(int32_t), s));
    { init_degree_counts<<<b, 256, 0, s>>>(rowptr, n_local, nT, cnt); GNN_LAUNCHED(1); }
    if (nnz > 0) { count_halo_columns<<<152 * 16, 256, 0, s>>>(colidx, nnz, n_local, cnt); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    { dinv_from_counts<<<b, 256, 0, s>>>(cnt, nT, dinv); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    GNN_CUDA_TRY(cudaFreeAsync(cnt, s));
    return GNN_OK;
}

__global__ void sage_invcnt_kernel(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ colidx,
                                   int64_t n_local, float *out) {
    int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (v >= n_local) return;
    int32_t c = 0;
    for (int64_t e = rowptr[v] + lane; e < rowptr[v + 1]; e += 32) c += colidx[e] != v;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) out[v] = c > 0 ? 1.0f / (float)c : 0.0f;
}

gnn_status launch_sage_invcnt(const int32_t *rowptr, const int32_t *colidx, int64_t n_local, float *out,
                              cudaStream_t s) {
    if (n_local == 0) return GNN_OK;
    { sage_invcnt_kernel<<<(unsigned)ceil_div(n_local * 32, 256), 256, 0, s>>>(rowptr, colidx, n_local, out); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

__global__ void entry_weights_kernel(const int32_t *__restrict__ rowptr, const int32_t *__restrict__ colidx,
                                     int64_t n_rows, const float *__restrict__ colw, int skip_self,
                                     float *__restrict__ w) {
    const int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (r >= n_rows) return;
    for (int64_t e = rowptr[r] + lane; e < rowptr[r + 1]; e += 32) {
        const int32_t c = colidx[e];
        float v = colw ? colw[c] : 1.0f;
        if (skip_self && (int64_t)c == r) v = 0.0f;
        w[e] = v;
    }
}

// the sign bit of the weight of every row's last entry marks the row's end
__global__ void mark_row_ends_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, float *__restrict__ w) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_rows) return;
    const int32_t e = rowptr[r + 1];
    if (e > rowptr[r]) w[e - 1] = __uint_as_float(__float_as_uint(w[e - 1]) | 0x80000000u);
}

gnn_status launch_mark_row_ends(const int32_t *rowptr, int64_t n_rows, float *w, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    { mark_row_ends_kernel<<<(unsigned)ceil_div(n_rows, 256), 256, 0, s>>>(rowptr, n_rows, w); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_entry_weights(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, const float *colw,
                                bool skip_self, float *w, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    { entry_weights_kernel<<<(unsigned)ceil_div(n_rows * 32, 256), 256, 0, s>>>(rowptr, colidx, n_rows, colw,
                                                                               skip_self ? 1 : 0, w); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

// ---------------------------------------------------------------------------
// stable transpose: row ids of every entry, LSD radix sort of the column ids
// (8-bit digits, 4096-entry tiles, warp ranks by match_any), then counts
// ---------------------------------------------------------------------------
constexpr int kRsThreads = 256;
constexpr int kRsWarps = kRsThreads / 32;
constexpr int kRsRounds = 16;
constexpr int kRsTile = kRsThreads * kRsRounds;  // 4096 entries

__global__ void expand_rows_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, int32_t *__restrict__ row_of) {
    int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    int lane = threadIdx.x & 31;
    if (r >= n_rows) return;
    for (int64_t e = rowptr[r] + lane; e < rowptr[r + 1]; e += 32) row_of[e] = (int32_t)r;
}

template <bool kScatter>
__global__ void __launch_bounds__(kRsThreads) radix_pass_kernel(const uint32_t *__restrict__ keys_in,
                                                                const int32_t *__restrict__ vals_in,
                                                                uint32_t *__restrict__ keys_out,
                                                                int32_t *__restrict__ vals_out, int64_t n, int shift,
                                                                int32_t *__restrict__ hist, int64_t n_tiles) {
    __shared__ int32_t wcount[kRsWarps][257];
    __shared__ int32_t wofs[kRsWarps][256];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int i = threadIdx.x; i < kRsWarps * 257; i += kRsThreads) (&wcount[0][0])[i] = 0;
    __syncthreads();
    const int64_t base = (int64_t)blockIdx.x * kRsTile + (int64_t)warp * (kRsTile / kRsWarps);
    uint32_t key[kRsRounds];
    int32_t pos[kRsRounds];
    uint32_t dig[kRsRounds];
#pragma unroll
    for (int j = 0; j < kRsRounds; ++j) {
        int64_t i = base + j * 32 + lane;
        key[j] = i < n ? keys_in[i] : 0u;
        uint32_t d = i < n ? (key[j] >> shift) & 255u : 256u;
        dig[j] = d;
        unsigned peers = __match_any_sync(0xffffffffu, d);
        int rank = __popc(peers & ((1u << lane) - 1u));
        int before = wcount[warp][d];
        pos[j] = before + rank;
        __syncwarp();
        if (lane == __ffs(peers) - 1) wcount[warp][d] = before + __popc(peers);
        __syncwarp();
    }
    __syncthreads();
    if (!kScatter) {
        int d = threadIdx.x;  // 256 threads = 256 digits
        int32_t sum = 0;
#pragma unroll
        for (int w = 0; w < kRsWarps; ++w) sum += wcount[w][d];
        hist[(int64_t)d * n_tiles + blockIdx.x] = sum;
        return;
    }
    {
        int d = threadIdx.x;
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < kRsWarps; ++w) {
            wofs[w][d] = run;
            run += wcount[w][d];
        }
    }
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kRsRounds; ++j) {
        int64_t i = base + j * 32 + lane;
        if (i < n) {
            uint32_t d = dig[j];
            int64_t dst = (int64_t)hist[(int64_t)d * n_tiles + blockIdx.x] + wofs[warp][d] + pos[j];
            keys_out[dst] = key[j];
            vals_out[dst] = vals_in ? vals_in[i] : (int32_t)i;
        }
    }
}

__global__ void count_columns_kernel(const int32_t *__restrict__ colidx, int64_t nnz, int32_t *cnt) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) atomicAdd(&cnt[colidx[e]], 1);
}

__global__ void gather_rows_kernel(const int32_t *__restrict__ perm, const int32_t *__restrict__ row_of, int64_t nnz,
                                   int32_t *__restrict__ colidxT) {
    int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < nnz; k += stride) colidxT[k] = row_of[perm[k]];
}

gnn_status csr_transpose(const int32_t *rowptr, const int32_t *colidx, int64_t n_rows, int64_t n_cols, int64_t nnz,
                         int32_t *rowptrT, int32_t *colidxT, int32_t *permT, cudaStream_t s) {
    // row pointers of the transpose: column counts, then an exclusive scan
    GNN_CUDA_TRY(cudaMemsetAsync(rowptrT, 0, (size_t)(n_cols + 1) * sizeof(int32_t), s));
    if (nnz == 0) return GNN_OK;
    { count_columns_kernel<<<152 * 16, 256, 0, s>>>(colidx, nnz, rowptrT); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    gnn_status st = exclusive_scan_i32(rowptrT, rowptrT, n_cols, true, s);
    if (st != GNN_OK) return st;

    int32_t *row_of = nullptr, *vals_b = nullptr, *hist = nullptr;
    uint32_t *keys_a = nullptr, *keys_b = nullptr;
    int64_t n_tiles = ceil_div(nnz, kRsTile);
    GNN_CUDA_TRY(cudaMallocAsync((void **)&row_of, (size_t)nnz * sizeof(int32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&keys_a, (size_t)nnz * sizeof(uint32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&keys_b, (size_t)nnz * sizeof(uint32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&vals_b, (size_t)nnz * sizeof(int32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&hist, (size_t)(256 * n_tiles) * sizeof(int32_t), s));
    if (n_rows > 0) {
        { expand_rows_kernel<<<(unsigned)ceil_div(n_rows * 32, 256), 256, 0, s>>>(rowptr, n_rows, row_of); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    int bits = 0;
    while (bits < 31 && ((int64_t)1 << bits) < n_cols) ++bits;
    int passes = bits <= 8 ? 1 : (bits + 7) / 8;
    // pass p reads (keys, vals) from src and writes to dst; the result must end
    // in (keys_x, permT), so choose the first destination by the pass parity
    const uint32_t *ksrc = reinterpret_cast<const uint32_t *>(colidx);
    const int32_t *vsrc = nullptr;
    for (int p = 0; p < passes; ++p) {
        bool last_to_perm = ((passes - 1 - p) % 2) == 0;
        uint32_t *kdst = last_to_perm ? keys_a : keys_b;
        int32_t *vdst = last_to_perm ? permT : vals_b;
        int shift = 8 * p;
        { radix_pass_kernel<false><<<(unsigned)n_tiles, kRsThreads, 0, s>>>(ksrc, vsrc, nullptr, nullptr, nnz, shift,
                                                                          hist, n_tiles); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        st = exclusive_scan_i32(hist, hist, 256 * n_tiles, false, s);
        if (st != GNN_OK) return st;
        { radix_pass_kernel<true><<<(unsigned)n_tiles, kRsThreads, 0, s>>>(ksrc, vsrc, kdst, vdst, nnz, shift, hist,
                                                                         n_tiles); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        ksrc = kdst;
        vsrc = vdst;
    }
    { gather_rows_kernel<<<152 * 16, 256, 0, s>>>(permT, row_of, nnz, colidxT); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    GNN_CUDA_TRY(cudaFreeAsync(row_of, s));
    GNN_CUDA_TRY(cudaFreeAsync(keys_a, s));
    GNN_CUDA_TRY(cudaFreeAsync(keys_b, s));
    GNN_CUDA_TRY(cudaFreeAsync(vals_b, s));
    GNN_CUDA_TRY(cudaFreeAsync(hist, s));
    return GNN_OK;
}

// ---------------------------------------------------------------------------
// heavy-row schedule
// ---------------------------------------------------------------------------
// Rows the fix-up writes: heavy rows (their chunk partials summed) and empty
// rows (no chunk: the fix-up writes their zero / self term).  Row groups hold
// the other rows, each with at least one entry, so the end of every row of a
// group is marked on an entry.
__device__ __forceinline__ bool fixup_row(int32_t d) { return d > kHeavyNnz || d == 0; }

__global__ void sched_count_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, int32_t *nch, int32_t *flag) {
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_rows) return;
    int32_t d = rowptr[r + 1] - rowptr[r];
    int32_t c = d > kHeavyNnz ? (d + kChunkNnz - 1) / kChunkNnz : 0;
    nch[r] = c;
    flag[r] = fixup_row(d);
}

__global__ void sched_fill_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, const int32_t *__restrict__ choff,
                                  const int32_t *__restrict__ hidx, int32_t *heavy_rows, int32_t *heavy_choff,
                                  int32_t *chunk_row, int32_t *chunk_begin, int32_t *chunk_end) {
    int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_rows) return;
    int32_t c0 = choff[r], c1 = choff[r + 1];
    if (hidx[r + 1] == hidx[r]) return;  // not a fix-up row
    int32_t h = hidx[r];
    heavy_rows[h] = (int32_t)r;
    heavy_choff[h] = c0;
    int32_t b = rowptr[r], e = rowptr[r + 1];
    for (int32_t c = c0; c < c1; ++c) {
        int32_t lo = b + (c - c0) * kChunkNnz;
        int32_t hi = lo + kChunkNnz < e ? lo + kChunkNnz : e;
        chunk_row[c] = (int32_t)r;
        chunk_begin[c] = lo;
        chunk_end[c] = hi;
    }
}

// row r (light) starts a group when it is the first row, follows a fix-up row
// (heavy or empty), starts in another kGroupNnz-entry window than row r - 1,
// or is a multiple of kGroupRows
__device__ __forceinline__ bool is_heavy_row(const int32_t *__restrict__ rowptr, int64_t r) {
    return fixup_row(rowptr[r + 1] - rowptr[r]);
}
__global__ void group_flag_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, int32_t *flag) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_rows) return;
    int32_t f = 0;
    if (!is_heavy_row(rowptr, r))
        f = r == 0 || is_heavy_row(rowptr, r - 1) || rowptr[r] / kGroupNnz != rowptr[r - 1] / kGroupNnz ||
            r % kGroupRows == 0;
    flag[r] = f;
}
// flag: exclusive scan of the start flags (start flags recomputed here)
__global__ void group_fill_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, const int32_t *__restrict__ gidx,
                                  int32_t *group_r0, int32_t *group_r1) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= n_rows || is_heavy_row(rowptr, r)) return;
    const bool start = gidx[r + 1] != gidx[r];
    const int32_t g = start ? gidx[r] : gidx[r] - 1;  // the group row r belongs to
    if (start) group_r0[g] = (int32_t)r;
    const bool last = r + 1 == n_rows || is_heavy_row(rowptr, r + 1) || gidx[r + 2] != gidx[r + 1];
    if (last) group_r1[g] = (int32_t)(r + 1);
}

void free_schedule(Schedule *sc) {
    cudaFree(sc->group_r0);
    cudaFree(sc->group_r1);
    cudaFree(sc->heavy_rows);
    cudaFree(sc->heavy_choff);
    cudaFree(sc->chunk_row);
    cudaFree(sc->chunk_begin);
    cudaFree(sc->chunk_end);
    *sc = Schedule();
}

gnn_status build_schedule(const int32_t *rowptr, int64_t n_rows, Schedule *sc, cudaStream_t s) {
    *sc = Schedule();
    sc->n_rows = n_rows;
    if (n_rows == 0) return GNN_OK;
    int32_t *nch = nullptr, *flag = nullptr;
    GNN_CUDA_TRY(cudaMallocAsync((void **)&nch, (size_t)(n_rows + 1) * sizeof(int32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&flag, (size_t)(n_rows + 1) * sizeof(int32_t), s));
    unsigned b = (unsigned)ceil_div(n_rows, 256);
    { sched_count_kernel<<<b, 256, 0, s>>>(rowptr, n_rows, nch, flag); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    gnn_status st = exclusive_scan_i32(nch, nch, n_rows, true, s);
    if (st != GNN_OK) return st;
    st = exclusive_scan_i32(flag, flag, n_rows, true, s);
    if (st != GNN_OK) return st;
    int32_t tot[2];
    GNN_CUDA_TRY(cudaMemcpyAsync(&tot[0], nch + n_rows, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_CUDA_TRY(cudaMemcpyAsync(&tot[1], flag + n_rows, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_CUDA_TRY(cudaStreamSynchronize(s));
    sc->n_chunks = tot[0];
    sc->n_heavy = tot[1];
    if (sc->n_heavy > 0) {
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->heavy_rows, (size_t)sc->n_heavy * sizeof(int32_t)));
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->heavy_choff, (size_t)(sc->n_heavy + 1) * sizeof(int32_t)));
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->chunk_row, (size_t)sc->n_chunks * sizeof(int32_t)));
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->chunk_begin, (size_t)sc->n_chunks * sizeof(int32_t)));
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->chunk_end, (size_t)sc->n_chunks * sizeof(int32_t)));
        { sched_fill_kernel<<<b, 256, 0, s>>>(rowptr, n_rows, nch, flag, sc->heavy_rows, sc->heavy_choff, sc->chunk_row,
                                            sc->chunk_begin, sc->chunk_end); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        int32_t nc = (int32_t)sc->n_chunks;
        GNN_CUDA_TRY(cudaMemcpyAsync(sc->heavy_choff + sc->n_heavy, &nc, sizeof(int32_t), cudaMemcpyHostToDevice, s));
        GNN_CUDA_TRY(cudaStreamSynchronize(s));
    }
    // row groups of the light rows (flag reused: start flags, then their exclusive scan)
    { group_flag_kernel<<<b, 256, 0, s>>>(rowptr, n_rows, flag); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    st = exclusive_scan_i32(flag, flag, n_rows, true, s);
    if (st != GNN_OK) return st;
    int32_t ng = 0;
    GNN_CUDA_TRY(cudaMemcpyAsync(&ng, flag + n_rows, sizeof(int32_t), cudaMemcpyDeviceToHost, s));
    GNN_CUDA_TRY(cudaStreamSynchronize(s));
    sc->n_groups = ng;
    if (ng > 0) {
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->group_r0, (size_t)ng * sizeof(int32_t)));
        GNN_CUDA_TRY(cudaMalloc((void **)&sc->group_r1, (size_t)ng * sizeof(int32_t)));
        { group_fill_kernel<<<b, 256, 0, s>>>(rowptr, n_rows, flag, sc->group_r0, sc->group_r1); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    GNN_CUDA_TRY(cudaFreeAsync(nch, s));
    GNN_CUDA_TRY(cudaFreeAsync(flag, s));
    return GNN_OK;
}

// ---------------------------------------------------------------------------
// hotness tiers (L2 residency hints of the aggregation)
// ---------------------------------------------------------------------------
__device__ __forceinline__ int count_bin(int32_t c) {
    // 8 bins per octave: 1 + 8 * floor(log2 c) + the 3 bits below the leading one
    if (c <= 0) return 0;
    const int lz = 31 - __clz(c);
    const int sub = lz >= 3 ? (c >> (lz - 3)) & 7 : (c << (3 - lz)) & 7;
    return 1 + 8 * lz + sub;
}

__global__ void count_bins_kernel(const int32_t *__restrict__ ptr, int64_t n, int32_t *hist) {
    __shared__ int32_t h[256];
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0;
    __syncthreads();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += stride)
        atomicAdd(&h[count_bin(ptr[x + 1] - ptr[x])], 1);
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&hist[i], h[i]);
}

__global__ void tag_tiers_kernel(int32_t *__restrict__ colidx, int64_t nnz, const int32_t *__restrict__ ptr,
                                 const uint8_t *__restrict__ tier_of_bin) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < nnz; e += stride) {
        const int32_t c = colidx[e];
        const uint32_t t = tier_of_bin[count_bin(ptr[c + 1] - ptr[c])];
        colidx[e] = (int32_t)((uint32_t)c | (t << kTierShift));
    }
}

__global__ void untag_kernel(const int32_t *__restrict__ src, int32_t *__restrict__ dst, int64_t n, uint32_t mask) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride)
        dst[i] = (int32_t)((uint32_t)src[i] & mask);
}

gnn_status copy_untagged(const int32_t *src, int32_t *dst, int64_t n, uint32_t mask, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    { untag_kernel<<<152 * 8, 256, 0, s>>>(src, dst, n, mask); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status tag_tiers(int32_t *colidx, int64_t nnz, const int32_t *ptr, int64_t n_cols, Schedule *sc, cudaStream_t s) {
    sc->tagged = false;
    for (int t = 0; t < kTiers; ++t) sc->tier_rows[t] = 0;
    if (n_cols >= ((int64_t)1 << kTierShift) || n_cols == 0 || nnz == 0) return GNN_OK;
    int32_t *hist = nullptr;
    uint8_t *tob = nullptr;
    GNN_CUDA_TRY(cudaMallocAsync((void **)&hist, 256 * sizeof(int32_t), s));
    GNN_CUDA_TRY(cudaMallocAsync((void **)&tob, 256, s));
    GNN_CUDA_TRY(cudaMemsetAsync(hist, 0, 256 * sizeof(int32_t), s));
    { count_bins_kernel<<<152 * 4, 256, 0, s>>>(ptr, n_cols, hist); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    int32_t h[256];
    GNN_CUDA_TRY(cudaMemcpyAsync(h, hist, sizeof(h), cudaMemcpyDeviceToHost, s));
    GNN_CUDA_TRY(cudaStreamSynchronize(s));
    // walk bins from the most accessed down; a bin's tier is the first whose rank
    // bound covers every column up to and including the bin
    uint8_t t_of[256];
    int64_t cum = 0;
    int t = 0;
    for (int b = 255; b >= 0; --b) {
        cum += h[b];
        while (t < kTiers - 1 && (double)cum > 1024.0 * exp2(0.5 * t)) ++t;
        t_of[b] = (uint8_t)t;
        sc->tier_rows[t] += h[b];
    }
    GNN_CUDA_TRY(cudaMemcpyAsync(tob, t_of, sizeof(t_of), cudaMemcpyHostToDevice, s));
    { tag_tiers_kernel<<<152 * 16, 256, 0, s>>>(colidx, nnz, ptr, tob); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    GNN_CUDA_TRY(cudaFreeAsync(hist, s));
    GNN_CUDA_TRY(cudaFreeAsync(tob, s));
    GNN_CUDA_TRY(cudaStreamSynchronize(s));
    sc->tagged = true;
    return GNN_OK;
}

// Stable counting sort of every row's entries by tier, hottest first, the
// weights moved with their entries.  With a row's hot entries next to each
// other, the four rows of one gather mostly share a tier and so an L2 policy
// (a gather takes one policy for its four rows).  One warp per row: a pass
// counts the tiers, a scan over the 32 tiers gives each its first slot, a
// second pass scatters (ranks inside a 32-entry window by match_any).
__global__ void __launch_bounds__(256) tier_sort_rows_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows,
                                                             const uint32_t *__restrict__ col_in,
                                                             const float *__restrict__ w_in,
                                                             uint32_t *__restrict__ col_out,
                                                             float *__restrict__ w_out) {
    __shared__ int32_t slot[8][kTiers];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int64_t nw = (int64_t)gridDim.x * 8;
    for (int64_t r = (int64_t)blockIdx.x * 8 + wib; r < n_rows; r += nw) {
        const int32_t b = rowptr[r], e = rowptr[r + 1];
        slot[wib][lane] = 0;
        __syncwarp();
        for (int32_t i = b; i < e; i += 32) {
            const bool in = i + lane < e;
            const uint32_t t = in ? col_in[i + lane] >> kTierShift : 0u;
            const unsigned peers = __match_any_sync(0xffffffffu, in ? t : (uint32_t)kTiers);
            if (in && lane == __ffs(peers) - 1) slot[wib][t] += __popc(peers);
            __syncwarp();
        }
        // exclusive scan of the counts: lane t gets the first slot of tier t
        const int32_t c = slot[wib][lane];
        int32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        __syncwarp();
        slot[wib][lane] = b + incl - c;
        __syncwarp();
        for (int32_t i = b; i < e; i += 32) {
            const bool in = i + lane < e;
            const uint32_t col = in ? col_in[i + lane] : 0u;
            const uint32_t t = col >> kTierShift;
            const unsigned peers = __match_any_sync(0xffffffffu, in ? t : (uint32_t)kTiers);
            if (in) {
                const int32_t dst = slot[wib][t] + __popc(peers & ((1u << lane) - 1u));
                col_out[dst] = col;
                w_out[dst] = w_in[i + lane];
            }
            __syncwarp();
            if (in && lane == __ffs(peers) - 1) slot[wib][t] += __popc(peers);
            __syncwarp();
        }
    }
}

gnn_status sort_rows_by_tier(const int32_t *rowptr, int64_t n_rows, const int32_t *col_in, const float *w_in,
                             int32_t *col_out, float *w_out, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n_rows, 8), (int64_t)num_sms() * 32);
    { tier_sort_rows_kernel<<<blocks, 256, 0, s>>>(rowptr, n_rows, reinterpret_cast<const uint32_t *>(col_in), w_in,
                                                    reinterpret_cast<uint32_t *>(col_out), w_out); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

int hot_tier_for(const Schedule &sc, int64_t row_bytes) {
    if (!sc.tagged) return kTiers;  // no tiers: every entry takes the keep policy
    static int64_t budget = 0;
    if (!budget) {
        int dev = 0, l2 = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev);
        // share of L2 given to rows gathered with evict_last: 0.55 by default,
        // GNN_L2_KEEP_SHARE (0 .. 1) overrides it for tuning
        double share = 0.55;
        if (const char *e = getenv("GNN_L2_KEEP_SHARE")) {
            const double v = atof(e);
            if (v >= 0.0 && v <= 1.0) share = v;
        }
        budget = (int64_t)((l2 > 0 ? l2 : 64 << 20) * share);
    }
    int64_t rows = 0;
    int hot = -1;
    for (int t = 0; t < kTiers; ++t) {
        rows += sc.tier_rows[t];
        if (rows * row_bytes > budget) break;
        hot = t;
    }
    return hot;
}

}  // namespace gnn
