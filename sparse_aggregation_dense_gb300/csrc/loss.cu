// loss.cu - training-harness helper (not a layer step): mean softmax
// cross-entropy over the local rows and its gradient with respect to the
// logits, G = (softmax - onehot) / n.  One warp per row; the mean is summed in
// a fixed order (fixed chunks, then the chunk sums in order), so the loss is
// reproducible bit for bit.
#include "gnn_internal.cuh"

namespace gnn {

namespace {

__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T, typename TG>
__global__ void softmax_ce_rows(const T *__restrict__ X, int64_t ld, int64_t n, int64_t C,
                                const int32_t *__restrict__ labels, TG *__restrict__ G, int64_t ld_g,
                                float *__restrict__ row_loss, float inv_n) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= n) return;
    const T *x = X + i * ld;
    float mx = -INFINITY;
    for (int64_t c = lane; c < C; c += 32) mx = fmaxf(mx, ld_elem(x + c));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float se = 0.f;
    for (int64_t c = lane; c < C; c += 32) se += expf(ld_elem(x + c) - mx);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
    const float lse = mx + logf(se);
    const int32_t y = labels[i];
    const bool ok = y >= 0 && y < C;
    for (int64_t c = lane; c < C; c += 32) {
        float p = expf(ld_elem(x + c) - lse);
        st_elem(G + i * ld_g + c, (p - (c == y ? 1.f : 0.f)) * inv_n);
    }
    if (lane == 0) row_loss[i] = ok ? lse - ld_elem(x + y) : NAN;
}

__device__ __forceinline__ void unpack_vec(const uint4 &q, float (&o)[4]) {
    o[0] = __uint_as_float(q.x);
    o[1] = __uint_as_float(q.y);
    o[2] = __uint_as_float(q.z);
    o[3] = __uint_as_float(q.w);
}
__device__ __forceinline__ void unpack_vec(const uint4 &q, float (&o)[8]) {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        o[2 * k] = __uint_as_float(w[k] << 16);
        o[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}
__device__ __forceinline__ uint4 pack_vec(const float (&v)[4]) {
    return make_uint4(__float_as_uint(v[0]), __float_as_uint(v[1]), __float_as_uint(v[2]), __float_as_uint(v[3]));
}
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half (first element)
    return *reinterpret_cast<uint32_t *>(&h);
}
__device__ __forceinline__ uint4 pack_vec(const float (&v)[8]) {
    return make_uint4(pack_bf2(v[0], v[1]), pack_bf2(v[2], v[3]), pack_bf2(v[4], v[5]), pack_bf2(v[6], v[7]));
}

// the EPV gradient values of one logits vector, stored as TG with streaming
// stores (16 bytes each; 8 bytes for four bf16 values)
template <int EPV>
__device__ __forceinline__ void store_vals(float *dst, const float (&o)[EPV]) {
#pragma unroll
    for (int k = 0; k < EPV; k += 4)
        __stcs(reinterpret_cast<uint4 *>(dst + k),
               make_uint4(__float_as_uint(o[k]), __float_as_uint(o[k + 1]), __float_as_uint(o[k + 2]),
                          __float_as_uint(o[k + 3])));
}
template <int EPV>
__device__ __forceinline__ void store_vals(__nv_bfloat16 *dst, const float (&o)[EPV]) {
    if constexpr (EPV == 8) {
        __stcs(reinterpret_cast<uint4 *>(dst), pack_vec(o));
    } else {
        __stcs(reinterpret_cast<uint2 *>(dst), make_uint2(pack_bf2(o[0], o[1]), pack_bf2(o[2], o[3])));
    }
}

// Rows of up to 32 * VPL 16-byte vectors of classes, rows 16-byte aligned:
// a warp takes RPW consecutive rows and loads all of them first (lane q holds
// vectors q, q + 32, ... of each row), so RPW rows' loads are in flight at
// once; then each row is reduced from registers and its gradient written back
// with 16-byte stores (element stores only for the vector that straddles C,
// so G's padding is left alone).
template <typename T, typename TG, int VPL, int RPW>
__global__ void __launch_bounds__(256) softmax_ce_rows_vec(const T *__restrict__ X, int64_t ld, int64_t n, int64_t C64,
                                                           const int32_t *__restrict__ labels, TG *__restrict__ G,
                                                           int64_t ld_g, float *__restrict__ row_loss, float inv_n) {
    constexpr int EPV = 16 / (int)sizeof(T);
    const int64_t i0 = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * RPW;
    const int lane = threadIdx.x & 31;
    if (i0 >= n) return;
    const int C = (int)C64;  // at most 32 * VPL * EPV classes
    float v[RPW][VPL][EPV];
    int32_t yl[RPW];
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t i = i0 + r;
        yl[r] = i < n ? labels[i] : -1;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int c0 = (lane + 32 * q) * EPV;
            if (i < n && c0 < C) {
                unpack_vec(__ldcs(reinterpret_cast<const uint4 *>(X + i * ld + c0)), v[r][q]);
            } else {
#pragma unroll
                for (int k = 0; k < EPV; ++k) v[r][q][k] = -INFINITY;
            }
        }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r) {
        const int64_t i = i0 + r;
        if (i >= n) break;
        float mx = -INFINITY;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int left = C - (lane + 32 * q) * EPV;  // classes of this vector inside the row
#pragma unroll
            for (int k = 0; k < EPV; ++k) {
                if (k >= left) v[r][q][k] = -INFINITY;
                mx = fmaxf(mx, v[r][q][k]);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float se = 0.f, xy = 0.f;
        const int32_t y = yl[r];
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int yk = y - (lane + 32 * q) * EPV;  // the label's slot in this vector, if any
#pragma unroll
            for (int k = 0; k < EPV; ++k) {
                if (k == yk) xy = v[r][q][k];
                v[r][q][k] = __expf(v[r][q][k] - mx);  // exp(-inf) = 0 past the row's end
                se += v[r][q][k];
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            se += __shfl_xor_sync(0xffffffffu, se, o);
            xy += __shfl_xor_sync(0xffffffffu, xy, o);
        }
        const float inv_se = 1.0f / se;
        TG *gr = G + i * ld_g;
#pragma unroll
        for (int q = 0; q < VPL; ++q) {
            const int c0 = (lane + 32 * q) * EPV;
            if (c0 >= C) continue;
            const int yk = y - c0;
            float o[EPV];
#pragma unroll
            for (int k = 0; k < EPV; ++k) o[k] = (v[r][q][k] * inv_se - (k == yk ? 1.f : 0.f)) * inv_n;
            if (c0 + EPV <= C) {
                store_vals<EPV>(gr + c0, o);
            } else {
                for (int k = 0; k < EPV && c0 + k < C; ++k) st_elem(gr + c0 + k, o[k]);
            }
        }
        if (lane == 0) row_loss[i] = (y >= 0 && y < C) ? mx + logf(se) - xy : NAN;
    }
}

// Deterministic mean of row_loss in two passes: block b sums the fixed chunk
// [b * kLossChunk, (b + 1) * kLossChunk) in a fixed order and stores the sum
// over the chunk's first element; one block then sums the chunk sums in order.
constexpr int kLossThreads = 1024;
constexpr int64_t kLossChunk = 8 * kLossThreads;

__device__ __forceinline__ float block_sum_fixed(float s, float *part) {
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = kLossThreads / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    return part[0];
}

__global__ void __launch_bounds__(kLossThreads) loss_chunk_sums(float *__restrict__ v, int64_t n) {
    __shared__ float part[kLossThreads];
    const int64_t b0 = (int64_t)blockIdx.x * kLossChunk;
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < (int)(kLossChunk / kLossThreads); ++k) {
        const int64_t i = b0 + (int64_t)k * kLossThreads + threadIdx.x;
        if (i < n) s += v[i];
    }
    const float tot = block_sum_fixed(s, part);
    if (threadIdx.x == 0) v[b0] = tot;  // every read of the chunk is done (barriers above)
}

__global__ void __launch_bounds__(kLossThreads) loss_mean_of_chunks(const float *__restrict__ v, int64_t n_mean,
                                                                     int64_t n_chunks, float *out) {
    __shared__ float part[kLossThreads];
    float s = 0.f;
    for (int64_t c = threadIdx.x; c < n_chunks; c += kLossThreads) s += v[c * kLossChunk];
    const float tot = block_sum_fixed(s, part);
    if (threadIdx.x == 0) *out = n_mean > 0 ? tot / (float)n_mean : 0.f;
}

}  // namespace

constexpr int kRowsPerWarp = 4;

namespace {

template <typename T, typename TG>
gnn_status softmax_rows_typed(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                              int64_t ld_g, float *row_loss, float inv_n, cudaStream_t s) {
    constexpr int epv = 16 / (int)sizeof(T);                // logits per 16-byte vector
    constexpr int gbytes = epv * (int)sizeof(TG);            // bytes of their gradient
    const T *X = static_cast<const T *>(logits);
    TG *Gt = static_cast<TG *>(G);
    const bool aligned = (reinterpret_cast<uintptr_t>(logits) & 15u) == 0 &&
                         (reinterpret_cast<uintptr_t>(G) % (gbytes < 16 ? gbytes : 16)) == 0 && ld % epv == 0 &&
                         (ld_g * (int64_t)sizeof(TG)) % 16 == 0;
    const unsigned blocks = (unsigned)ceil_div(n * 32, 256);
    const unsigned vblocks = (unsigned)ceil_div(ceil_div(n, kRowsPerWarp) * 32, 256);
    if (aligned && C <= 32 * epv) {
        { softmax_ce_rows_vec<T, TG, 1, kRowsPerWarp><<<vblocks, 256, 0, s>>>(X, ld, n, C, labels, Gt, ld_g,
                                                                             row_loss, inv_n); GNN_LAUNCHED(1); }
    } else if (aligned && C <= 64 * epv) {
        { softmax_ce_rows_vec<T, TG, 2, kRowsPerWarp><<<vblocks, 256, 0, s>>>(X, ld, n, C, labels, Gt, ld_g,
                                                                             row_loss, inv_n); GNN_LAUNCHED(1); }
    } else {
        { softmax_ce_rows<T, TG><<<blocks, 256, 0, s>>>(X, ld, n, C, labels, Gt, ld_g, row_loss, inv_n); GNN_LAUNCHED(1); }
    }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace

gnn_status launch_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                             int64_t ld_g, float *row_loss, float *loss, int64_t n_mean, gnn_dtype dt, gnn_dtype gdt,
                             cudaStream_t s) {
    const float inv_n = n_mean > 0 ? 1.0f / (float)n_mean : 0.f;
    if (n > 0) {
        gnn_status st;
        if (dt == GNN_BF16 && gdt == GNN_BF16)
            st = softmax_rows_typed<__nv_bfloat16, __nv_bfloat16>(logits, ld, n, C, labels, G, ld_g, row_loss, inv_n, s);
        else if (dt == GNN_BF16)
            st = softmax_rows_typed<__nv_bfloat16, float>(logits, ld, n, C, labels, G, ld_g, row_loss, inv_n, s);
        else if (gdt == GNN_BF16)
            st = softmax_rows_typed<float, __nv_bfloat16>(logits, ld, n, C, labels, G, ld_g, row_loss, inv_n, s);
        else
            st = softmax_rows_typed<float, float>(logits, ld, n, C, labels, G, ld_g, row_loss, inv_n, s);
        if (st != GNN_OK) return st;
    }
    const int64_t n_chunks = ceil_div(n, kLossChunk);
    if (n_chunks > 0) {
        { loss_chunk_sums<<<(unsigned)n_chunks, kLossThreads, 0, s>>>(row_loss, n); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    { loss_mean_of_chunks<<<1, kLossThreads, 0, s>>>(row_loss, n_mean, n_chunks, loss); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace gnn
