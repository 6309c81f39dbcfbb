// exchange.cu - the halo-gradient return of the backward pass (Sylvie page,
// backward propagation, Alg. 2: the feature gradients J of a partition's HALO
// vertices are sent to the partitions that own those vertices and added to
// their own gradients there).
//
// The exchange goes through a gradient table in HBM indexed by global vertex
// id (fp32, like the stale-representation table of DIGEST's pull / push):
//   send:    gtable[halo_ids[i]] += dH[n_local + i]      (i < n_halo)
//   receive: dH[v] += gtable[local_ids[v]]               (v < n_local)
// A partition's halo ids are distinct (checked with the push claim words, a
// repeated id is reported and its rows skipped), so one send launch has no
// conflicting updates; sends of several partitions are ordered on the stream,
// so the sums are formed in a fixed order (no atomics, reproducible bits).
// One warp per row (16 blocks per SM loop over the rows), 4 columns per lane
// per step.
#include <algorithm>

#include "gnn_internal.cuh"

namespace gnn {

namespace {

__device__ __forceinline__ float4 load4v(const float *p) { return *reinterpret_cast<const float4 *>(p); }
__device__ __forceinline__ float4 load4v(const __nv_bfloat16 *p) {
    const uint2 v = *reinterpret_cast<const uint2 *>(p);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xffff0000u));
}
__device__ __forceinline__ void store4v(float *p, float4 v) { *reinterpret_cast<float4 *>(p) = v; }
__device__ __forceinline__ void store4v(__nv_bfloat16 *p, float4 v) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<uint32_t *>(&a), *reinterpret_cast<uint32_t *>(&b));
}
template <typename T>
__device__ __forceinline__ float elem(const T *p);
template <>
__device__ __forceinline__ float elem(const float *p) {
    return *p;
}
template <>
__device__ __forceinline__ float elem(const __nv_bfloat16 *p) {
    return __bfloat162float(*p);
}
__device__ __forceinline__ void set_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void set_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) grad_send_kernel(const T *__restrict__ dH, int64_t ld_dh, int64_t row0,
                                                        const int64_t *__restrict__ ids, int64_t n, int64_t n_table,
                                                        const uint32_t *__restrict__ claim, uint32_t gen,
                                                        float *__restrict__ gt, int64_t ld_gt, int64_t f, int *err) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        const int64_t id = ids[i];
        if (id < 0 || id >= n_table) continue;  // reported by the claim pass
        if (claim[id] != ((gen << 2) | 1u)) {
            if (lane == 0) atomicOr(err, 1);  // repeated id: its rows are not sent
            continue;
        }
        const T *src = dH + (row0 + i) * ld_dh;
        float *dst = gt + id * ld_gt;
        for (int64_t c = (int64_t)lane * 4; c < f; c += 128) {
            if (c + 4 <= f) {
                const float4 a = load4v(dst + c), b = load4v(src + c);
                store4v(dst + c, make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w));
            } else {
                for (int64_t k = c; k < f; ++k) dst[k] += elem(src + k);
            }
        }
    }
}

template <typename T>
__global__ void __launch_bounds__(256) grad_recv_kernel(const float *__restrict__ gt, int64_t ld_gt, int64_t n_table,
                                                        const int64_t *__restrict__ ids, int64_t n,
                                                        T *__restrict__ dH, int64_t ld_dh, int64_t f, int *err) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < n; v += nw) {
        const int64_t id = ids[v];
        if (id < 0 || id >= n_table) {
            if (lane == 0) atomicOr(err, 1);
            continue;
        }
        const float *src = gt + id * ld_gt;
        T *dst = dH + v * ld_dh;
        for (int64_t c = (int64_t)lane * 4; c < f; c += 128) {
            if (c + 4 <= f) {
                const float4 a = load4v(dst + c), b = load4v(src + c);
                store4v(dst + c, make_float4(a.x + b.x, a.y + b.y, a.z + b.z, a.w + b.w));
            } else {
                for (int64_t k = c; k < f; ++k) set_elem(dst + k, elem(dst + k) + src[k]);
            }
        }
    }
}

// dst[i, 0:f] = src[ids[i], 0:f], bit-exact: one warp per row, 16-byte pieces
// (rows start on 16-byte boundaries) and element copies for the tail
template <typename T>
__global__ void __launch_bounds__(256) gather_rows_kernel(const T *__restrict__ src, int64_t ld_src, int64_t n_src,
                                                          const int64_t *__restrict__ ids, int64_t n,
                                                          T *__restrict__ dst, int64_t ld_dst, int64_t f, int *err) {
    constexpr int EPV = 16 / (int)sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        const int64_t id = ids[i];
        if (id < 0 || id >= n_src) {
            if (lane == 0 && err) atomicOr(err, kErrIndex);
            continue;
        }
        const T *a = src + id * ld_src;
        T *b = dst + i * ld_dst;
        const int64_t nv = f / EPV;
        for (int64_t v = lane; v < nv; v += 32)
            reinterpret_cast<uint4 *>(b)[v] = __ldg(reinterpret_cast<const uint4 *>(a) + v);
        for (int64_t c = nv * EPV + lane; c < f; c += 32) b[c] = a[c];
    }
}

// dst[ids[i], 0:f] += src[i, 0:f] (fp32 sum, stored as T); the ids of one launch
// are distinct, so rows never collide
template <typename T>
__global__ void __launch_bounds__(256) scatter_add_rows_kernel(const T *__restrict__ src, int64_t ld_src,
                                                               const int64_t *__restrict__ ids, int64_t n,
                                                               T *__restrict__ dst, int64_t ld_dst, int64_t n_dst,
                                                               int64_t f, int *err) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        const int64_t id = ids[i];
        if (id < 0 || id >= n_dst) {
            if (lane == 0 && err) atomicOr(err, kErrIndex);
            continue;
        }
        const T *a = src + i * ld_src;
        T *b = dst + id * ld_dst;
        for (int64_t c = (int64_t)lane * 4; c < f; c += 128) {
            if (c + 4 <= f) {
                const float4 x = load4v(b + c), y = load4v(a + c);
                store4v(b + c, make_float4(x.x + y.x, x.y + y.y, x.z + y.z, x.w + y.w));
            } else {
                for (int64_t k = c; k < f; ++k) set_elem(b + k, elem(b + k) + elem(a + k));
            }
        }
    }
}

}  // namespace

gnn_status launch_gather_rows(const void *src, int64_t ld_src, int64_t n_src, const int64_t *ids, int64_t n,
                              void *dst, int64_t ld_dst, int64_t f, gnn_dtype dt, int *err, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n * 32, 256), (int64_t)num_sms() * 16);
    if (dt == GNN_BF16)
        { gather_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(src), ld_src,
                                                                   n_src, ids, n, static_cast<__nv_bfloat16 *>(dst),
                                                                   ld_dst, f, err); GNN_LAUNCHED(1); }
    else
        { gather_rows_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(src), ld_src, n_src, ids, n,
                                                           static_cast<float *>(dst), ld_dst, f, err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_scatter_add_rows(const void *src, int64_t ld_src, const int64_t *ids, int64_t n, void *dst,
                                   int64_t ld_dst, int64_t n_dst, int64_t f, gnn_dtype dt, int *err, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n * 32, 256), (int64_t)num_sms() * 16);
    if (dt == GNN_BF16)
        { scatter_add_rows_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(src), ld_src, ids, n, static_cast<__nv_bfloat16 *>(dst), ld_dst, n_dst,
            f, err); GNN_LAUNCHED(1); }
    else
        { scatter_add_rows_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(src), ld_src, ids, n,
                                                                static_cast<float *>(dst), ld_dst, n_dst, f, err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_grad_send(gnn_graph *g, const void *dH, int64_t ld_dh, int64_t f, const int64_t *halo_ids,
                            float *gtable, int64_t ld_gt, int64_t n_table, gnn_dtype dt, cudaStream_t s) {
    const int64_t n = g->n_halo;
    if (n == 0) return GNN_OK;
    uint32_t gen = 0;
    gnn_status st = launch_push_claim(g, halo_ids, n, n_table, &gen, s);
    if (st != GNN_OK) return st;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n * 32, 256), (int64_t)num_sms() * 16);
    if (dt == GNN_BF16)
        { grad_send_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(dH), ld_dh,
                                                                 g->n_local, halo_ids, n, n_table, g->claim, gen,
                                                                 gtable, ld_gt, f, g->err); GNN_LAUNCHED(1); }
    else
        { grad_send_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(dH), ld_dh, g->n_local, halo_ids,
                                                         n, n_table, g->claim, gen, gtable, ld_gt, f, g->err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_grad_recv(gnn_graph *g, const float *gtable, int64_t ld_gt, int64_t n_table,
                            const int64_t *local_ids, void *dH, int64_t ld_dh, int64_t f, gnn_dtype dt,
                            cudaStream_t s) {
    const int64_t n = g->n_local;
    if (n == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n * 32, 256), (int64_t)num_sms() * 16);
    if (dt == GNN_BF16)
        { grad_recv_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(gtable, ld_gt, n_table, local_ids, n,
                                                                 static_cast<__nv_bfloat16 *>(dH), ld_dh, f, g->err); GNN_LAUNCHED(1); }
    else
        { grad_recv_kernel<float><<<blocks, 256, 0, s>>>(gtable, ld_gt, n_table, local_ids, n,
                                                         static_cast<float *>(dH), ld_dh, f, g->err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace gnn
