// loss.cu - training-harness helper (not a layer step): mean softmax
// cross-entropy over the local rows and its gradient with respect to the
// logits, G = (softmax - onehot) / n.  One warp per row; the mean is summed in
// a fixed order by one block, so the loss is reproducible bit for bit.
#include "gnn_internal.cuh"

namespace gnn {

namespace {

__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void softmax_ce_rows(const T *__restrict__ X, int64_t ld, int64_t n, int64_t C,
                                const int32_t *__restrict__ labels, T *__restrict__ G, int64_t ld_g,
                                float *__restrict__ row_loss) {
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
    const float inv_n = 1.0f / (float)n;
    for (int64_t c = lane; c < C; c += 32) {
        float p = expf(ld_elem(x + c) - lse);
        st_elem(G + i * ld_g + c, (p - (c == y ? 1.f : 0.f)) * inv_n);
    }
    if (lane == 0) row_loss[i] = ok ? lse - ld_elem(x + y) : NAN;
}

// rows of up to 32 * CPL classes: each lane keeps its logits in registers, so a
// row is read once
template <typename T, int CPL>
__global__ void softmax_ce_rows_reg(const T *__restrict__ X, int64_t ld, int64_t n, int64_t C,
                                    const int32_t *__restrict__ labels, T *__restrict__ G, int64_t ld_g,
                                    float *__restrict__ row_loss) {
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (i >= n) return;
    const T *x = X + i * ld;
    float v[CPL];
    float mx = -INFINITY;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        const int64_t c = lane + 32 * q;
        v[q] = c < C ? ld_elem(x + c) : -INFINITY;
        mx = fmaxf(mx, v[q]);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    float se = 0.f;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        v[q] = lane + 32 * q < C ? expf(v[q] - mx) : 0.f;
        se += v[q];
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) se += __shfl_xor_sync(0xffffffffu, se, o);
    const int32_t y = labels[i];
    const float inv_n = 1.0f / (float)n, inv_se = 1.0f / se;
#pragma unroll
    for (int q = 0; q < CPL; ++q) {
        const int64_t c = lane + 32 * q;
        if (c < C) st_elem(G + i * ld_g + c, (v[q] * inv_se - (c == y ? 1.f : 0.f)) * inv_n);
    }
    if (lane == 0) row_loss[i] = (y >= 0 && y < C) ? mx + logf(se) - ld_elem(x + y) : NAN;
}

__global__ void mean_fixed_order(const float *__restrict__ v, int64_t n, float *out) {
    __shared__ float part[1024];
    float s = 0.f;
    for (int64_t i = threadIdx.x; i < n; i += blockDim.x) s += v[i];
    part[threadIdx.x] = s;
    __syncthreads();
    for (int w = blockDim.x / 2; w > 0; w >>= 1) {
        if ((int)threadIdx.x < w) part[threadIdx.x] += part[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) *out = n > 0 ? part[0] / (float)n : 0.f;
}

}  // namespace

gnn_status launch_softmax_ce(const void *logits, int64_t ld, int64_t n, int64_t C, const int32_t *labels, void *G,
                             int64_t ld_g, float *row_loss, float *loss, gnn_dtype dt, cudaStream_t s) {
    if (n > 0 && C <= 256) {
        const unsigned blocks = (unsigned)ceil_div(n * 32, 256);
        if (dt == GNN_BF16)
            { softmax_ce_rows_reg<__nv_bfloat16, 8><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(logits), ld,
                                                                          n, C, labels,
                                                                          static_cast<__nv_bfloat16 *>(G), ld_g,
                                                                          row_loss); GNN_LAUNCHED(1); }
        else
            { softmax_ce_rows_reg<float, 8><<<blocks, 256, 0, s>>>(static_cast<const float *>(logits), ld, n, C, labels,
                                                                  static_cast<float *>(G), ld_g, row_loss); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    } else if (n > 0) {
        const unsigned blocks = (unsigned)ceil_div(n * 32, 256);
        if (dt == GNN_BF16)
            { softmax_ce_rows<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(logits), ld, n,
                                                                   C, labels, static_cast<__nv_bfloat16 *>(G), ld_g,
                                                                   row_loss); GNN_LAUNCHED(1); }
        else
            { softmax_ce_rows<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(logits), ld, n, C, labels,
                                                          static_cast<float *>(G), ld_g, row_loss); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    { mean_fixed_order<<<1, 1024, 0, s>>>(row_loss, n, loss); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace gnn
