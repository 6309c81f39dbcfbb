// update_simt.cu - the dense update of the layer on the CUDA cores (fp32 FMA),
// used for fp32 data, where tensor-core inputs would round to tf32 / bf16.
//
// Forward (CAGNET page, GNN section):  H_out = act(Z W)
// Backward (chain rule):               dY = G * 1[H_out > 0] (or G)
//                                      dZ = dY W^T
//                                      dW = Z^T dY  (split over row slabs; the
//                                      slabs' partials are added in slab order)
// W is the packed fp32 matrix Wp (Kp x N, leading dimension ld_w): the rows of
// the aggregation layout, with zero rows at GraphSAGE padding columns.
#include "gnn_internal.cuh"

namespace gnn {

namespace {

constexpr int BM = 64, BN = 64, BK = 16, NT = 256;

__device__ __forceinline__ float ld_elem(const float *p) { return *p; }
__device__ __forceinline__ float ld_elem(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void st_elem(float *p, float v) { *p = v; }
__device__ __forceinline__ void st_elem(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

// C[n x N] = A[n x K] * B[K x N]; A element (i, k) and B element (k, j) come
// from the loaders; 4 x 4 outputs per thread.
// A and C have type TA (the forward's Z and H_out, or the backward's G and dZ),
// the mask operand M the activations' type TM.
template <typename TA, typename TM, int AMODE>
__global__ void __launch_bounds__(NT) gemm_simt_kernel(const TA *__restrict__ A, int64_t lda,
                                                       const TM *__restrict__ M, int64_t ldm,
                                                       const float *__restrict__ Wp, int64_t ldw, int64_t n,
                                                       int64_t K, int64_t N, int relu, TA *__restrict__ C,
                                                       int64_t ldc) {
    // AMODE 0: A = Z (n x K), B[k][j] = Wp[k][j]          (forward)
    // AMODE 1: A = dY = G * mask (n x K=N_out), B[k][j] = Wp[j][k]   (dZ = dY Wp^T)
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t m0 = (int64_t)blockIdx.x * BM, n0 = (int64_t)blockIdx.y * BN;
    float acc[4][4] = {};
    for (int64_t k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            int idx = tid + q * NT;  // 0..1023
            int mm = idx / BK, kk = idx % BK;
            int64_t i = m0 + mm, k = k0 + kk;
            float a = 0.f;
            if (i < n && k < K) {
                a = ld_elem(A + i * lda + k);
                if (AMODE == 1 && relu && !(ld_elem(M + i * ldm + k) > 0.f)) a = 0.f;
                // bf16 activations: dY is a bf16 operand of the products, as on the tensor cores
                if (AMODE == 1 && sizeof(TA) == 4 && sizeof(TM) == 2) a = __bfloat162float(__float2bfloat16_rn(a));
            }
            As[kk][mm] = a;
            int kb = idx / BN, jb = idx % BN;
            int64_t kg = k0 + kb, jg = n0 + jb;
            float bv = 0.f;
            if (kg < K && jg < N) bv = AMODE == 0 ? Wp[kg * ldw + jg] : Wp[jg * ldw + kg];
            Bs[kb][jb] = bv;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], bb[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = As[kk][ty * 4 + q];
                bb[q] = Bs[kk][tx * 4 + q];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], bb[y], acc[x][y]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        int64_t i = m0 + ty * 4 + x;
        if (i >= n) continue;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            int64_t j = n0 + tx * 4 + y;
            if (j >= N) continue;
            float v = acc[x][y];
            if (AMODE == 0 && relu && !(v > 0.f)) v = 0.f;
            st_elem(C + i * ldc + j, v);
        }
    }
}

// dWp partial of one row slab: P[s][k][j] = sum_{i in slab s} Z[i][k] * dY[i][j]
// Z and H_out have the activations' type T, G the gradients' type TG
template <typename T, typename TG>
__global__ void __launch_bounds__(NT) wgrad_simt_kernel(const T *__restrict__ Z, int64_t ldz, const TG *__restrict__ G,
                                                        int64_t ldg, const T *__restrict__ Hout, int64_t ldh, int relu,
                                                        int64_t n, int64_t Kp, int64_t N, int64_t rows_per_slab,
                                                        float *__restrict__ P) {
    __shared__ float Zs[BK][BM + 4];
    __shared__ float Ys[BK][BN + 4];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int64_t k0 = (int64_t)blockIdx.y * BM, j0 = (int64_t)blockIdx.x * BN;
    const int64_t slab = blockIdx.z;
    const int64_t r0 = slab * rows_per_slab;
    const int64_t r1 = min(n, r0 + rows_per_slab);
    float acc[4][4] = {};
    for (int64_t i0 = r0; i0 < r1; i0 += BK) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            int idx = tid + q * NT;
            int ii = idx / BM, cc = idx % BM;
            int64_t i = i0 + ii;
            float z = 0.f, y = 0.f;
            if (i < r1) {
                if (k0 + cc < Kp) z = ld_elem(Z + i * ldz + k0 + cc);
                if (j0 + cc < N) {
                    y = ld_elem(G + i * ldg + j0 + cc);
                    if (relu && !(ld_elem(Hout + i * ldh + j0 + cc) > 0.f)) y = 0.f;
                    // bf16 activations: dY is a bf16 operand of the products, as on the tensor cores
                    if (sizeof(TG) == 4 && sizeof(T) == 2) y = __bfloat162float(__float2bfloat16_rn(y));
                }
            }
            Zs[ii][cc] = z;
            Ys[ii][cc] = y;
        }
        __syncthreads();
#pragma unroll
        for (int ii = 0; ii < BK; ++ii) {
            float a[4], b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = Zs[ii][ty * 4 + q];
                b[q] = Ys[ii][tx * 4 + q];
            }
#pragma unroll
            for (int x = 0; x < 4; ++x)
#pragma unroll
                for (int y = 0; y < 4; ++y) acc[x][y] = fmaf(a[x], b[y], acc[x][y]);
        }
        __syncthreads();
    }
    float *Ps = P + slab * Kp * N;
#pragma unroll
    for (int x = 0; x < 4; ++x) {
        int64_t k = k0 + ty * 4 + x;
        if (k >= Kp) continue;
#pragma unroll
        for (int y = 0; y < 4; ++y) {
            int64_t j = j0 + tx * 4 + y;
            if (j < N) Ps[k * N + j] = acc[x][y];
        }
    }
}

// slab partials added in slab order, in double: the result does not depend on
// scheduling and the fp32 error stays that of the short per-slab chains
__global__ void sum_slabs_kernel(const float *__restrict__ P, int64_t slabs, int64_t KN, float *__restrict__ dWp) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= KN) return;
    double s = 0.0;
    for (int64_t q = 0; q < slabs; ++q) s += (double)P[q * KN + x];
    dWp[x] = (float)s;
}

// Rows per slab: fp32 data keeps each fp32 chain short (<= 256 rows, up to 4096
// slabs); bf16 data (whose inputs carry 8-bit mantissas) uses about four slabs
// per SM.
int64_t wgrad_slabs(int64_t n, int64_t Kp, int64_t N, bool fine) {
    if (fine) {
        int64_t sl = ceil_div(n, 256);
        if (sl > 4096) sl = 4096;
        return sl < 1 ? 1 : sl;
    }
    int64_t tiles = ceil_div(Kp, BM) * ceil_div(N, BN);
    int64_t want = ceil_div(152 * 4, tiles);
    int64_t max_by_rows = ceil_div(n, 2048);
    int64_t sl = want < max_by_rows ? want : max_by_rows;
    if (sl < 1) sl = 1;
    if (sl > 1024) sl = 1024;
    return sl;
}

template <typename T>
gnn_status update_fwd_t(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                        int relu, void *out, int64_t ld_o, cudaStream_t s) {
    dim3 grid((unsigned)ceil_div(n, BM), (unsigned)ceil_div(N, BN));
    { gemm_simt_kernel<T, T, 0><<<grid, NT, 0, s>>>(static_cast<const T *>(Z), ld_z, nullptr, 0, Wp, ld_w, n, Kp, N,
                                                  relu, static_cast<T *>(out), ld_o); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

template <typename T, typename TG>
gnn_status update_bwd_t(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                        int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N, float *dWp,
                        void *dZ, int64_t ld_dz, float *ws, cudaStream_t s) {
    const TG *Gt = static_cast<const TG *>(G);
    const T *Ht = static_cast<const T *>(Hout);
    if (dZ) {
        dim3 grid((unsigned)ceil_div(n, BM), (unsigned)ceil_div(Kp, BN));
        { gemm_simt_kernel<TG, T, 1><<<grid, NT, 0, s>>>(Gt, ld_g, Ht, ld_h, Wp, ld_w, n, N, Kp, relu,
                                                       static_cast<TG *>(dZ), ld_dz); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    const int64_t slabs = wgrad_slabs(n, Kp, N, sizeof(T) == 4);
    const int64_t rows_per_slab = ceil_div(n, slabs);
    dim3 grid((unsigned)ceil_div(N, BN), (unsigned)ceil_div(Kp, BM), (unsigned)slabs);
    { wgrad_simt_kernel<T, TG><<<grid, NT, 0, s>>>(static_cast<const T *>(Z), ld_z, Gt, ld_g, Ht, ld_h, relu, n, Kp,
                                                  N, rows_per_slab, ws); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    { sum_slabs_kernel<<<(unsigned)ceil_div(Kp * N, 256), 256, 0, s>>>(ws, slabs, Kp * N, dWp); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace

size_t update_bwd_ws_bytes(int64_t n, int64_t Kp, int64_t N, gnn_dtype dt) {
    return (size_t)wgrad_slabs(n, Kp, N, dt == GNN_F32) * (size_t)Kp * (size_t)N * sizeof(float);
}

gnn_status launch_update_fwd(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w,
                             int64_t N, int relu, void *out, int64_t ld_o, gnn_dtype dt, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    if (dt == GNN_BF16) return update_fwd_t<__nv_bfloat16>(Z, ld_z, n, Kp, Wp, ld_w, N, relu, out, ld_o, s);
    return update_fwd_t<float>(Z, ld_z, n, Kp, Wp, ld_w, N, relu, out, ld_o, s);
}

gnn_status launch_update_bwd(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                             int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                             float *dWp, void *dZ, int64_t ld_dz, gnn_dtype dt, gnn_dtype gdt, float *ws,
                             size_t ws_bytes, cudaStream_t s) {
    if (ws_bytes < update_bwd_ws_bytes(n, Kp, N, dt)) return GNN_EINVAL;
    if (n == 0) {
        GNN_CUDA_TRY(cudaMemsetAsync(dWp, 0, (size_t)Kp * (size_t)N * sizeof(float), s));
        return GNN_OK;
    }
    if (dt == GNN_BF16 && gdt == GNN_BF16)
        return update_bwd_t<__nv_bfloat16, __nv_bfloat16>(G, ld_g, Hout, ld_h, relu, Z, ld_z, n, Kp, Wp, ld_w, N, dWp,
                                                          dZ, ld_dz, ws, s);
    if (dt == GNN_BF16)
        return update_bwd_t<__nv_bfloat16, float>(G, ld_g, Hout, ld_h, relu, Z, ld_z, n, Kp, Wp, ld_w, N, dWp, dZ,
                                                  ld_dz, ws, s);
    if (gdt != GNN_F32) return GNN_EINVAL;
    return update_bwd_t<float, float>(G, ld_g, Hout, ld_h, relu, Z, ld_z, n, Kp, Wp, ld_w, N, dWp, dZ, ld_dz, ws, s);
}

}  // namespace gnn
