// gat.cu - the graph-attention (GAT) layer's own steps.  The Sylvie page names
// GAT among the models it trains and the DIGEST page benchmarks it; neither
// prints the layer, so this is the textbook single-head form:
//   T = H W (every row),  s_src[u] = T[u] . a_src,  s_dst[v] = T[v] . a_dst,
//   alpha_vu = softmax over row v of LeakyReLU_0.2(s_dst[v] + s_src[u]),
//   Y[v] = sum_u alpha_vu T[u],  H_out = act(Y).
// The products T = H W, dW = H^T dT, dH = dT W^T run on the update kernels and
// the two weighted sums (forward over the block, backward over its transpose)
// on the aggregation kernel with the attention as per-entry weights; this file
// holds the rest: the scores, the row softmax, its backward (an SDDMM: one dot
// product dY[v] . T[u] per entry), the per-column score sums over the
// transpose, the rank-1 terms and the attention vectors' gradients.
// Every sum is formed in a fixed order (no float atomics).
#include <algorithm>

#include "gnn_internal.cuh"

namespace gnn {

namespace {

constexpr float kSlope = 0.2f;  // LeakyReLU slope of the scores

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}
__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}
__device__ __forceinline__ float lrelu(float z) { return z > 0.f ? z : kSlope * z; }
__device__ __forceinline__ float flag_end(float a) { return __uint_as_float(__float_as_uint(a) | 0x80000000u); }
__device__ __forceinline__ float unflag(float a) { return __uint_as_float(__float_as_uint(a) & 0x7fffffffu); }

// s_src[u] = T[u] . a_src (u < n_total), s_dst[v] = T[v] . a_dst (v < n_local): one warp per row
template <typename T>
__global__ void __launch_bounds__(256) gat_scores_kernel(const T *__restrict__ Tm, int64_t ld, int64_t n_total,
                                                         int64_t n_local, int64_t f, const float *__restrict__ a_src,
                                                         const float *__restrict__ a_dst, float *__restrict__ s_src,
                                                         float *__restrict__ s_dst) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < n_total; u += nw) {
        const T *t = Tm + u * ld;
        float ps = 0.f, pd = 0.f;
        for (int64_t c = lane; c < f; c += 32) {
            const float x = ldf(t + c);
            ps = fmaf(x, a_src[c], ps);
            if (u < n_local) pd = fmaf(x, a_dst[c], pd);
        }
        ps = warp_sum(ps);
        pd = warp_sum(pd);
        if (lane == 0) {
            s_src[u] = ps;
            if (u < n_local) s_dst[u] = pd;
        }
    }
}

// alpha[e] over the entries of row v (the library's entry order): softmax of
// LeakyReLU(s_dst[v] + s_src[col]); the last entry of each row carries the
// sign bit (the aggregation's row end).  One warp per row, three passes.
__global__ void __launch_bounds__(256) gat_softmax_kernel(const int32_t *__restrict__ rowptr,
                                                          const uint32_t *__restrict__ colidx, uint32_t colmask,
                                                          int64_t n_local, const float *__restrict__ s_src,
                                                          const float *__restrict__ s_dst, float *__restrict__ alpha) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < n_local; v += nw) {
        const int32_t b = rowptr[v], e = rowptr[v + 1];
        if (e == b) continue;
        const float sd = s_dst[v];
        float mx = -INFINITY;
        for (int32_t k = b + lane; k < e; k += 32) mx = fmaxf(mx, lrelu(sd + s_src[colidx[k] & colmask]));
        mx = warp_max(mx);
        float sum = 0.f;
        for (int32_t k = b + lane; k < e; k += 32) {
            const float x = __expf(lrelu(sd + s_src[colidx[k] & colmask]) - mx);
            alpha[k] = x;
            sum += x;
        }
        sum = warp_sum(sum);
        const float inv = 1.0f / sum;
        __syncwarp();
        for (int32_t k = b + lane; k < e; k += 32) {
            const float a = alpha[k] * inv;
            alpha[k] = k == e - 1 ? flag_end(a) : a;
        }
    }
}

// dY = relu ? G * 1[H_out > 0] : G, stored in G's type
template <typename TG, typename TA>
__global__ void gat_mask_kernel(const TG *__restrict__ G, int64_t ld_g, const TA *__restrict__ Hout, int64_t ld_h,
                                int64_t n, int64_t f, TG *__restrict__ Y, int64_t ld_y) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n * f) return;
    const int64_t r = x / f, c = x % f;
    const TG g = G[r * ld_g + c];
    Y[r * ld_y + c] = (!Hout || ldf(Hout + r * ld_h + c) > 0.f) ? g : TG(0.f);
}

// four consecutive values c .. c + 3 of a row as fp32 (values at or past f: 0)
__device__ __forceinline__ void ld4(const float *p, int64_t c, int64_t f, float (&v)[4]) {
    if (c + 4 <= f) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(p + c));
        v[0] = q.x, v[1] = q.y, v[2] = q.z, v[3] = q.w;
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = c + j < f ? p[c + j] : 0.f;
    }
}
__device__ __forceinline__ void ld4(const __nv_bfloat16 *p, int64_t c, int64_t f, float (&v)[4]) {
    if (c + 4 <= f) {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(p + c));
        v[0] = __uint_as_float(q.x << 16), v[1] = __uint_as_float(q.x & 0xffff0000u);
        v[2] = __uint_as_float(q.y << 16), v[3] = __uint_as_float(q.y & 0xffff0000u);
    } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = c + j < f ? __bfloat162float(p[c + j]) : 0.f;
    }
}

// The score gradient's first factor for every entry e of the block (library
// order): dz[e] = dY[row e] . T[col e].  G lanes per entry (four values per
// lane per step), so the work spreads evenly whatever the row lengths; the
// row of each entry comes from the graph's entry-row map.
template <typename TG, typename TA, int G>
__global__ void __launch_bounds__(256) gat_sddmm_kernel(const int32_t *__restrict__ erow,
                                                        const uint32_t *__restrict__ colidx, uint32_t colmask,
                                                        int64_t nnz, const TG *__restrict__ dY, int64_t ld_y,
                                                        const TA *__restrict__ Tm, int64_t ld_t, int64_t f,
                                                        float *__restrict__ dz) {
    constexpr int EPW = 32 / G;  // entries per warp and step
    const int lane = threadIdx.x & 31, sub = lane % G;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t kb = warp * EPW; kb < nnz; kb += nw * EPW) {  // the same trip count for the whole warp
        const int64_t k = kb + lane / G;
        float p = 0.f;
        if (k < nnz) {
            const TG *y = dY + (int64_t)erow[k] * ld_y;
            const TA *t = Tm + (int64_t)(colidx[k] & colmask) * ld_t;
            for (int64_t c = 4 * sub; c < f; c += 4 * G) {
                float a[4], b[4];
                ld4(y, c, f, a);
                ld4(t, c, f, b);
#pragma unroll
                for (int j = 0; j < 4; ++j) p = fmaf(a[j], b[j], p);
            }
        }
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) p += __shfl_xor_sync(0xffffffffu, p, o);
        if (k < nnz && sub == 0) dz[k] = p;
    }
}

// The softmax backward of row v, from dz[e] = dY[v] . T[col_e]:
// dz_e <- alpha_e (dz_e - sum_e' alpha_e' dz_e') * LeakyReLU'(z_e), and
// ds_dst[v] = sum_e dz_e.  One warp per row, the lanes over its entries.
__global__ void __launch_bounds__(256) gat_softmax_backward_kernel(
    const int32_t *__restrict__ rowptr, const uint32_t *__restrict__ colidx, uint32_t colmask, int64_t n_local,
    const float *__restrict__ s_src, const float *__restrict__ s_dst, const float *__restrict__ alpha,
    float *__restrict__ dz, float *__restrict__ ds_dst) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < n_local; v += nw) {
        const int32_t b = rowptr[v], e = rowptr[v + 1];
        float dsum = 0.f;
        for (int32_t k = b + lane; k < e; k += 32) dsum = fmaf(unflag(alpha[k]), dz[k], dsum);
        dsum = warp_sum(dsum);
        const float sd = s_dst[v];
        float s = 0.f;
        for (int32_t k = b + lane; k < e; k += 32) {
            const float a = unflag(alpha[k]);
            const float z = sd + s_src[colidx[k] & colmask];
            const float g = a * (dz[k] - dsum) * (z > 0.f ? 1.f : kSlope);
            dz[k] = g;
            s += g;
        }
        s = warp_sum(s);
        if (lane == 0) ds_dst[v] = s;
    }
}

// entry-row map of a CSR: erow[k] = v for k in [rowptr[v], rowptr[v + 1])
__global__ void entry_rows_kernel(const int32_t *__restrict__ rowptr, int64_t n_rows, int32_t *__restrict__ erow) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < n_rows; v += nw)
        for (int32_t k = rowptr[v] + lane; k < rowptr[v + 1]; k += 32) erow[k] = (int32_t)v;
}

// Over the transpose: ds_src[u] = sum of dz over the entries holding column u,
// and the attention in the transpose's entry order (row ends flagged).  t2b[k]
// is the block entry (library order) behind transpose entry k.
__global__ void __launch_bounds__(256) gat_transpose_kernel(const int32_t *__restrict__ rowptrT, int64_t n_total,
                                                            const int32_t *__restrict__ t2b,
                                                            const float *__restrict__ dz,
                                                            const float *__restrict__ alpha,
                                                            float *__restrict__ ds_src, float *__restrict__ alphaT) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t u = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; u < n_total; u += nw) {
        const int32_t b = rowptrT[u], e = rowptrT[u + 1];
        float s = 0.f;
        for (int32_t k = b + lane; k < e; k += 32) {
            const int32_t be = t2b[k];
            s += dz[be];
            const float a = unflag(alpha[be]);
            alphaT[k] = k == e - 1 ? flag_end(a) : a;
        }
        s = warp_sum(s);
        if (lane == 0) ds_src[u] = s;
    }
}

// dT[u] += ds_src[u] a_src + [u < n_local] ds_dst[u] a_dst (fp32, stored as TG)
template <typename TG>
__global__ void gat_rank1_kernel(TG *__restrict__ dT, int64_t ld, int64_t n_total, int64_t n_local, int64_t f,
                                 const float *__restrict__ ds_src, const float *__restrict__ ds_dst,
                                 const float *__restrict__ a_src, const float *__restrict__ a_dst) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n_total * f) return;
    const int64_t u = x / f, c = x % f;
    float d = ldf(dT + u * ld + c) + ds_src[u] * a_src[c];
    if (u < n_local) d += ds_dst[u] * a_dst[c];
    stf(dT + u * ld + c, d);
}

// partial[b][c] = sum over the rows of chunk b of w[u] T[u][c]: four running
// sums over the rows u = r0 + 4i + j (j = 0..3), so four loads are in flight,
// added as (s0 + s1) + (s2 + s3); the host-side launch then adds the chunks'
// partials in chunk order (a fixed order: the result is reproducible)
template <typename TA>
__global__ void gat_colsum_kernel(const TA *__restrict__ Tm, int64_t ld, int64_t n_rows, int64_t f,
                                  const float *__restrict__ w, int64_t rows_per_chunk, float *__restrict__ partial) {
    const int64_t bch = blockIdx.y;
    const int64_t r0 = bch * rows_per_chunk;
    const int64_t r1 = min(n_rows, r0 + rows_per_chunk);
    for (int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; c < f; c += (int64_t)gridDim.x * blockDim.x) {
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        int64_t u = r0;
        for (; u + 4 <= r1; u += 4) {
#pragma unroll
            for (int j = 0; j < 4; ++j) s[j] = fmaf(w[u + j], ldf(Tm + (u + j) * ld + c), s[j]);
        }
        for (int j = 0; u < r1; ++u, ++j) s[j] = fmaf(w[u], ldf(Tm + u * ld + c), s[j]);
        partial[bch * f + c] = (s[0] + s[1]) + (s[2] + s[3]);
    }
}

__global__ void gat_chunks_sum_kernel(const float *__restrict__ partial, int64_t chunks, int64_t f,
                                      float *__restrict__ out) {
    const int64_t c = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= f) return;
    double s = 0.0;
    for (int64_t b = 0; b < chunks; ++b) s += (double)partial[b * f + c];
    out[c] = (float)s;
}

__global__ void iota_kernel(int32_t *__restrict__ out, int64_t n) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) out[i] = (int32_t)i;
}

// inv[perm[i]] = i
__global__ void invert_kernel(const int32_t *__restrict__ perm, int64_t n, int32_t *__restrict__ inv) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) inv[perm[i]] = (int32_t)i;
}

// t2b[k] = fpos[permT[tperm[k]]] (tperm null: identity)
__global__ void compose_kernel(const int32_t *__restrict__ tperm, const int32_t *__restrict__ permT,
                               const int32_t *__restrict__ fpos, int64_t n, int32_t *__restrict__ t2b) {
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t k = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; k < n; k += stride) {
        const int32_t ks = tperm ? tperm[k] : (int32_t)k;
        const int32_t eo = permT[ks];
        t2b[k] = fpos ? fpos[eo] : eo;
    }
}

}  // namespace

gnn_status launch_iota(int32_t *out, int64_t n, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    { iota_kernel<<<(unsigned)std::min<int64_t>(ceil_div(n, 256), (int64_t)num_sms() * 8), 256, 0, s>>>(out, n); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_entry_map(const int32_t *fperm, const int32_t *tperm, const int32_t *permT, int64_t nnz,
                                int32_t *t2b, int32_t *scratch, cudaStream_t s) {
    if (nnz == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(nnz, 256), (int64_t)num_sms() * 8);
    if (fperm) {
        { invert_kernel<<<blocks, 256, 0, s>>>(fperm, nnz, scratch); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    { compose_kernel<<<blocks, 256, 0, s>>>(tperm, permT, fperm ? scratch : nullptr, nnz, t2b); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_scores(const void *T, int64_t ld, int64_t n_total, int64_t n_local, int64_t f,
                             const float *a_src, const float *a_dst, float *s_src, float *s_dst, gnn_dtype dt,
                             cudaStream_t s) {
    if (n_total == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n_total * 32, 256), (int64_t)num_sms() * 16);
    if (dt == GNN_BF16)
        { gat_scores_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const __nv_bfloat16 *>(T), ld, n_total,
                                                                  n_local, f, a_src, a_dst, s_src, s_dst); GNN_LAUNCHED(1); }
    else
        { gat_scores_kernel<float><<<blocks, 256, 0, s>>>(static_cast<const float *>(T), ld, n_total, n_local, f,
                                                          a_src, a_dst, s_src, s_dst); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_softmax(const gnn_graph *g, const float *s_src, const float *s_dst, float *alpha,
                              cudaStream_t s) {
    if (g->n_local == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(g->n_local * 32, 256), (int64_t)num_sms() * 16);
    { gat_softmax_kernel<<<blocks, 256, 0, s>>>(g->rowptr, reinterpret_cast<const uint32_t *>(g->colidx),
                                                g->fwd.tagged ? kColMask : 0xffffffffu, g->n_local, s_src, s_dst,
                                                alpha); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_mask(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int64_t n, int64_t f,
                           void *Y, int64_t ld_y, gnn_dtype dt, gnn_dtype gdt, cudaStream_t s) {
    if (n * f == 0) return GNN_OK;
    const unsigned blocks = (unsigned)ceil_div(n * f, 256);
    if (gdt == GNN_F32 && dt == GNN_BF16)
        { gat_mask_kernel<float, __nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<const float *>(G), ld_g,
                                                                       static_cast<const __nv_bfloat16 *>(Hout), ld_h,
                                                                       n, f, static_cast<float *>(Y), ld_y); GNN_LAUNCHED(1); }
    else if (gdt == GNN_F32)
        { gat_mask_kernel<float, float><<<blocks, 256, 0, s>>>(static_cast<const float *>(G), ld_g,
                                                               static_cast<const float *>(Hout), ld_h, n, f,
                                                               static_cast<float *>(Y), ld_y); GNN_LAUNCHED(1); }
    else
        { gat_mask_kernel<__nv_bfloat16, __nv_bfloat16><<<blocks, 256, 0, s>>>(
            static_cast<const __nv_bfloat16 *>(G), ld_g, static_cast<const __nv_bfloat16 *>(Hout), ld_h, n, f,
            static_cast<__nv_bfloat16 *>(Y), ld_y); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_edge_backward(const gnn_graph *g, const float *s_src, const float *s_dst, const float *alpha,
                                    const void *dY, int64_t ld_y, const void *T, int64_t ld_t, int64_t f, float *dz,
                                    float *ds_dst, gnn_dtype dt, gnn_dtype gdt, cudaStream_t s) {
    if (g->n_local == 0) return GNN_OK;
    const uint32_t cm = g->fwd.tagged ? kColMask : 0xffffffffu;
    const uint32_t *ci = reinterpret_cast<const uint32_t *>(g->colidx);
    if (g->nnz > 0) {
        if (!g->erow) return GNN_EINVAL;
        constexpr int G = 8;
        const unsigned eb = (unsigned)std::min<int64_t>(ceil_div(g->nnz * G, 256), (int64_t)num_sms() * 32);
        if (gdt == GNN_F32 && dt == GNN_BF16)
            { gat_sddmm_kernel<float, __nv_bfloat16, G><<<eb, 256, 0, s>>>(
                g->erow, ci, cm, g->nnz, static_cast<const float *>(dY), ld_y,
                static_cast<const __nv_bfloat16 *>(T), ld_t, f, dz); GNN_LAUNCHED(1); }
        else if (gdt == GNN_F32)
            { gat_sddmm_kernel<float, float, G><<<eb, 256, 0, s>>>(g->erow, ci, cm, g->nnz,
                                                                    static_cast<const float *>(dY), ld_y,
                                                                    static_cast<const float *>(T), ld_t, f, dz); GNN_LAUNCHED(1); }
        else
            { gat_sddmm_kernel<__nv_bfloat16, __nv_bfloat16, G><<<eb, 256, 0, s>>>(
                g->erow, ci, cm, g->nnz, static_cast<const __nv_bfloat16 *>(dY), ld_y,
                static_cast<const __nv_bfloat16 *>(T), ld_t, f, dz); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(g->n_local * 32, 256), (int64_t)num_sms() * 16);
    { gat_softmax_backward_kernel<<<blocks, 256, 0, s>>>(g->rowptr, ci, cm, g->n_local, s_src, s_dst, alpha, dz,
                                                         ds_dst); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_entry_rows(const int32_t *rowptr, int64_t n_rows, int32_t *erow, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n_rows * 32, 256), (int64_t)num_sms() * 16);
    { entry_rows_kernel<<<blocks, 256, 0, s>>>(rowptr, n_rows, erow); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_transpose(const gnn_graph *g, const float *dz, const float *alpha, float *ds_src,
                                float *alphaT, cudaStream_t s) {
    const int64_t nT = g->n_local + g->n_halo;
    if (nT == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(nT * 32, 256), (int64_t)num_sms() * 16);
    { gat_transpose_kernel<<<blocks, 256, 0, s>>>(g->rowptrT, nT, g->t2b, dz, alpha, ds_src, alphaT); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

gnn_status launch_gat_rank1(void *dT, int64_t ld, int64_t n_total, int64_t n_local, int64_t f, const float *ds_src,
                            const float *ds_dst, const float *a_src, const float *a_dst, gnn_dtype gdt,
                            cudaStream_t s) {
    if (n_total * f == 0) return GNN_OK;
    const unsigned blocks = (unsigned)ceil_div(n_total * f, 256);
    if (gdt == GNN_BF16)
        { gat_rank1_kernel<__nv_bfloat16><<<blocks, 256, 0, s>>>(static_cast<__nv_bfloat16 *>(dT), ld, n_total,
                                                                 n_local, f, ds_src, ds_dst, a_src, a_dst); GNN_LAUNCHED(1); }
    else
        { gat_rank1_kernel<float><<<blocks, 256, 0, s>>>(static_cast<float *>(dT), ld, n_total, n_local, f, ds_src,
                                                         ds_dst, a_src, a_dst); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

// chunks of at least 256 rows, at most 4096 chunks
int64_t gat_colsum_chunks(int64_t n_rows) {
    return std::min<int64_t>(std::max<int64_t>(ceil_div(n_rows, 256), 1), 4096);
}

size_t gat_colsum_ws_floats(int64_t n_rows, int64_t f) { return (size_t)gat_colsum_chunks(n_rows) * (size_t)f; }

gnn_status launch_gat_colsum(const void *T, int64_t ld, int64_t n_rows, int64_t f, const float *w, float *out,
                             float *ws, gnn_dtype dt, cudaStream_t s) {
    if (f == 0) return GNN_OK;
    if (n_rows == 0) {
        GNN_CUDA_TRY(cudaMemsetAsync(out, 0, (size_t)f * sizeof(float), s));
        return GNN_OK;
    }
    const int64_t chunks = gat_colsum_chunks(n_rows);
    const int64_t rpc = ceil_div(n_rows, chunks);
    dim3 grid((unsigned)ceil_div(f, 128), (unsigned)chunks);
    if (dt == GNN_BF16)
        { gat_colsum_kernel<__nv_bfloat16><<<grid, 128, 0, s>>>(static_cast<const __nv_bfloat16 *>(T), ld, n_rows, f,
                                                                w, rpc, ws); GNN_LAUNCHED(1); }
    else
        { gat_colsum_kernel<float><<<grid, 128, 0, s>>>(static_cast<const float *>(T), ld, n_rows, f, w, rpc, ws); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    { gat_chunks_sum_kernel<<<(unsigned)ceil_div(f, 128), 128, 0, s>>>(ws, chunks, f, out); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace gnn
