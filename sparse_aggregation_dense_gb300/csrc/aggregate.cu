// aggregate.cu - the sparse aggregation (CSR SpMM) of the layer, forward and
// backward, with the degree normalisation fused in.
//
// Forward, GCN (CAGNET page, GNN section; Sylvie Alg. 1 matrix form):
//   Z[v] = dinv[v] * sum_{u in row v} dinv[u] * H[u]
// Forward, GraphSAGE mean (Sylvie page names GraphSAGE; textbook mean form):
//   Z[v] = [ H[v] | inv_cnt[v] * sum_{u in row v, u != v} H[u] ]
// Backward over the transpose CSR (A^T kept explicitly, CAGNET GNN section):
//   GCN:  dH[u] = dinv[u] * sum_{v in rowT u} dinv[v] * dZ[v]
//   SAGE: dH[u] = [u local] dZ_self[u] + sum_{v in rowT u, v != u} inv_cnt[v] * dZ_mean[v]
//
// Design (HBM-bound gather): one warp per work item.  An item is a whole light
// row (<= kHeavyNnz entries) or one kChunkNnz-entry chunk of a heavy row;
// chunks are scheduled first so hub rows spread over all SMs.  Lanes of a warp
// split the feature row into 16-byte vectors; a warp handles 32 / LPG entries
// at once (LPG lanes per entry) and keeps U entries' loads in flight.  Column
// ids and weights are loaded 32 at a time, coalesced, and broadcast by
// shuffles.  Accumulation is fp32.  A chunk writes an fp32 partial; a fix-up
// pass adds a heavy row's partials in chunk order, so the result does not
// depend on scheduling (no atomics).
#include "gnn_internal.cuh"

namespace gnn {

namespace {

__device__ __forceinline__ void unpack16(const float *, const uint4 &v, float *o) {
    o[0] = __uint_as_float(v.x);
    o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z);
    o[3] = __uint_as_float(v.w);
}
__device__ __forceinline__ void unpack16(const __nv_bfloat16 *, const uint4 &v, float *o) {
    o[0] = __uint_as_float(v.x << 16);
    o[1] = __uint_as_float(v.x & 0xffff0000u);
    o[2] = __uint_as_float(v.y << 16);
    o[3] = __uint_as_float(v.y & 0xffff0000u);
    o[4] = __uint_as_float(v.z << 16);
    o[5] = __uint_as_float(v.z & 0xffff0000u);
    o[6] = __uint_as_float(v.w << 16);
    o[7] = __uint_as_float(v.w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // a -> low half (first element)
    return *reinterpret_cast<uint32_t *>(&h);
}

// store EPV consecutive values (16 bytes) with columns >= f_left zeroed
__device__ __forceinline__ void store16(float *dst, const float *v, int f_left) {
    float4 o;
    o.x = 0 < f_left ? v[0] : 0.f;
    o.y = 1 < f_left ? v[1] : 0.f;
    o.z = 2 < f_left ? v[2] : 0.f;
    o.w = 3 < f_left ? v[3] : 0.f;
    *reinterpret_cast<float4 *>(dst) = o;
}
__device__ __forceinline__ void store16(__nv_bfloat16 *dst, const float *v, int f_left) {
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = k < f_left ? v[k] : 0.f;
    uint4 o;
    o.x = pack_bf16x2(w[0], w[1]);
    o.y = pack_bf16x2(w[2], w[3]);
    o.z = pack_bf16x2(w[4], w[5]);
    o.w = pack_bf16x2(w[6], w[7]);
    *reinterpret_cast<uint4 *>(dst) = o;
}
// store 4 consecutive values (fix-up granularity)
__device__ __forceinline__ void store4(float *dst, float4 v) { *reinterpret_cast<float4 *>(dst) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16 *dst, float4 v) {
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2 *>(dst) = o;
}
__device__ __forceinline__ float4 load4(const float *src) { return *reinterpret_cast<const float4 *>(src); }
__device__ __forceinline__ float4 load4(const __nv_bfloat16 *src) {
    uint2 v = *reinterpret_cast<const uint2 *>(src);
    return make_float4(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xffff0000u), __uint_as_float(v.y << 16),
                       __uint_as_float(v.y & 0xffff0000u));
}

template <typename T, int LPG, int VPT, int U>
__global__ void __launch_bounds__(256) aggregate_kernel(const AggParams p, const int32_t *__restrict__ chunk_row,
                                                        const int32_t *__restrict__ chunk_begin,
                                                        const int32_t *__restrict__ chunk_end, int64_t n_chunks,
                                                        float *__restrict__ partial, int64_t pld) {
    constexpr int EPV = 16 / (int)sizeof(T);
    constexpr int GROUPS = 32 / LPG;
    static_assert(GROUPS * U <= 32 && (32 % (GROUPS * U)) == 0, "step must divide the warp");
    const int lane = threadIdx.x & 31;
    const int g = lane / LPG, gl = lane % LPG;
    const int64_t item = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;

    int64_t r;
    int32_t b, e;
    bool is_chunk;
    if (item < n_chunks) {
        r = chunk_row[item];
        if (r >= p.n_rows) return;
        b = chunk_begin[item];
        e = chunk_end[item];
        is_chunk = true;
    } else {
        r = item - n_chunks;
        if (r >= p.n_rows) return;
        b = p.rowptr[r];
        e = p.rowptr[r + 1];
        if (e - b > kHeavyNnz) return;  // handled by its chunks and the fix-up
        is_chunk = false;
    }

    const T *__restrict__ X = static_cast<const T *>(p.X);
    const bool skip_self = p.mode != AGG_GCN;
    const bool col_weight = p.mode != AGG_SAGE_FWD;
    const int64_t f = p.f;

    float acc[VPT][EPV];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int k = 0; k < EPV; ++k) acc[v][k] = 0.f;

    for (int32_t base = b; base < e; base += 32) {
        const int n_here = min(32, e - base);
        int32_t c = 0;
        float w = 0.f;
        if (lane < n_here) {
            c = __ldg(p.colidx + base + lane);
            w = col_weight ? __ldg(p.colw + c) : 1.f;
            if (skip_self && (int64_t)c == r) w = 0.f;
        }
        for (int j = 0; j < n_here; j += GROUPS * U) {
            uint4 raw[U][VPT];
            float wu[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int jj = j + u * GROUPS + g;
                const int32_t cc = __shfl_sync(0xffffffffu, c, jj);
                const float ww = __shfl_sync(0xffffffffu, w, jj);
                const bool live = jj < n_here;
                wu[u] = live ? ww : 0.f;
                const T *row = X + (int64_t)cc * p.ldx;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int64_t col = (int64_t)(v * LPG + gl) * EPV;
                    if (live && col < f)
                        raw[u][v] = __ldg(reinterpret_cast<const uint4 *>(row + col));
                    else
                        raw[u][v] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float x[EPV];
                    unpack16(X, raw[u][v], x);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) acc[v][k] = fmaf(wu[u], x[k], acc[v][k]);
                }
        }
    }
    // reduce the GROUPS partial sums of the warp (fixed butterfly order)
#pragma unroll
    for (int off = LPG; off < 32; off <<= 1)
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
            for (int k = 0; k < EPV; ++k) acc[v][k] += __shfl_xor_sync(0xffffffffu, acc[v][k], off);
    if (g != 0) return;

    if (is_chunk) {
        float *dst = partial + item * pld;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int64_t col = (int64_t)(v * LPG + gl) * EPV;
            if (col < f) {
#pragma unroll
                for (int k = 0; k < EPV; k += 4)
                    *reinterpret_cast<float4 *>(dst + col + k) =
                        make_float4(acc[v][k], acc[v][k + 1], acc[v][k + 2], acc[v][k + 3]);
            }
        }
        return;
    }

    const float scale = p.mode == AGG_SAGE_BWD ? 1.f : __ldg(p.colw + r);
    T *out = static_cast<T *>(p.out) + r * p.ldo;
    const T *selfrow = nullptr;
    if (p.mode == AGG_SAGE_FWD) selfrow = X + r * p.ldx;
    if (p.mode == AGG_SAGE_BWD && r < p.n_self) selfrow = static_cast<const T *>(p.self) + r * p.ld_self;
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        const int64_t col = (int64_t)(v * LPG + gl) * EPV;
        if (col >= f) continue;
        float o[EPV];
#pragma unroll
        for (int k = 0; k < EPV; ++k) o[k] = acc[v][k] * scale;
        if (selfrow) {
            float s[EPV];
            unpack16(X, __ldg(reinterpret_cast<const uint4 *>(selfrow + col)), s);
            if (p.mode == AGG_SAGE_BWD) {
#pragma unroll
                for (int k = 0; k < EPV; ++k) o[k] += s[k];
            } else {
                store16(out + col, s, (int)(f - col));
            }
        }
        store16(out + p.out_off + col, o, (int)(f - col));
    }
}

template <typename T>
__global__ void __launch_bounds__(256) aggregate_fixup_kernel(const AggParams p, const int32_t *__restrict__ heavy_rows,
                                                              const int32_t *__restrict__ heavy_choff, int64_t n_heavy,
                                                              const float *__restrict__ partial, int64_t pld) {
    constexpr int EPV = 16 / (int)sizeof(T);
    const int lane = threadIdx.x & 31;
    const int64_t h = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (h >= n_heavy) return;
    const int64_t r = heavy_rows[h];
    if (r >= p.n_rows) return;
    const int32_t c0 = heavy_choff[h], c1 = heavy_choff[h + 1];
    const int64_t f = p.f;
    const int64_t fpad = (f + EPV - 1) / EPV * EPV;
    const float scale = p.mode == AGG_SAGE_BWD ? 1.f : __ldg(p.colw + r);
    const T *X = static_cast<const T *>(p.X);
    T *out = static_cast<T *>(p.out) + r * p.ldo;
    const T *selfrow = nullptr;
    if (p.mode == AGG_SAGE_FWD) selfrow = X + r * p.ldx;
    if (p.mode == AGG_SAGE_BWD && r < p.n_self) selfrow = static_cast<const T *>(p.self) + r * p.ld_self;
    for (int64_t col = (int64_t)lane * 4; col < fpad; col += 128) {
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
        if (col < f) {
            for (int32_t c = c0; c < c1; ++c) {
                float4 q = *reinterpret_cast<const float4 *>(partial + (int64_t)c * pld + col);
                s.x += q.x;
                s.y += q.y;
                s.z += q.z;
                s.w += q.w;
            }
        }
        float4 o = make_float4(s.x * scale, s.y * scale, s.z * scale, s.w * scale);
        if (selfrow) {
            float4 sv = col < f ? load4(selfrow + col) : make_float4(0.f, 0.f, 0.f, 0.f);
            if (p.mode == AGG_SAGE_BWD) {
                o.x += sv.x;
                o.y += sv.y;
                o.z += sv.z;
                o.w += sv.w;
            } else {
                if (col + 0 >= f) sv.x = 0.f;
                if (col + 1 >= f) sv.y = 0.f;
                if (col + 2 >= f) sv.z = 0.f;
                if (col + 3 >= f) sv.w = 0.f;
                store4(out + col, sv);
            }
        }
        if (col + 0 >= f) o.x = 0.f;
        if (col + 1 >= f) o.y = 0.f;
        if (col + 2 >= f) o.z = 0.f;
        if (col + 3 >= f) o.w = 0.f;
        store4(out + p.out_off + col, o);
    }
}

template <typename T, int LPG, int VPT, int U>
gnn_status launch_cfg(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    const int64_t items = sc.n_chunks + p.n_rows;
    if (items > 0) {
        const int64_t blocks = ceil_div(items * 32, 256);
        { aggregate_kernel<T, LPG, VPT, U><<<(unsigned)blocks, 256, 0, s>>>(p, sc.chunk_row, sc.chunk_begin,
                                                                           sc.chunk_end, sc.n_chunks, partial, pld); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    if (sc.n_heavy > 0) {
        const int64_t blocks = ceil_div(sc.n_heavy * 32, 256);
        { aggregate_fixup_kernel<T><<<(unsigned)blocks, 256, 0, s>>>(p, sc.heavy_rows, sc.heavy_choff, sc.n_heavy,
                                                                   partial, pld); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    return GNN_OK;
}

template <typename T>
gnn_status launch_typed(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    const int64_t bytes = p.f * (int64_t)sizeof(T);
    if (bytes <= 128) return launch_cfg<T, 8, 1, 8>(p, sc, partial, pld, s);
    if (bytes <= 256) return launch_cfg<T, 16, 1, 8>(p, sc, partial, pld, s);
    if (bytes <= 512) return launch_cfg<T, 32, 1, 8>(p, sc, partial, pld, s);
    if (bytes <= 1024) return launch_cfg<T, 32, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 1536) return launch_cfg<T, 32, 3, 2>(p, sc, partial, pld, s);
    if (bytes <= 2048) return launch_cfg<T, 32, 4, 2>(p, sc, partial, pld, s);
    if (bytes <= 2560) return launch_cfg<T, 32, 5, 2>(p, sc, partial, pld, s);
    if (bytes <= 3072) return launch_cfg<T, 32, 6, 1>(p, sc, partial, pld, s);
    if (bytes <= 4096) return launch_cfg<T, 32, 8, 1>(p, sc, partial, pld, s);
    return GNN_EUNSUPPORTED;
}

}  // namespace

size_t aggregate_partial_bytes(const Schedule &sc, int64_t f) {
    return (size_t)sc.n_chunks * (size_t)round_up(f, 8) * sizeof(float);
}

gnn_status launch_aggregate(const AggParams &p, const Schedule &sc, gnn_dtype dt, float *partial, cudaStream_t s) {
    if (p.n_rows == 0) return GNN_OK;
    const int64_t pld = round_up(p.f, 8);
    if (dt == GNN_BF16) return launch_typed<__nv_bfloat16>(p, sc, partial, pld, s);
    return launch_typed<float>(p, sc, partial, pld, s);
}

}  // namespace gnn
