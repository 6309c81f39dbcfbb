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
// The column factors live in per-entry weights built with the graph, so the
// kernel streams (column id, weight) pairs and gathers feature rows.
//
// Design (a gather bound by memory latency and DRAM traffic):
//  - one warp per work item: a whole light row (<= kHeavyNnz entries) or one
//    kChunkNnz-entry chunk of a heavy row; chunks are scheduled first so hub
//    rows spread over all SMs; a chunk writes an fp32 partial and a fix-up adds
//    a heavy row's partials in chunk order (deterministic, no atomics);
//  - lanes split a feature row into 16-byte vectors; LPG lanes serve one entry
//    and the warp serves 32 / LPG entries at once;
//  - the gathers are software-pipelined: U loads per lane group are always in
//    flight - each slot is consumed and immediately refilled with the entry U
//    slots ahead - and the next 32 column ids are loaded one batch ahead;
//  - L2 residency: column ids carry a hotness tier (access-count rank); rows
//    of the hottest tiers that fit a share of L2 are loaded with an evict_last
//    policy, the rest and the streamed ids / weights / outputs with evict_first.
#include <mutex>

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

__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// read-only 16-byte load with an L2 eviction policy
__device__ __forceinline__ uint4 ld_policy(const void *ptr, uint64_t pol) {
    uint4 v;
    asm("ld.global.nc.L2::cache_hint.v4.u32 {%0, %1, %2, %3}, [%4], %5;"
        : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
        : "l"(ptr), "l"(pol));
    return v;
}
// streamed 4-byte loads (no L1 allocation, evict_first in L2)
__device__ __forceinline__ uint32_t ld_stream_u32(const void *ptr, uint64_t pol) {
    uint32_t v;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.u32 %0, [%1], %2;" : "=r"(v) : "l"(ptr), "l"(pol));
    return v;
}
__device__ __forceinline__ void st_policy(void *ptr, const uint4 &v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(ptr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

// store EPV consecutive values (16 bytes) with columns >= f_left zeroed
__device__ __forceinline__ void store16(float *dst, const float *v, int f_left, uint64_t pol) {
    uint4 o;
    o.x = __float_as_uint(0 < f_left ? v[0] : 0.f);
    o.y = __float_as_uint(1 < f_left ? v[1] : 0.f);
    o.z = __float_as_uint(2 < f_left ? v[2] : 0.f);
    o.w = __float_as_uint(3 < f_left ? v[3] : 0.f);
    st_policy(dst, o, pol);
}
__device__ __forceinline__ void store16(__nv_bfloat16 *dst, const float *v, int f_left, uint64_t pol) {
    float w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = k < f_left ? v[k] : 0.f;
    uint4 o;
    o.x = pack_bf16x2(w[0], w[1]);
    o.y = pack_bf16x2(w[2], w[3]);
    o.z = pack_bf16x2(w[4], w[5]);
    o.w = pack_bf16x2(w[6], w[7]);
    st_policy(dst, o, pol);
}
// 4 consecutive values (fix-up granularity)
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

constexpr uint32_t kHotBit = 0x80000000u;

// one batch of 32 entries: lane i holds (column | hot bit, weight) of entry base + i
__device__ __forceinline__ void load_batch(const uint32_t *__restrict__ colidx, const float *__restrict__ wts,
                                           uint32_t colmask, int hot_tier, int32_t b, int32_t n, int32_t base,
                                           int lane, uint64_t pol_stream, uint32_t &c, float &w) {
    c = 0;
    w = 0.f;
    if (base + lane < n) {
        const uint32_t raw = ld_stream_u32(colidx + b + base + lane, pol_stream);
        w = __uint_as_float(ld_stream_u32(wts + b + base + lane, pol_stream));
        const uint32_t col = raw & colmask;
        const int tier = colmask == kColMask ? (int)(raw >> kTierShift) : 0;
        c = col | (tier <= hot_tier ? kHotBit : 0u);
    }
}

// cp.async of 16 bytes into shared memory with an L2 eviction policy
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc, uint64_t pol) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
                 "l"(gsrc), "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Shared memory of one warp: a ring of D steps; a step holds, for every lane,
// VPT 16-byte vectors of the row its lane group gathers and the entry weight.
template <int VPT, int D>
struct WarpRing {
    static constexpr int kVecs = D * VPT * 32;  // uint4 per warp
    static constexpr int kBytes = kVecs * 16 + D * 32 * 4;
};

// One work item: a whole light row or one chunk of a heavy row.
struct Item {
    int64_t r;
    int32_t b, e;
    bool chunk;
    bool skip;  // no work for this warp (heavy row in the row range, or past n_rows)
};

__device__ __forceinline__ Item load_item(int64_t it, int64_t n_chunks, const int32_t *__restrict__ chunk_row,
                                          const int32_t *__restrict__ chunk_begin,
                                          const int32_t *__restrict__ chunk_end, const int32_t *__restrict__ rowptr,
                                          int64_t n_rows) {
    Item x;
    if (it < n_chunks) {
        x.r = chunk_row[it];
        x.b = chunk_begin[it];
        x.e = chunk_end[it];
        x.chunk = true;
        x.skip = x.r >= n_rows;
    } else {
        x.r = it - n_chunks;
        x.chunk = false;
        if (x.r < n_rows) {
            x.b = rowptr[x.r];
            x.e = rowptr[x.r + 1];
            x.skip = x.e - x.b > kHeavyNnz;  // handled by its chunks and the fix-up
        } else {
            x.b = x.e = 0;
            x.skip = true;
        }
    }
    return x;
}

// Persistent warps: warp w of W handles items w, w + W, w + 2W, ... as one
// continuous stream of entries.  The issue side runs D steps ahead of the
// consume side (a step: every lane group gathers one entry into the warp's
// shared-memory ring with cp.async); the consume side accumulates a step and
// finishes an item (writes its row or partial) when its steps are done, so
// the gather pipeline never drains between rows.
template <typename T, int LPG, int VPT, int D, int MINB>
__global__ void __launch_bounds__(256, MINB)
    aggregate_kernel(const AggParams p, const int32_t *__restrict__ chunk_row, const int32_t *__restrict__ chunk_begin,
                     const int32_t *__restrict__ chunk_end, int64_t n_chunks, float *__restrict__ partial,
                     int64_t pld) {
    constexpr int EPV = 16 / (int)sizeof(T);
    constexpr int GROUPS = 32 / LPG;
    static_assert(D >= 1 && D <= 32, "ring depth");
    extern __shared__ uint4 smem_ring[];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int g = lane / LPG, gl = lane % LPG;
    uint4 *ring = smem_ring + wib * WarpRing<VPT, D>::kVecs;
    float *wring = reinterpret_cast<float *>(smem_ring + 8 * WarpRing<VPT, D>::kVecs) + wib * D * 32;

    const int64_t W = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + wib;
    const int64_t n_items = n_chunks + p.n_rows;
    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_stream = policy_evict_first();
    const T *__restrict__ X = static_cast<const T *>(p.X);
    const int64_t f = p.f, ldx = p.ldx;
    const uint32_t *__restrict__ colidx = p.colidx;
    const float *__restrict__ wts = p.wts;
    const uint32_t colmask = p.colmask;
    const int hot_tier = p.hot_tier;
    const int32_t *__restrict__ rowptr = p.rowptr;
    const int64_t n_rows = p.n_rows;

    // ---- issue side: item it_i, next entry pos_i, column-id batches ----
    int64_t it_i = w0;
    Item cur_i = it_i < n_items ? load_item(it_i, n_chunks, chunk_row, chunk_begin, chunk_end, rowptr, n_rows) : Item{0, 0, 0, false, true};
    int32_t pos_i = 0, bbase = 0;
    uint32_t c_cur = 0, c_next = 0;
    float w_cur = 0.f, w_next = 0.f;
    bool issue_live = it_i < n_items;
    // advance the issue side to an item with entries (or the end); load its batches
    auto settle_issue = [&]() {
        while (issue_live && (cur_i.skip || pos_i >= cur_i.e - cur_i.b)) {
            it_i += W;
            if (it_i >= n_items) {
                issue_live = false;
                break;
            }
            cur_i = load_item(it_i, n_chunks, chunk_row, chunk_begin, chunk_end, rowptr, n_rows);
            pos_i = 0;
            if (!cur_i.skip && cur_i.e > cur_i.b) {
                bbase = 0;
                load_batch(colidx, wts, colmask, hot_tier, cur_i.b, cur_i.e - cur_i.b, 0, lane, pol_stream, c_cur,
                           w_cur);
                load_batch(colidx, wts, colmask, hot_tier, cur_i.b, cur_i.e - cur_i.b, 32, lane, pol_stream,
                           c_next, w_next);
            }
        }
    };
    if (issue_live && !cur_i.skip && cur_i.e > cur_i.b) {
        load_batch(colidx, wts, colmask, hot_tier, cur_i.b, cur_i.e - cur_i.b, 0, lane, pol_stream, c_cur, w_cur);
        load_batch(colidx, wts, colmask, hot_tier, cur_i.b, cur_i.e - cur_i.b, 32, lane, pol_stream, c_next,
                   w_next);
    }
    settle_issue();
    int64_t s_issue = 0;  // steps issued (ring slot = s % D)
    auto issue_step = [&]() {
        if (!issue_live) return;
        const int32_t n = cur_i.e - cur_i.b;
        if (pos_i >= bbase + 32) {
            bbase += 32;
            c_cur = c_next;
            w_cur = w_next;
            load_batch(colidx, wts, colmask, hot_tier, cur_i.b, n, bbase + 32, lane, pol_stream, c_next, w_next);
        }
        const int src = pos_i - bbase + g;
        const uint32_t cc = __shfl_sync(0xffffffffu, c_cur, src);
        const float ww = __shfl_sync(0xffffffffu, w_cur, src);
        const bool live = pos_i + g < n;
        const int slot = (int)(s_issue % D);
        uint4 *dst = ring + slot * VPT * 32 + lane;
        wring[slot * 32 + lane] = live ? ww : 0.f;
        const T *row = X + (int64_t)(cc & ~kHotBit) * ldx;
        const uint64_t pol = (cc & kHotBit) ? pol_keep : pol_stream;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int64_t col = (int64_t)(v * LPG + gl) * EPV;
            if (col < f) {
                if (live)
                    cp_async16(dst + v * 32, row + col, pol);
                else
                    dst[v * 32] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        ++s_issue;
        pos_i += GROUPS;
        settle_issue();
    };

    // ---- consume side ----
    const uint64_t pol_out = pol_stream;
    float acc[VPT][EPV];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int k = 0; k < EPV; ++k) acc[v][k] = 0.f;

    // finish item x (id it): reduce the lane groups and write the row or the partial
    auto finish = [&](const Item &x, int64_t it) {
#pragma unroll
        for (int off = LPG; off < 32; off <<= 1)
#pragma unroll
            for (int v = 0; v < VPT; ++v)
#pragma unroll
                for (int k = 0; k < EPV; ++k) acc[v][k] += __shfl_xor_sync(0xffffffffu, acc[v][k], off);
        if (g == 0) {
            if (x.chunk) {
                float *dst = partial + it * pld;
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
            } else {
                const float scale = p.rowscale ? __ldg(p.rowscale + x.r) : 1.f;
                T *out = static_cast<T *>(p.out) + x.r * p.ldo;
                const T *selfrow = nullptr;
                if (p.self_mode == SELF_COPY) selfrow = X + x.r * ldx;
                if (p.self_mode == SELF_ADD && x.r < p.n_self) selfrow = static_cast<const T *>(p.self) + x.r * p.ld_self;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int64_t col = (int64_t)(v * LPG + gl) * EPV;
                    if (col >= f) continue;
                    float o[EPV];
#pragma unroll
                    for (int k = 0; k < EPV; ++k) o[k] = acc[v][k] * scale;
                    if (selfrow) {
                        float sv[EPV];
                        unpack16(X, __ldg(reinterpret_cast<const uint4 *>(selfrow + col)), sv);
                        if (p.self_mode == SELF_ADD) {
#pragma unroll
                            for (int k = 0; k < EPV; ++k) o[k] += sv[k];
                        } else {
                            store16(out + col, sv, (int)(f - col), pol_out);
                        }
                    }
                    store16(out + p.out_off + col, o, (int)(f - col), pol_out);
                }
            }
        }
#pragma unroll
        for (int v = 0; v < VPT; ++v)
#pragma unroll
            for (int k = 0; k < EPV; ++k) acc[v][k] = 0.f;
    };

    // prologue: D steps in flight
#pragma unroll 1
    for (int d = 0; d < D; ++d) {
        issue_step();
        cp_async_commit();
    }
    int64_t it_c = w0;
    int64_t s_cons = 0;
#pragma unroll 1
    while (it_c < n_items) {
        const Item x = load_item(it_c, n_chunks, chunk_row, chunk_begin, chunk_end, rowptr, n_rows);
        if (!x.skip) {
            const int32_t steps = (x.e - x.b + GROUPS - 1) / GROUPS;
#pragma unroll 1
            for (int32_t t = 0; t < steps; ++t) {
                cp_async_wait<D - 1>();
                const int slot = (int)(s_cons % D);
                const float w = wring[slot * 32 + lane];
                const uint4 *src = ring + slot * VPT * 32 + lane;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    float xv[EPV];
                    unpack16(X, src[v * 32], xv);
#pragma unroll
                    for (int k = 0; k < EPV; ++k) acc[v][k] = fmaf(w, xv[k], acc[v][k]);
                }
                ++s_cons;
                issue_step();
                cp_async_commit();
            }
            finish(x, it_c);
        }
        it_c += W;
    }
    cp_async_wait<0>();
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
    const float scale = p.rowscale ? __ldg(p.rowscale + r) : 1.f;
    const T *X = static_cast<const T *>(p.X);
    T *out = static_cast<T *>(p.out) + r * p.ldo;
    const T *selfrow = nullptr;
    if (p.self_mode == SELF_COPY) selfrow = X + r * p.ldx;
    if (p.self_mode == SELF_ADD && r < p.n_self) selfrow = static_cast<const T *>(p.self) + r * p.ld_self;
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
            if (p.self_mode == SELF_ADD) {
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

template <typename T, int LPG, int VPT, int D, int MINB>
gnn_status launch_cfg(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    const int64_t items = sc.n_chunks + p.n_rows;
    if (items > 0) {
        const int smem = 8 * WarpRing<VPT, D>::kBytes;
        auto kern = aggregate_kernel<T, LPG, VPT, D, MINB>;
        GNN_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        // persistent warps: as many blocks as fit on the GPU at once
        int per_sm = 0;
        GNN_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, smem));
        if (per_sm < 1) per_sm = 1;
        int64_t blocks = (int64_t)num_sms() * per_sm;
        if (blocks > ceil_div(items, 8)) blocks = ceil_div(items, 8);
        { kern<<<(unsigned)blocks, 256, smem, s>>>(p, sc.chunk_row, sc.chunk_begin, sc.chunk_end, sc.n_chunks,
                                                    partial, pld); GNN_LAUNCHED(1); }
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
    // steps in flight per warp D: D * 512 * VPT bytes of gathered rows per warp;
    // shared memory (8 warps per block) then sets the blocks per SM (MINB)
    const int64_t bytes = p.f * (int64_t)sizeof(T);
    if (bytes <= 128) return launch_cfg<T, 8, 1, 8, 5>(p, sc, partial, pld, s);
    if (bytes <= 256) return launch_cfg<T, 16, 1, 8, 5>(p, sc, partial, pld, s);
    if (bytes <= 512) return launch_cfg<T, 32, 1, 8, 5>(p, sc, partial, pld, s);
    if (bytes <= 1024) return launch_cfg<T, 32, 2, 4, 4>(p, sc, partial, pld, s);
    if (bytes <= 1536) return launch_cfg<T, 32, 3, 3, 4>(p, sc, partial, pld, s);
    if (bytes <= 2048) return launch_cfg<T, 32, 4, 2, 3>(p, sc, partial, pld, s);
    if (bytes <= 2560) return launch_cfg<T, 32, 5, 2, 3>(p, sc, partial, pld, s);
    if (bytes <= 3072) return launch_cfg<T, 32, 6, 2, 2>(p, sc, partial, pld, s);
    if (bytes <= 4096) return launch_cfg<T, 32, 8, 1, 2>(p, sc, partial, pld, s);
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

// ---------------------------------------------------------------------------
// Forward aggregation that allocates nothing (gnn_aggregate_forward_noalloc).
//
// The only scratch the aggregation needs is the fp32 partial of each chunk of a
// heavy row.  This entry point keeps those partials in the fixed array below
// instead of the graph's growing workspace, so a call never allocates device
// memory.  The array is part of the library image: every GPU that loads
// libgnn holds it until the process exits.  Every chunk overwrites its own
// partial before the fix-up reads it, so nothing in the array has to start at
// zero; calls that overlap on the GPU (two streams, or two threads) share the
// array and race.
// ---------------------------------------------------------------------------
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB
constexpr size_t kNoAllocScratchFloats = kNoAllocScratchBytes / sizeof(float);
constexpr int kMaxDevices = 64;

__device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

std::mutex g_noalloc_mutex;
float *g_noalloc_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the host-side name of the array is not a device address).
gnn_status noalloc_scratch(float **out) {
    int dev = 0;
    GNN_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return GNN_EUNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        GNN_CUDA_TRY(cudaGetSymbolAddress(&p, g_noalloc_scratch));
        g_noalloc_addr[dev] = static_cast<float *>(p);
    }
    *out = g_noalloc_addr[dev];
    return GNN_OK;
}

bool rows_ok(const void *p, int64_t rows, int64_t ld, int64_t f, gnn_dtype t) {
    if (rows == 0) return true;
    if (!p || (reinterpret_cast<uintptr_t>(p) & 15u)) return false;
    return ld >= f && ld % elems_per_16b(t) == 0;
}

}  // namespace

}  // namespace gnn

extern "C" gnn_status gnn_aggregate_forward_noalloc(const gnn_graph *g, const void *H, int64_t ld_h, int64_t f,
                                                    void *Z, int64_t ld_z, gnn_dtype dtype, void *stream) {
    using namespace gnn;
    if (!g || (dtype != GNN_F32 && dtype != GNN_BF16) || f <= 0) return GNN_EINVAL;
    const bool sage = g->agg == GNN_AGG_SAGE_MEAN;
    const int64_t nL = g->n_local, nT = g->n_local + g->n_halo;
    const int64_t half = gnn_sage_half_offset(f, dtype);
    const int64_t Kp = sage ? 2 * half : f;
    if (!rows_ok(H, nT, ld_h, f, dtype) || !rows_ok(Z, nL, ld_z, Kp, dtype)) return GNN_EINVAL;
    if (f * elem_size(dtype) > 4096) return GNN_EUNSUPPORTED;
    if (aggregate_partial_bytes(g->fwd, f) > kNoAllocScratchBytes) return GNN_EUNSUPPORTED;
    if (nL == 0) return GNN_OK;
    float *scratch = nullptr;
    gnn_status st = noalloc_scratch(&scratch);
    if (st != GNN_OK) return st;
    AggParams p{};
    p.rowptr = g->rowptr;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidx);
    p.wts = g->wfwd;
    p.rowscale = g->colw;
    p.n_rows = nL;
    p.colmask = g->fwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->fwd, round_up(f * elem_size(dtype), 32));
    p.X = H;
    p.ldx = ld_h;
    p.f = f;
    p.self_mode = sage ? SELF_COPY : SELF_NONE;
    p.out = Z;
    p.ldo = ld_z;
    p.out_off = sage ? half : 0;
    return launch_aggregate(p, g->fwd, dtype, scratch, static_cast<cudaStream_t>(stream));
}

