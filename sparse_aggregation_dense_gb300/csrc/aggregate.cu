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
//  - work items: row groups (runs of consecutive light rows, <= kHeavyNnz
//    entries each, whose entries form one range) and kChunkNnz-entry chunks of
//    heavy rows; chunks are scheduled first so hub rows spread over all SMs; a
//    chunk writes an fp32 partial and a fix-up adds a heavy row's partials in
//    chunk order (deterministic, no atomics);
//  - a warp streams an item's entries in batches that may span rows; the 32
//    lanes split a feature row into VW-byte pieces (VPT boxes of 32 * VW bytes)
//    and walk the batch entry by entry, writing each row out where it ends;
//  - the gathers are TMA gathers of four rows (tile::gather4) into a per-warp
//    shared-memory ring of NS slots (a slot: BE entries), completed on one
//    mbarrier per slot; the warp consumes one slot while the next NS - 1 are
//    in flight, and the next 64 column ids sit in registers, fetched ahead;
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

// TMA gather of four rows r0..r3 of the tensor behind `map`, columns [x, x + box):
// the rows land one after another at smem_dst; completion is counted in bytes
// on the mbarrier
__device__ __forceinline__ void tma_gather4(void *smem_dst, const CUtensorMap *map, int32_t x, int32_t r0, int32_t r1,
                                            int32_t r2, int32_t r3, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4, %5, %6}], [%7], %8;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst))),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(r0), "r"(r1), "r"(r2), "r"(r3),
        "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void bar_init(uint64_t *bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                 : "memory");
}
__device__ __forceinline__ void bar_expect(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                     static_cast<uint32_t>(__cvta_generic_to_shared(bar))),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar))), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait: false after ~2 s
__device__ __forceinline__ bool bar_wait(uint64_t *bar, uint32_t parity) {
    if (bar_try(bar, parity)) return true;
    uint64_t t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    for (;;) {
        if (bar_try(bar, parity)) return true;
        uint64_t t;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
        if (t - t0 > 2000000000ull) return false;
    }
}

// Shared memory of one warp: NS slots of BE gathered rows (R bytes each), the
// entries' weights (each stored twice, as a packed-FMA operand) and one
// mbarrier per slot.  A slot is laid out box-major:
// box v (bytes [v * LPG * 16, (v + 1) * LPG * 16) of every row) holds the BE
// rows one after another, as the TMA gathers deliver them.
template <int R, int BE, int NS>
struct BulkRing {
    static constexpr int kRowBytes = NS * BE * R;
    static constexpr int kBytes = kRowBytes + NS * BE * 8 + NS * 8;  // rows, weight pairs, mbarriers
};

// One work item: a row group (consecutive light rows, one entry range) or one
// chunk of a heavy row.  Rows at or past n_rows (halo rows of a transpose whose
// gradient is not wanted) are cut off.
struct Item {
    int32_t r0, r1;  // rows [r0, r1); a chunk: its row, r0 + 1
    int32_t b, e;    // entries [b, e)
    bool chunk;
    bool skip;       // nothing to compute (all its rows at or past n_rows)
};

__device__ __forceinline__ Item load_item(int64_t it, int64_t n_chunks, const int32_t *__restrict__ chunk_row,
                                          const int32_t *__restrict__ chunk_begin,
                                          const int32_t *__restrict__ chunk_end, const int32_t *__restrict__ group_r0,
                                          const int32_t *__restrict__ group_r1, const int32_t *__restrict__ rowptr,
                                          int64_t n_rows) {
    Item x;
    if (it < n_chunks) {
        x.r0 = chunk_row[it];
        x.r1 = x.r0 + 1;
        x.b = chunk_begin[it];
        x.e = chunk_end[it];
        x.chunk = true;
        x.skip = x.r0 >= n_rows;
    } else {
        const int64_t gi = it - n_chunks;
        x.r0 = group_r0[gi];
        x.r1 = group_r1[gi];
        if (x.r1 > n_rows) x.r1 = (int32_t)n_rows;
        x.chunk = false;
        x.skip = x.r0 >= x.r1;
        x.b = x.skip ? 0 : rowptr[x.r0];
        x.e = x.skip ? 0 : rowptr[x.r1];
    }
    return x;
}

// this lane's VW bytes of a gathered row in shared memory, as 32-bit words
template <int VW>
__device__ __forceinline__ void lds_words(const uint8_t *p, uint32_t (&w)[VW / 4]) {
    if constexpr (VW == 16) {
        const uint4 q = *reinterpret_cast<const uint4 *>(p);
        w[0] = q.x;
        w[1] = q.y;
        w[2] = q.z;
        w[3] = q.w;
    } else if constexpr (VW == 8) {
        const uint2 q = *reinterpret_cast<const uint2 *>(p);
        w[0] = q.x;
        w[1] = q.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    }
}

// Accumulators and weights live as pairs of fp32 in one 64-bit register (low
// half = the even column), the operand form of the packed FMA fma.rn.f32x2;
// a bf16 pair is widened by placing each half in the top 16 bits of an fp32.
template <typename T, int VW>
struct Lane {
    static constexpr int kWords = VW / 4;                                       // 32-bit words per piece
    static constexpr int kPairs = sizeof(T) == 2 ? kWords : (kWords + 1) / 2;  // fp32 pairs per piece
};

// a += ww * (the values in words q), one packed FMA per pair
template <typename T, int VW>
__device__ __forceinline__ void fma_piece(unsigned long long (&a)[Lane<T, VW>::kPairs], const uint32_t (&q)[VW / 4],
                                          unsigned long long ww) {
    if constexpr (sizeof(T) == 2) {
#pragma unroll
        for (int k = 0; k < VW / 4; ++k)
            asm("{\n\t.reg .b32 lo, hi;\n\t.reg .b64 x;\n\t"
                "shl.b32 lo, %1, 16;\n\tand.b32 hi, %1, 0xffff0000;\n\tmov.b64 x, {lo, hi};\n\t"
                "fma.rn.f32x2 %0, x, %2, %0;\n\t}"
                : "+l"(a[k])
                : "r"(q[k]), "l"(ww));
    } else if constexpr (VW >= 8) {
#pragma unroll
        for (int k = 0; k < VW / 8; ++k)
            asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%1, %2};\n\tfma.rn.f32x2 %0, x, %3, %0;\n\t}"
                : "+l"(a[k])
                : "r"(q[2 * k]), "r"(q[2 * k + 1]), "l"(ww));
    } else {
        asm("{\n\t.reg .b64 x;\n\tmov.b64 x, {%1, 0};\n\tfma.rn.f32x2 %0, x, %2, %0;\n\t}"
            : "+l"(a[0])
            : "r"(q[0]), "l"(ww));
    }
}

// acc += w * (this lane's VW-byte pieces of one gathered row); `row` points at
// the lane's piece in box 0, box v sits v * BE * 32 * VW bytes further; ww
// holds the weight twice
template <typename T, int VW, int VPT, int BE>
__device__ __forceinline__ void accumulate_entry(unsigned long long (&acc)[VPT][Lane<T, VW>::kPairs],
                                                 const uint8_t *row, unsigned long long ww) {
#pragma unroll
    for (int v = 0; v < VPT; ++v) {
        uint32_t q[VW / 4];
        lds_words<VW>(row + v * (BE * 32 * VW), q);
        fma_piece<T, VW>(acc[v], q, ww);
    }
}

// the VW / sizeof(T) fp32 values held in a piece's pairs
template <typename T, int VW>
__device__ __forceinline__ void pairs_to_vals(const unsigned long long (&a)[Lane<T, VW>::kPairs],
                                              float (&v)[VW / sizeof(T)]) {
#pragma unroll
    for (int k = 0; k < (int)(VW / sizeof(T)); ++k)
        v[k] = __uint_as_float((uint32_t)(a[k / 2] >> (32 * (k & 1))));
}

// global <-> registers for this lane's VW bytes (VW / sizeof(T) values)
template <int VW>
__device__ __forceinline__ void ldg_words(const void *p, uint32_t (&w)[VW / 4]) {
    if constexpr (VW == 16) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(p));
        w[0] = q.x;
        w[1] = q.y;
        w[2] = q.z;
        w[3] = q.w;
    } else if constexpr (VW == 8) {
        const uint2 q = __ldg(reinterpret_cast<const uint2 *>(p));
        w[0] = q.x;
        w[1] = q.y;
    } else {
        w[0] = __ldg(reinterpret_cast<const uint32_t *>(p));
    }
}
template <int VW>
__device__ __forceinline__ void stg_words(void *p, const uint32_t (&w)[VW / 4], uint64_t pol) {
    if constexpr (VW == 16) {
        asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(w[0]), "r"(w[1]),
                     "r"(w[2]), "r"(w[3]), "l"(pol)
                     : "memory");
    } else if constexpr (VW == 8) {
        asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(w[0]), "r"(w[1]), "l"(pol)
                     : "memory");
    } else {
        asm volatile("st.global.L2::cache_hint.u32 [%0], %1, %2;" ::"l"(p), "r"(w[0]), "l"(pol) : "memory");
    }
}
template <typename T, int VW>
__device__ __forceinline__ void words_to_vals(const uint32_t (&w)[VW / 4], float (&v)[VW / sizeof(T)]) {
#pragma unroll
    for (int k = 0; k < VW / 4; ++k) {
        if constexpr (sizeof(T) == 2) {
            v[2 * k] = __uint_as_float(w[k] << 16);
            v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
        } else {
            v[k] = __uint_as_float(w[k]);
        }
    }
}
// values at or past f_left are stored as 0
template <typename T, int VW>
__device__ __forceinline__ void vals_to_words(const float (&v)[VW / sizeof(T)], int f_left, uint32_t (&w)[VW / 4]) {
#pragma unroll
    for (int k = 0; k < VW / 4; ++k) {
        if constexpr (sizeof(T) == 2) {
            w[k] = pack_bf16x2(2 * k < f_left ? v[2 * k] : 0.f, 2 * k + 1 < f_left ? v[2 * k + 1] : 0.f);
        } else {
            w[k] = __float_as_uint(k < f_left ? v[k] : 0.f);
        }
    }
}

// Advance `it` by W to the next item that has entries to gather (or the end).
__device__ __forceinline__ bool next_work_item(int64_t &it, Item &x, int64_t W, int64_t n_items, int64_t n_chunks,
                                               const int32_t *__restrict__ chunk_row,
                                               const int32_t *__restrict__ chunk_begin,
                                               const int32_t *__restrict__ chunk_end,
                                               const int32_t *__restrict__ group_r0,
                                               const int32_t *__restrict__ group_r1,
                                               const int32_t *__restrict__ rowptr, int64_t n_rows) {
    for (;;) {
        it += W;
        if (it >= n_items) return false;
        x = load_item(it, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0, group_r1, rowptr, n_rows);
        if (!x.skip && x.e > x.b) return true;
    }
}

// lane j: column id (tier bits kept) and weight of entry base + j of item x
__device__ __forceinline__ void fetch_window(const Item &x, bool valid, int32_t base,
                                             const uint32_t *__restrict__ colidx, const float *__restrict__ wts,
                                             int lane, uint64_t pol, uint32_t &c, float &w) {
    c = 0;
    w = 0.f;
    if (valid && base + lane < x.e - x.b) {
        c = ld_stream_u32(colidx + x.b + base + lane, pol);
        w = __uint_as_float(ld_stream_u32(wts + x.b + base + lane, pol));
    }
}

// Persistent warps: warp w of W handles items w, w + W, ... as one stream of
// batches (a batch: up to BE consecutive entries of one item, which may span
// several rows of a row group).  Lane j of a batch holds entry j's column id
// and weight; every fourth lane gathers its four entries' rows with one TMA
// gather per box into the warp's slot (a short last group repeats its last
// row, weighted 0).  The consume side, NS - 1 batches behind, walks the
// batch's entries in order: it accumulates runs of entries of one row and
// writes a row out (or, for a chunk of a heavy row, its fp32 partial) where
// the row ends.  Each lane owns VW bytes of each of the VPT boxes of a row.
template <typename T, int VW, int VPT, int BE, int NS, int WPC>
__global__ void __launch_bounds__(WPC * 32)
    aggregate_kernel(const AggParams p, const __grid_constant__ CUtensorMap xmap, const int32_t *__restrict__ chunk_row,
                     const int32_t *__restrict__ chunk_begin, const int32_t *__restrict__ chunk_end, int64_t n_chunks,
                     const int32_t *__restrict__ group_r0, const int32_t *__restrict__ group_r1, int64_t n_groups,
                     float *__restrict__ partial, int64_t pld) {
    constexpr int EPL = VW / (int)sizeof(T);  // values of a row per lane per box
    constexpr int BOX = 32 * VW;              // bytes of one gathered box of a row
    constexpr int R = VPT * BOX;
    static_assert(VW == 4 || VW == 8 || VW == 16, "lane piece of 4, 8 or 16 bytes");
    static_assert(BE <= 32 && BE % 4 == 0 && 32 % BE == 0, "whole groups of four entries inside one id window");
    static_assert(BOX % 128 == 0, "TMA destinations stay 128-byte aligned");
    using Ring = BulkRing<R, BE, NS>;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    // TMA destinations must be 128-byte aligned: round the dynamic base up
    // (the launch adds 128 bytes for this)
    uint8_t *smem_bulk = smem_raw + ((128u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    uint8_t *rows = smem_bulk + wib * Ring::kRowBytes;
    unsigned long long *wring =
        reinterpret_cast<unsigned long long *>(smem_bulk + WPC * Ring::kRowBytes) + wib * NS * BE;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem_bulk + WPC * Ring::kRowBytes + WPC * NS * BE * 8) + wib * NS;

    const int64_t W = (int64_t)gridDim.x * WPC;
    const int64_t w0 = (int64_t)blockIdx.x * WPC + wib;
    const int64_t n_items = n_chunks + n_groups;
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

    if (lane == 0)
        for (int s = 0; s < NS; ++s) bar_init(&bars[s]);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncwarp();

    // ---- issue side ----
    // The column ids and weights of the next 64 entries of the current item
    // sit in registers (lane j holds entry wb + j in (ic0, iw0) and wb + 32 + j
    // in (ic1, iw1)); the next item with its first 32 ids is fetched one item
    // ahead.  Issuing a batch therefore never waits on an index load.
    Item ci = Item{0, 0, 0, 0, false, true}, ni = Item{0, 0, 0, 0, false, true};
    int64_t it_i = w0 - W;
    bool more = next_work_item(it_i, ci, W, n_items, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0, group_r1,
                               rowptr, n_rows);
    int64_t it_n = it_i;
    bool nmore = more && next_work_item(it_n, ni, W, n_items, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0,
                                        group_r1, rowptr, n_rows);
    int32_t off_i = 0, wb = 0;
    uint32_t ic0, ic1, nc0;
    float iw0, iw1, nw0;
    fetch_window(ci, more, 0, colidx, wts, lane, pol_stream, ic0, iw0);
    fetch_window(ci, more, 32, colidx, wts, lane, pol_stream, ic1, iw1);
    fetch_window(ni, nmore, 0, colidx, wts, lane, pol_stream, nc0, nw0);
    uint32_t s_i = 0;
    bool ok = true;

#define GNN_ISSUE_BATCH()                                                                                   \
    do {                                                                                                    \
        if (!more) break;                                                                                   \
        const int slot = (int)(s_i % NS);                                                                   \
        const int32_t n_ci = ci.e - ci.b;                                                                   \
        const int32_t left = n_ci - off_i;                                                                  \
        const int cnt = left < BE ? left : BE;                                                              \
        /* lanes past the batch repeat its last entry: a valid row, weight 0 */                           \
        const int src = (off_i - wb + (lane < cnt ? lane : cnt - 1)) & 31;                                  \
        const uint32_t raw = __shfl_sync(0xffffffffu, ic0, src);                                            \
        const float wv = __shfl_sync(0xffffffffu, iw0, src);                                                \
        if (lane < BE) {                                                                                    \
            const uint32_t wb32 = __float_as_uint(lane < cnt ? wv : 0.f);                                   \
            wring[slot * BE + lane] = ((unsigned long long)wb32 << 32) | wb32;                              \
        }                                                                                                   \
        const int32_t col = (int32_t)(raw & colmask);                                                       \
        const int tier = colmask == kColMask ? (int)(raw >> kTierShift) : 0;                                \
        const uint32_t hot = __ballot_sync(0xffffffffu, lane < cnt && tier <= hot_tier);                    \
        const int32_t c1 = __shfl_down_sync(0xffffffffu, col, 1);                                           \
        const int32_t c2 = __shfl_down_sync(0xffffffffu, col, 2);                                           \
        const int32_t c3 = __shfl_down_sync(0xffffffffu, col, 3);                                           \
        const int ngr = (cnt + 3) >> 2;                                                                     \
        if (lane == 0) bar_expect(&bars[slot], (uint32_t)(ngr * VPT * 4 * BOX));                            \
        __syncwarp();                                                                                       \
        if ((lane & 3) == 0 && lane < 4 * ngr) {                                                            \
            /* keep the group in L2 when most of its rows are hot */                                        \
            const uint64_t pol = __popc((hot >> lane) & 0xfu) >= 2 ? pol_keep : pol_stream;                 \
            uint8_t *dst = rows + slot * BE * R + lane * BOX;                                               \
            _Pragma("unroll") for (int v = 0; v < VPT; ++v)                                                \
                tma_gather4(dst + v * BE * BOX, &xmap, v * (BOX / (int)sizeof(T)), col, c1, c2, c3,         \
                            &bars[slot], pol);                                                              \
        }                                                                                                   \
        ++s_i;                                                                                              \
        off_i += BE;                                                                                        \
        if (off_i >= n_ci) {                                                                                \
            more = nmore;                                                                                   \
            if (more) {                                                                                     \
                ci = ni;                                                                                    \
                off_i = 0;                                                                                  \
                wb = 0;                                                                                     \
                ic0 = nc0;                                                                                  \
                iw0 = nw0;                                                                                  \
                fetch_window(ci, true, 32, colidx, wts, lane, pol_stream, ic1, iw1);                        \
                nmore = next_work_item(it_n, ni, W, n_items, n_chunks, chunk_row, chunk_begin, chunk_end,   \
                                       group_r0, group_r1, rowptr, n_rows);                                 \
                fetch_window(ni, nmore, 0, colidx, wts, lane, pol_stream, nc0, nw0);                        \
            }                                                                                               \
        } else if (off_i >= wb + 32) {                                                                      \
            wb += 32;                                                                                       \
            ic0 = ic1;                                                                                      \
            iw0 = iw1;                                                                                      \
            fetch_window(ci, true, wb + 32, colidx, wts, lane, pol_stream, ic1, iw1);                      \
        }                                                                                                   \
    } while (0)

#pragma unroll 1
    for (int s = 0; s < NS; ++s) GNN_ISSUE_BATCH();

    // ---- consume side ----
    const int64_t f_store = (f * (int64_t)sizeof(T) + 15) / 16 * 16 / (int64_t)sizeof(T);  // f, padded to 16 bytes
    constexpr int NP = Lane<T, VW>::kPairs;
    unsigned long long acc[VPT][NP];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int k = 0; k < NP; ++k) acc[v][k] = 0ull;
    uint32_t s_c = 0;
#pragma unroll 1
    for (int64_t it_c = w0; it_c < n_items && ok; it_c += W) {
        const Item x =
            load_item(it_c, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0, group_r1, rowptr, n_rows);
        if (x.skip) continue;
        // rows [wbase, wbase + 32) of a group: lane i holds row wbase + i's end
        // entry and its scale
        int32_t r = x.r0, wbase = x.r0, rwin = x.e;
        float swin = 1.f;
        auto load_rows = [&](int32_t base) {
            wbase = base;
            rwin = x.e;
            swin = 1.f;
            if (!x.chunk && base + lane < x.r1) {
                rwin = rowptr[base + lane + 1];
                if (p.rowscale) swin = __ldg(p.rowscale + base + lane);
            }
        };
        load_rows(x.r0);
        int32_t rend = x.chunk ? x.e : __shfl_sync(0xffffffffu, rwin, 0);
        // write row r (or the chunk's partial) and clear the accumulator
        auto finish_row = [&]() {
            if (r - wbase >= 32) load_rows(r);
            if (x.chunk) {
                float *dst = partial + it_c * pld;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int64_t c0 = (int64_t)(v * 32 + lane) * EPL;
                    if (c0 < pld) {
                        float a[EPL];
                        pairs_to_vals<T, VW>(acc[v], a);
#pragma unroll
                        for (int k = 0; k < EPL; ++k) dst[c0 + k] = a[k];
                    }
                }
            } else {
                const float scale = __shfl_sync(0xffffffffu, swin, r - wbase);
                T *out = static_cast<T *>(p.out) + (int64_t)r * p.ldo;
                const T *selfrow = nullptr;
                if (p.self_mode == SELF_COPY) selfrow = X + (int64_t)r * ldx;
                if (p.self_mode == SELF_ADD && r < p.n_self)
                    selfrow = static_cast<const T *>(p.self) + (int64_t)r * p.ld_self;
#pragma unroll
                for (int v = 0; v < VPT; ++v) {
                    const int64_t c0 = (int64_t)(v * 32 + lane) * EPL;
                    if (c0 >= f_store) continue;
                    const int f_left = (int)(f - c0 < EPL ? f - c0 : EPL);
                    float o[EPL];
                    pairs_to_vals<T, VW>(acc[v], o);
#pragma unroll
                    for (int k = 0; k < EPL; ++k) o[k] *= scale;
                    if (selfrow) {
                        uint32_t q[VW / 4];
                        float sv[EPL];
                        ldg_words<VW>(selfrow + c0, q);
                        words_to_vals<T, VW>(q, sv);
                        if (p.self_mode == SELF_ADD) {
#pragma unroll
                            for (int k = 0; k < EPL; ++k) o[k] += sv[k];
                        } else {
                            vals_to_words<T, VW>(sv, f_left, q);
                            stg_words<VW>(out + c0, q, pol_stream);
                        }
                    }
                    if (p.relu) {
#pragma unroll
                        for (int k = 0; k < EPL; ++k) o[k] = o[k] > 0.f ? o[k] : 0.f;
                    }
                    uint32_t q[VW / 4];
                    vals_to_words<T, VW>(o, f_left, q);
                    stg_words<VW>(out + p.out_off + c0, q, pol_stream);
                }
            }
#pragma unroll
            for (int v = 0; v < VPT; ++v)
#pragma unroll
                for (int k = 0; k < NP; ++k) acc[v][k] = 0ull;
        };
        int32_t pos = x.b;
#pragma unroll 1
        for (int32_t off = 0; off < x.e - x.b; off += BE) {
            const int slot = (int)(s_c % NS);
            if (!bar_wait(&bars[slot], (s_c / NS) & 1u)) {
                ok = false;
                break;
            }
            const int32_t left = x.e - x.b - off;
            const int cnt = left < BE ? left : BE;
            const uint8_t *sr = rows + slot * BE * R + lane * VW;  // this lane's piece of the slot's first row
            const unsigned long long *ws = wring + slot * BE;
            if (cnt == BE && rend - pos >= BE) {
                // the whole batch lies in the current row
#pragma unroll
                for (int k = 0; k < BE; ++k) accumulate_entry<T, VW, VPT, BE>(acc, sr + k * BOX, ws[k]);
                pos += BE;
            } else {
                int j = 0;
#pragma unroll 1
                while (j < cnt) {
                    // rows that end here (empty rows too) are written out first
#pragma unroll 1
                    while (pos == rend) {
                        finish_row();
                        ++r;
                        if (r - wbase >= 32) load_rows(r);
                        rend = __shfl_sync(0xffffffffu, rwin, r - wbase);
                    }
                    const int run = rend - pos < cnt - j ? rend - pos : cnt - j;
                    const uint8_t *rp = sr + j * BOX;
                    const unsigned long long *wp = ws + j;
                    if constexpr (VPT <= 2) {
                        // short rows: the run two entries at a time, then the odd one
                        int k = run;
#pragma unroll 1
                        for (; k >= 2; k -= 2, rp += 2 * BOX, wp += 2) {
                            accumulate_entry<T, VW, VPT, BE>(acc, rp, wp[0]);
                            accumulate_entry<T, VW, VPT, BE>(acc, rp + BOX, wp[1]);
                        }
                        if (k) accumulate_entry<T, VW, VPT, BE>(acc, rp, wp[0]);
                    } else {
#pragma unroll 1
                        for (int k = 0; k < run; ++k) accumulate_entry<T, VW, VPT, BE>(acc, rp + k * BOX, wp[k]);
                    }
                    j += run;
                    pos += run;
                }
            }
            ++s_c;
            __syncwarp();
            // the slot's rows were read through the generic proxy; the next
            // TMA gather into it is an async-proxy write
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            GNN_ISSUE_BATCH();
        }
        if (!ok) break;
        // the last row, then any empty rows after it
#pragma unroll 1
        while (r < x.r1) {
            finish_row();
            ++r;
        }
    }
#undef GNN_ISSUE_BATCH
    if (!ok) {
        // a copy never completed: report, then let every copy still in flight
        // land (bounded) before the warp's shared memory is released
        if (lane == 0 && p.err) atomicOr(p.err, 4);
        for (uint32_t s = s_c; s < s_i; ++s) bar_wait(&bars[s % NS], (s / NS) & 1u);
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
        if (p.relu) {
            o.x = o.x > 0.f ? o.x : 0.f;
            o.y = o.y > 0.f ? o.y : 0.f;
            o.z = o.z > 0.f ? o.z : 0.f;
            o.w = o.w > 0.f ? o.w : 0.f;
        }
        if (col + 0 >= f) o.x = 0.f;
        if (col + 1 >= f) o.y = 0.f;
        if (col + 2 >= f) o.z = 0.f;
        if (col + 3 >= f) o.w = 0.f;
        store4(out + p.out_off + col, o);
    }
}

template <typename T, int VW, int VPT, int BE, int NS, int WPC>
gnn_status launch_cfg(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    const int64_t items = sc.n_chunks + sc.n_groups;
    if (items > 0) {
        constexpr int R = 32 * VW * VPT;
        const int smem = WPC * BulkRing<R, BE, NS>::kBytes + 128;
        // the gathered matrix, one row high boxes of 32 * VW bytes (zero past column f)
        CUtensorMap xmap;
        memset(&xmap, 0, sizeof(xmap));
        if (p.n_x > 0 && !make_map_rows(&xmap, sizeof(T) == 2, p.X, (uint64_t)p.f, (uint64_t)p.n_x,
                                        (uint64_t)p.ldx * sizeof(T), (uint32_t)(32 * VW / (int)sizeof(T))))
            return GNN_ECUDA;
        auto kern = aggregate_kernel<T, VW, VPT, BE, NS, WPC>;
        GNN_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        // persistent warps: as many blocks as fit on the GPU at once
        int per_sm = 0;
        GNN_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, WPC * 32, smem));
        if (per_sm < 1) per_sm = 1;
        int64_t blocks = (int64_t)num_sms() * per_sm;
        if (blocks > ceil_div(items, WPC)) blocks = ceil_div(items, WPC);
        { kern<<<(unsigned)blocks, WPC * 32, smem, s>>>(p, xmap, sc.chunk_row, sc.chunk_begin, sc.chunk_end,
                                                        sc.n_chunks, sc.group_r0, sc.group_r1, sc.n_groups, partial,
                                                        pld); GNN_LAUNCHED(1); }
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
    // a warp keeps NS batches of BE rows in flight (8-16 KB of shared memory)
    if (bytes <= 128) return launch_cfg<T, 4, 1, 32, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 256) return launch_cfg<T, 8, 1, 16, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 512) return launch_cfg<T, 16, 1, 8, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 1024) return launch_cfg<T, 16, 2, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 1536) return launch_cfg<T, 16, 3, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 2048) return launch_cfg<T, 16, 4, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 2560) return launch_cfg<T, 16, 5, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 3072) return launch_cfg<T, 16, 6, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 4096) return launch_cfg<T, 16, 8, 4, 2, 2>(p, sc, partial, pld, s);
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
    p.err = g->err;
    p.rowptr = g->rowptr;
    p.colidx = reinterpret_cast<const uint32_t *>(g->colidx);
    p.wts = g->wfwd;
    p.rowscale = g->colw;
    p.n_rows = nL;
    p.colmask = g->fwd.tagged ? kColMask : 0xffffffffu;
    p.hot_tier = hot_tier_for(g->fwd, round_up(f * elem_size(dtype), 32));
    p.X = H;
    p.ldx = ld_h;
    p.n_x = g->n_local + g->n_halo;
    p.f = f;
    p.self_mode = sage ? SELF_COPY : SELF_NONE;
    p.out = Z;
    p.ldo = ld_z;
    p.out_off = sage ? half : 0;
    return launch_aggregate(p, g->fwd, dtype, scratch, static_cast<cudaStream_t>(stream));
}

