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
// Design (a gather bound by DRAM traffic and by instruction issue):
//  - work items: row groups (runs of consecutive non-empty light rows, <=
//    kHeavyNnz entries each, whose entries form one range) and kChunkNnz-entry
//    chunks of heavy rows; chunks are scheduled first so hub rows spread over
//    all SMs; a chunk writes an fp32 partial and a fix-up adds a heavy row's
//    partials in chunk order (deterministic, no atomics); the fix-up also
//    writes the empty rows;
//  - each item's entries stream through a producer / consumer warp pair in
//    batches that may span rows: the producer issues TMA gathers of four rows
//    (tile::gather4) into the pair's shared-memory ring, the consumer only
//    waits, loads from shared memory, multiplies-adds and writes rows out; the
//    end of a row is the sign bit of its last entry's weight (set at graph
//    creation), so the consumer never walks row pointers;
//  - L2 residency: column ids carry a hotness tier (access-count rank); rows
//    of the hottest tiers that fit a share of L2 are loaded with an evict_last
//    policy, the rest and the streamed ids / weights / outputs with evict_first.
#include <atomic>
#include <cstdlib>
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

// Shared memory of one producer / consumer pair: NS slots, each holding BE
// gathered rows (R bytes each), then the slots' weights (each stored twice, as
// a packed-FMA operand), their row-end masks, and a "full" and an "empty"
// mbarrier per slot.  A slot is laid out box-major: box v (bytes
// [v * 32 * VW, (v + 1) * 32 * VW) of every row) holds the BE rows one after
// another, as the TMA gathers deliver them.
template <int R, int BE, int NS>
struct PairRing {
    static constexpr int kSlotBytes = BE * R;
    static constexpr int kWeightOff = NS * kSlotBytes;                 // NS x BE weight pairs
    static constexpr int kMaskOff = kWeightOff + NS * BE * 8;          // NS row-end masks
    static constexpr int kBarOff = (kMaskOff + NS * 4 + 7) / 8 * 8;    // NS full, then NS empty mbarriers
    static constexpr int kBytes = (kBarOff + 2 * NS * 8 + 127) / 128 * 128;  // the next pair's rows stay 128-aligned
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

// bounded wait of one warp: every lane polls the barrier; the warp gives up
// together when any lane's wait ran out (after ~2 s) or, with a flag, when the
// CTA's abort flag is raised
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort, uint64_t limit_ns) {
    bool ok = bar_try(bar, parity);
    if (!__all_sync(0xffffffffu, ok)) {
        uint64_t t0;
        asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
        for (;;) {
            ok = bar_try(bar, parity);
            if (__all_sync(0xffffffffu, ok)) break;
            uint64_t t;
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
            const bool give_up = (abort && *abort) || t - t0 > limit_ns;
            if (__any_sync(0xffffffffu, give_up)) return false;
        }
    }
    return true;
}

__device__ __forceinline__ void bar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(static_cast<uint32_t>(__cvta_generic_to_shared(bar)))
                 : "memory");
}

// Producer / consumer warp pairs.  Pair q of P handles work items q, q + P, ...
// (row groups and heavy-row chunks) as one stream of batches of up to BE
// consecutive entries of one item.
//  - The producer warp reads an item's column ids and weights 32 entries at a
//    time (lane j: entry j), takes the row ends from the weights' sign bits and
//    the L2 policy of each group of four rows from their hotness tiers, then
//    per batch: waits for the slot to be free, stores the weights and the
//    row-end mask, and issues one TMA gather of four rows per group and box.
//  - The consumer warp waits for the batch, accumulates its entries (each lane
//    owns VW bytes of each of the VPT boxes of a row; packed fp32x2 FMA on
//    64-bit accumulator pairs), writes a row out at each marked row end (a
//    chunk of a heavy row writes its fp32 partial at the chunk's end instead),
//    and frees the slot.
// The consumer never reads row pointers or column ids: a group's rows are
// consecutive and non-empty, so its k-th row end is row r0 + k.
template <typename T, int VW, int VPT, int BE, int NS, int PPC, int MINB>
__global__ void __launch_bounds__(PPC * 64, MINB)
    aggregate_kernel(const AggParams p, const __grid_constant__ CUtensorMap xmap, const int32_t *__restrict__ chunk_row,
                     const int32_t *__restrict__ chunk_begin, const int32_t *__restrict__ chunk_end, int64_t n_chunks,
                     const int32_t *__restrict__ group_r0, const int32_t *__restrict__ group_r1, int64_t n_groups,
                     float *__restrict__ partial, int64_t pld) {
    constexpr int EPL = VW / (int)sizeof(T);  // values of a row per lane per box
    constexpr int BOX = 32 * VW;              // bytes of one gathered box of a row
    constexpr int R = VPT * BOX;
    static_assert(VW == 4 || VW == 8 || VW == 16, "lane piece of 4, 8 or 16 bytes");
    static_assert(BE == 4 || BE == 8 || BE == 16, "batches of whole groups of four inside one 32-entry window");
    static_assert(BOX % 128 == 0, "TMA destinations stay 128-byte aligned");
    using Ring = PairRing<R, BE, NS>;
    constexpr uint32_t kBatchMask = (1u << BE) - 1u;
    extern __shared__ __align__(128) uint8_t smem_raw[];
    __shared__ int abort_flag;
    // TMA destinations must be 128-byte aligned: round the dynamic base up
    // (the launch adds 128 bytes for this)
    uint8_t *smem = smem_raw + ((128u - (static_cast<uint32_t>(__cvta_generic_to_shared(smem_raw)) & 127u)) & 127u);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool producer = warp >= PPC;
    const int pair = producer ? warp - PPC : warp;
    uint8_t *rows = smem + pair * Ring::kBytes;
    unsigned long long *wring = reinterpret_cast<unsigned long long *>(rows + Ring::kWeightOff);
    uint32_t *emask = reinterpret_cast<uint32_t *>(rows + Ring::kMaskOff);
    uint64_t *full = reinterpret_cast<uint64_t *>(rows + Ring::kBarOff);
    uint64_t *empty = full + NS;
    if (threadIdx.x == 0) abort_flag = 0;
    if (!producer && lane == 0)
        for (int s = 0; s < NS; ++s) {
            bar_init(&full[s]);
            bar_init(&empty[s]);
        }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    __syncthreads();

    const int64_t P = (int64_t)gridDim.x * PPC;
    const int64_t q0 = (int64_t)blockIdx.x * PPC + pair;
    const int64_t n_items = n_chunks + n_groups;
    const int32_t *__restrict__ rowptr = p.rowptr;
    const int64_t n_rows = p.n_rows;

    if (producer) {
        const uint64_t pol_keep = policy_evict_last();
        const uint64_t pol_stream = policy_evict_first();
        const uint32_t *__restrict__ colidx = p.colidx;
        const float *__restrict__ wts = p.wts;
        const uint32_t colmask = p.colmask;
        const bool tagged = colmask == kColMask;
        const int hot_tier = p.hot_tier;
        uint32_t s_i = 0;  // batches issued
        int p_slot = 0;
        uint32_t p_phase = 0;
        bool ok = true;
        // the window being issued (raw column ids, weight bits; lane j: entry
        // wb + j of item x) and the next one, loaded a window ahead so issuing
        // never waits on an index load; the item after x is looked up an item
        // ahead for the same reason
        Item x, xn;
        int64_t it = q0 - P;
        bool have = next_work_item(it, x, P, n_items, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0, group_r1,
                                   rowptr, n_rows);
        int64_t itn = it;
        bool have_n = have && next_work_item(itn, xn, P, n_items, n_chunks, chunk_row, chunk_begin, chunk_end,
                                             group_r0, group_r1, rowptr, n_rows);
        auto load_window = [&](const Item &y, int32_t base, uint32_t &raw, uint32_t &wbits) {
            raw = 0;
            wbits = 0;
            if (base + lane < y.e - y.b) {
                raw = ld_stream_u32(colidx + y.b + base + lane, pol_stream);
                wbits = ld_stream_u32(wts + y.b + base + lane, pol_stream);
            }
        };
        uint32_t raw = 0, wbits = 0, raw_n = 0, wbits_n = 0;
        int32_t wb = 0;
        if (have) load_window(x, 0, raw, wbits);
#pragma unroll 1
        while (ok && have) {
            const int32_t n = x.e - x.b;
            const bool more_in_item = wb + 32 < n;
            if (more_in_item) load_window(x, wb + 32, raw_n, wbits_n);
            else if (have_n) load_window(xn, 0, raw_n, wbits_n);
            {
                const int nb = n - wb < 32 ? n - wb : 32;  // entries of this window
                const bool valid = lane < nb;
                const uint32_t ends = __ballot_sync(0xffffffffu, wbits >> 31);  // last entries of rows
                const uint32_t wa = wbits & 0x7fffffffu;
                const int tier = tagged ? (int)(raw >> kTierShift) : 0;
                const uint32_t hot = __ballot_sync(0xffffffffu, valid && tier <= hot_tier);
                // lanes past the window's entries repeat its last entry: a valid row (its weight is 0)
                const int32_t col = (int32_t)(__shfl_sync(0xffffffffu, raw, valid ? lane : nb - 1) & colmask);
                const int32_t c1 = __shfl_down_sync(0xffffffffu, col, 1);
                const int32_t c2 = __shfl_down_sync(0xffffffffu, col, 2);
                const int32_t c3 = __shfl_down_sync(0xffffffffu, col, 3);
#pragma unroll 1
                for (int k0 = 0; k0 < nb; k0 += BE) {
                    const int slot = p_slot;
                    if (!warp_wait(&empty[slot], p_phase ^ 1u, &abort_flag, p.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const int cnt = nb - k0 < BE ? nb - k0 : BE;
                    if (lane >= k0 && lane < k0 + BE)
                        wring[slot * BE + (lane - k0)] = ((unsigned long long)wa << 32) | wa;
                    if (lane == 0) emask[slot] = (ends >> k0) & kBatchMask;
                    const int ngr = (cnt + 3) >> 2;
                    __syncwarp();
                    // the arrive releases the weights and the mask; the gathers complete the phase
                    if (lane == 0) bar_expect(&full[slot], (uint32_t)(ngr * VPT * 4 * BOX));
                    __syncwarp();
                    const bool starved = p.starve && q0 == 0 && s_i == 0;  // failure test: never issued
                    if ((lane & 3) == 0 && lane >= k0 && lane < k0 + 4 * ngr && !starved) {
                        // keep the group in L2 when most of its rows are hot
                        const uint64_t pol = __popc((hot >> lane) & 0xfu) >= 2 ? pol_keep : pol_stream;
                        uint8_t *dst = rows + slot * Ring::kSlotBytes + (lane - k0) * BOX;
#pragma unroll
                        for (int v = 0; v < VPT; ++v)
                            tma_gather4(dst + v * BE * BOX, &xmap, v * (BOX / (int)sizeof(T)), col, c1, c2, c3,
                                        &full[slot], pol);
                    }
                    ++s_i;
                    if (++p_slot == NS) {
                        p_slot = 0;
                        p_phase ^= 1u;
                    }
                }
            }
            raw = raw_n;
            wbits = wbits_n;
            if (more_in_item) {
                wb += 32;
            } else {
                wb = 0;
                have = have_n;
                x = xn;
                if (have)
                    have_n = next_work_item(itn, xn, P, n_items, n_chunks, chunk_row, chunk_begin, chunk_end,
                                            group_r0, group_r1, rowptr, n_rows);
            }
        }
        if (!ok) {
            // the consumer gave up: let the gathers still in flight land (bounded)
            // before the CTA's shared memory is released
            for (uint32_t k = s_i > (uint32_t)NS ? s_i - NS : 0u; k < s_i; ++k)
                if (!(p.starve && q0 == 0 && k == 0)) warp_wait(&full[k % NS], (k / NS) & 1u, nullptr, p.wait_ns);
        }
        return;
    }

    // ---- consumer ----
    const T *__restrict__ X = static_cast<const T *>(p.X);
    const int64_t f = p.f, ldx = p.ldx;
    const uint64_t pol_out = policy_evict_first();
    const int64_t f_store = (f * (int64_t)sizeof(T) + 15) / 16 * 16 / (int64_t)sizeof(T);  // f, padded to 16 bytes
    constexpr int NP = Lane<T, VW>::kPairs;
    unsigned long long acc[VPT][NP];
#pragma unroll
    for (int v = 0; v < VPT; ++v)
#pragma unroll
        for (int k = 0; k < NP; ++k) acc[v][k] = 0ull;
    // per-row scales of a group, prefetched 32 rows at a time into the lanes
    // (lane i holds the scale of row sbase + i; the next 32 wait in snext)
    int32_t sbase = 0;
    float swin = 1.f, snext = 1.f;
    auto load_scales = [&](int32_t base, int32_t r1, float &dst) {
        dst = 1.f;
        if (p.rowscale && base + lane < r1) dst = __ldg(p.rowscale + base + lane);
    };
    // write row r of the output and clear the accumulator
    auto finish_row = [&](int32_t r, int32_t r1) {
        if (r - sbase >= 32) {  // rows run into the next window of 32
            sbase += 32;
            swin = snext;
            load_scales(sbase + 32, r1, snext);
        }
        const float scale = __shfl_sync(0xffffffffu, swin, r - sbase);
        T *out = static_cast<T *>(p.out) + (int64_t)r * p.ldo;
        const T *selfrow = nullptr;
        if (p.self_mode == SELF_COPY) selfrow = X + (int64_t)r * ldx;
        if (p.self_mode == SELF_ADD && r < p.n_self) selfrow = static_cast<const T *>(p.self) + (int64_t)r * p.ld_self;
#pragma unroll
        for (int v = 0; v < VPT; ++v) {
            const int64_t c0 = (int64_t)(v * 32 + lane) * EPL;
            if (c0 < f_store) {
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
                        stg_words<VW>(out + p.self_off + c0, q, pol_out);
                    }
                }
                if (p.relu) {
#pragma unroll
                    for (int k = 0; k < EPL; ++k) o[k] = o[k] > 0.f ? o[k] : 0.f;
                }
                uint32_t q[VW / 4];
                vals_to_words<T, VW>(o, f_left, q);
                stg_words<VW>(out + p.out_off + c0, q, pol_out);
            }
#pragma unroll
            for (int k = 0; k < NP; ++k) acc[v][k] = 0ull;
        }
    };
    int c_slot = 0;
    uint32_t c_phase = 0;
    bool ok = true;
#pragma unroll 1
    for (int64_t it = q0; it < n_items && ok; it += P) {
        const Item x = load_item(it, n_chunks, chunk_row, chunk_begin, chunk_end, group_r0, group_r1, rowptr, n_rows);
        if (x.skip || x.e <= x.b) continue;
        int32_t r = x.r0;
        const int32_t n = x.e - x.b;
        if (!x.chunk) {
            sbase = x.r0;
            load_scales(x.r0, x.r1, swin);
            load_scales(x.r0 + 32, x.r1, snext);
        }
#pragma unroll 1
        for (int32_t off = 0; off < n; off += BE) {
            const int slot = c_slot;
            if (!warp_wait(&full[slot], c_phase, &abort_flag, p.wait_ns)) {
                ok = false;
                break;
            }
            const int cnt = n - off < BE ? n - off : BE;
            const uint8_t *sr = rows + slot * Ring::kSlotBytes + lane * VW;  // this lane's piece of the first row
            const unsigned long long *ws = wring + slot * BE;
            const uint32_t em = x.chunk ? 0u : emask[slot];
            if (em == 0u) {
                if (cnt == BE) {
#pragma unroll
                    for (int k = 0; k < BE; ++k) accumulate_entry<T, VW, VPT, BE>(acc, sr + k * BOX, ws[k]);
                } else {
#pragma unroll 1
                    for (int k = 0; k < cnt; ++k) accumulate_entry<T, VW, VPT, BE>(acc, sr + k * BOX, ws[k]);
                }
            } else if constexpr (BE <= 8) {
#pragma unroll
                for (int k = 0; k < BE; ++k) {
                    if (k < cnt) {
                        accumulate_entry<T, VW, VPT, BE>(acc, sr + k * BOX, ws[k]);
                        if (em & (1u << k)) finish_row(r++, x.r1);
                    }
                }
            } else {
                // larger batches: one copy of the row end in the code
#pragma unroll 1
                for (int k = 0; k < cnt; ++k) {
                    accumulate_entry<T, VW, VPT, BE>(acc, sr + k * BOX, ws[k]);
                    if (em & (1u << k)) finish_row(r++, x.r1);
                }
            }
            // the slot was read through the generic proxy; the next gathers into it
            // are async-proxy writes
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) bar_arrive(&empty[slot]);
            if (++c_slot == NS) {
                c_slot = 0;
                c_phase ^= 1u;
            }
        }
        if (!ok) break;
        if (x.chunk) {
            float *dst = partial + it * pld;
#pragma unroll
            for (int v = 0; v < VPT; ++v) {
                const int64_t c0 = (int64_t)(v * 32 + lane) * EPL;
                if (c0 < pld) {
                    float a[EPL];
                    pairs_to_vals<T, VW>(acc[v], a);
#pragma unroll
                    for (int k = 0; k < EPL; ++k) dst[c0 + k] = a[k];
                }
#pragma unroll
                for (int k = 0; k < NP; ++k) acc[v][k] = 0ull;
            }
        }
    }
    if (!ok) {
        // a batch never arrived: report and make the producer stop
        if (lane == 0) {
            abort_flag = 1;
            if (p.err) atomicOr(p.err, kErrWaitAgg);
        }
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
                store4(out + p.self_off + col, sv);
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

template <typename T, int VW, int VPT, int BE, int NS, int PPC, int MINB>
gnn_status launch_cfg(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    const int64_t items = sc.n_chunks + sc.n_groups;
    if (items > 0) {
        constexpr int R = 32 * VW * VPT;
        const int smem = PPC * PairRing<R, BE, NS>::kBytes + 128;
        // the gathered matrix, one row high boxes of 32 * VW bytes (zero past column f)
        CUtensorMap xmap;
        memset(&xmap, 0, sizeof(xmap));
        if (p.n_x > 0 && !make_map_rows(&xmap, sizeof(T) == 2, p.X, (uint64_t)p.f, (uint64_t)p.n_x,
                                        (uint64_t)p.ldx * sizeof(T), (uint32_t)(32 * VW / (int)sizeof(T))))
            return GNN_ECUDA;
        auto kern = aggregate_kernel<T, VW, VPT, BE, NS, PPC, MINB>;
        GNN_CUDA_TRY(cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
        // persistent pairs: as many blocks as fit on the GPU at once
        int per_sm = 0;
        GNN_CUDA_TRY(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, PPC * 64, smem));
        if (per_sm < 1) per_sm = 1;
        int64_t blocks = (int64_t)num_sms() * per_sm;
        if (blocks > ceil_div(items, PPC)) blocks = ceil_div(items, PPC);
        { kern<<<(unsigned)blocks, PPC * 64, smem, s>>>(p, xmap, sc.chunk_row, sc.chunk_begin, sc.chunk_end,
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

// pipeline shape of the aggregation (GNN_AGG_PIPE, for tuning): 0 = by row
// size (measured best on the R-MAT partitions: four pairs per block with three
// slots of 8 or 16 entries for rows of up to 512 bytes; two pairs with three
// slots of 8 entries for 1 KB rows); 1 = two pairs with six slots; 2 = batches
// of 16 entries for 512-byte rows, two pairs with three slots
int agg_pipe() {
    static int v = -1;
    if (v < 0) {
        const char *e = getenv("GNN_AGG_PIPE");
        v = e ? atoi(e) : kAggPipe;
        if (v < 0 || v > 2) v = kAggPipe;
    }
    return v;
}

template <typename T>
gnn_status launch_typed(const AggParams &p, const Schedule &sc, float *partial, int64_t pld, cudaStream_t s) {
    // a slot holds 2-16 KB of gathered rows (whole groups of four); the pairs a
    // SM holds are set by shared memory and registers, the bytes in flight by
    // pairs x slots
    const int64_t bytes = p.f * (int64_t)sizeof(T);
    const int pipe = agg_pipe();
    if (bytes <= 128) return launch_cfg<T, 4, 1, 16, 4, 4, 3>(p, sc, partial, pld, s);
    if (bytes <= 256) {
        if (pipe == 1) return launch_cfg<T, 8, 1, 16, 6, 2, 6>(p, sc, partial, pld, s);
        return launch_cfg<T, 8, 1, 16, 3, 4, 4>(p, sc, partial, pld, s);
    }
    if (bytes <= 512) {
        if (pipe == 1) return launch_cfg<T, 16, 1, 8, 6, 2, 6>(p, sc, partial, pld, s);
        if (pipe == 2) return launch_cfg<T, 16, 1, 16, 3, 2, 4>(p, sc, partial, pld, s);
        return launch_cfg<T, 16, 1, 8, 3, 4, 4>(p, sc, partial, pld, s);
    }
    if (bytes <= 1024) {
        if (pipe == 1) return launch_cfg<T, 16, 2, 4, 6, 2, 6>(p, sc, partial, pld, s);
        return launch_cfg<T, 16, 2, 8, 3, 2, 4>(p, sc, partial, pld, s);
    }
    // wider rows: two pairs per block with three or four slots (deeper rings
    // measured better than more pairs for 1 KB rows)
    if (bytes <= 1536) return launch_cfg<T, 16, 3, 4, 4, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 2048) return launch_cfg<T, 16, 4, 4, 3, 2, 4>(p, sc, partial, pld, s);
    if (bytes <= 2560) return launch_cfg<T, 16, 5, 4, 3, 2, 3>(p, sc, partial, pld, s);
    if (bytes <= 3072) return launch_cfg<T, 16, 6, 4, 3, 2, 2>(p, sc, partial, pld, s);
    if (bytes <= 4096) return launch_cfg<T, 16, 8, 4, 3, 1, 2>(p, sc, partial, pld, s);
    return GNN_EUNSUPPORTED;
}

}  // namespace

size_t aggregate_partial_bytes(const Schedule &sc, int64_t f) {
    return (size_t)sc.n_chunks * (size_t)round_up(f, 8) * sizeof(float);
}

namespace {
std::atomic<int64_t> g_expire_ns{0};  // armed by gnn_debug_expire_next_wait

// Rows wider than this many bytes are aggregated in column slices of this
// width, one pass per slice (0: one pass).  GNN_AGG_SLICE_BYTES overrides it
// (a multiple of 128).
int64_t agg_slice_bytes() {
    static int64_t v = -1;
    if (v < 0) {
        const char *e = getenv("GNN_AGG_SLICE_BYTES");
        int64_t x = e ? atoll(e) : kAggSliceBytes;
        v = (x > 0 && x % 128 == 0) ? x : 0;
    }
    return v;
}
}  // namespace

gnn_status launch_aggregate(const AggParams &p_in, const Schedule &sc, gnn_dtype dt, float *partial, cudaStream_t s) {
    if (p_in.n_rows == 0) return GNN_OK;
    AggParams p = p_in;
    p.wait_ns = 2000000000ull;
    p.starve = 0;
    if (sc.n_chunks + sc.n_groups > 0) {
        const int64_t ns = g_expire_ns.exchange(0);
        if (ns > 0) {
            p.wait_ns = (uint64_t)ns;
            p.starve = 1;
        }
    }
    const int64_t es = dt == GNN_BF16 ? 2 : 4;
    const int64_t slice = agg_slice_bytes();
    if (slice <= 0 || p.f * es <= slice) {
        const int64_t pld = round_up(p.f, 8);
        if (dt == GNN_BF16) return launch_typed<__nv_bfloat16>(p, sc, partial, pld, s);
        return launch_typed<float>(p, sc, partial, pld, s);
    }
    // column slices, one pass each: a pass gathers rows of `slice` bytes, so the
    // L2 holds more of the hot rows of the pass
    const int64_t fs = slice / es;
    for (int64_t c0 = 0; c0 < p.f; c0 += fs) {
        AggParams q = p;
        q.f = p.f - c0 < fs ? p.f - c0 : fs;
        q.X = static_cast<const char *>(p.X) + c0 * es;
        q.out_off = p.out_off + c0;
        q.self_off = p.self_off + c0;
        if (p.self) q.self = static_cast<const char *>(p.self) + c0 * es;
        q.hot_tier = hot_tier_for(sc, round_up(q.f * es, 32));
        if (c0 > 0) q.starve = 0;
        const int64_t pld = round_up(q.f, 8);
        const gnn_status st = dt == GNN_BF16 ? launch_typed<__nv_bfloat16>(q, sc, partial, pld, s)
                                             : launch_typed<float>(q, sc, partial, pld, s);
        if (st != GNN_OK) return st;
    }
    return GNN_OK;
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

extern "C" gnn_status gnn_debug_expire_next_wait(int64_t wait_ns) {
    gnn::g_expire_ns.store(wait_ns > 0 ? wait_ns : 0);
    return GNN_OK;
}

extern "C" gnn_status gnn_aggregate_forward_noalloc(const gnn_graph *g, const void *H, int64_t ld_h, int64_t f,
                                                    void *Z, int64_t ld_z, gnn_dtype dtype, void *stream) {
    using namespace gnn;
    if (!g || (dtype != GNN_F32 && dtype != GNN_BF16) || f <= 0 || g->agg == GNN_AGG_GAT) return GNN_EINVAL;
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

