// update_tc.cu - the dense update H_out = act(Z W) on the 5th-generation tensor
// cores (tcgen05, bf16 inputs, fp32 accumulation in TMEM), for bf16 data.
//
// Persistent kernel, one CTA per SM, 6 warps:
//   warp 0      TMA producer: W^T once (resident in shared memory for the whole
//               kernel), then 128-row x 64-column tiles of Z through a ring of
//               stages (128-byte swizzle)
//   warp 1      MMA issuer (one thread): for each 128-row tile, K/16 MMAs of
//               128 x N_pad x 16 into one of two TMEM accumulators
//   warps 2..5  epilogue: tcgen05.ld of the accumulator (each warp owns the 32
//               TMEM lanes of its quarter, each thread one row), ReLU, round to
//               bf16 into a swizzled 32 x 64 staging tile, TMA store of the tile;
//               then the accumulator is handed back to the MMA warp
// The double-buffered accumulator lets the epilogue of tile i overlap the MMAs
// of tile i + 1.  Every wait is bounded (see tc_common.cuh).
#include <cudaTypedefs.h>

#include "gnn_internal.cuh"
#include "tc_common.cuh"

namespace gnn {

namespace {

constexpr int kBM = 128;           // rows per tile = TMEM lanes
constexpr int kBK = 64;            // K per stage: one 128-byte swizzle atom of bf16
constexpr int kTileBytes = kBM * kBK * 2;
constexpr int kMaxStages = 8;
constexpr int kThreads = 192;
constexpr size_t kSmemLimit = 227 * 1024;
constexpr int kStageOut = 32 * 128;           // one 32-row x 64-column bf16 output tile
constexpr int kOutBytes = 4 * 2 * kStageOut;  // 4 epilogue warps x 2 buffers

struct Bars {
    uint64_t full[kMaxStages];
    uint64_t empty[kMaxStages];
    uint64_t tfull[2];
    uint64_t tempty[2];
    uint64_t wbar;
    uint64_t drain;
    uint32_t tmem_slot;
    int abort_flag;
};

__device__ __forceinline__ uint32_t pack2(float a, float b) {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(kThreads, 1)
    update_fwd_tc_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                         const __grid_constant__ CUtensorMap mapO, int64_t M, int N, int N_pad, int KC, int stages,
                         int relu, int64_t n_tiles, int *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sW = smem;
    const int w_chunk = N_pad * 128;
    uint8_t *sA = sW + KC * w_chunk;
    uint8_t *sO = sA + stages * kTileBytes;  // 1024-aligned: W chunks and A tiles are multiples of 1 KB
    Bars *bars = reinterpret_cast<Bars *>(sO + kOutBytes);
    volatile int *abort_flag = &bars->abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ncols = N_pad <= 128 ? 256u : 512u;
    const uint32_t acc_stride = ncols / 2;

    if (threadIdx.x == 0) {
        for (int s = 0; s < stages; ++s) {
            tc::mbar_init(&bars->full[s], 1);
            tc::mbar_init(&bars->empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            tc::mbar_init(&bars->tfull[b], 1);
            tc::mbar_init(&bars->tempty[b], 4);
        }
        tc::mbar_init(&bars->wbar, 1);
        tc::mbar_init(&bars->drain, 1);
        bars->abort_flag = 0;
        tc::fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bars->tmem_slot, ncols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&mapA);
        tc::prefetch_tmap(&mapB);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(&bars->wbar, (uint32_t)(KC * w_chunk));
            for (int kc = 0; kc < KC; ++kc) tc::tma_load_2d(sW + kc * w_chunk, &mapB, kc * kBK, 0, &bars->wbar);
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued = 0;  // stages with a load issued, for the abort drain
            uint32_t issued_parity = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int kc = 0; kc < KC; ++kc) {
                    if (!tc::mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)kTileBytes);
                    tc::tma_load_2d(sA + stage * kTileBytes, &mapA, kc * kBK, (int32_t)(t * kBM), &bars->full[stage]);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {  // let the loads already issued land before the CTA leaves
                int dummy = 0;
                for (int s = 0; s < stages; ++s)
                    if (issued & (1u << s))
                        tc::mbar_wait(&bars->full[s], (issued_parity >> s) & 1u, (volatile int *)&dummy);
                tc::mbar_wait(&bars->wbar, 0, (volatile int *)&dummy);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kBM, N_pad, 0, 0);
            bool ok = tc::mbar_wait(&bars->wbar, 0, abort_flag);
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                if (!tc::mbar_wait(&bars->tempty[acc], acc_phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t d = tmem_base + acc * acc_stride;
                for (int kc = 0; kc < KC; ++kc) {
                    if (!tc::mbar_wait(&bars->full[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(sA + stage * kTileBytes);
                    const uint32_t b0 = tc::smem_u32(sW + kc * w_chunk);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc::mma_bf16(d, tc::sw128_desc(a0 + k * 32, 16, 1024), tc::sw128_desc(b0 + k * 32, 16, 1024),
                                     idesc, (kc | k) != 0);
                    tc::mma_commit(&bars->empty[stage]);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc::mma_commit(&bars->tfull[acc]);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (!ok) {  // wait for the MMAs in flight before TMEM is released
                int dummy = 0;
                tc::mma_commit(&bars->drain);
                tc::mbar_wait(&bars->drain, 0, (volatile int *)&dummy);
            }
        }
    } else {
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t *stage_out = sO + (warp - 2) * 2 * kStageOut;
        int acc = 0, ob = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            if (!tc::mbar_wait(&bars->tfull[acc], acc_phase, abort_flag)) break;
            tc::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * acc_stride;
            for (int cc = 0; cc < N_pad; cc += 64) {
                // the TMA store that last read this buffer must be done with it
                if (lane == 0) tc::bulk_wait_read<1>();
                __syncwarp();
                uint8_t *buf = stage_out + ob * kStageOut;
#pragma unroll
                for (int sub = 0; sub < 4; ++sub) {
                    const int c = cc + sub * 16;
                    uint32_t r[16];
                    if (c < N_pad) {
                        tc::tmem_ld16(taddr + (uint32_t)c, r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = 0u;
                    }
                    float v[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float x = __uint_as_float(r[i]);
                        v[i] = (relu && !(x > 0.f)) ? 0.f : x;
                    }
                    // 16-byte chunks 2*sub and 2*sub+1 of this thread's 128-byte row, 128-byte swizzle
                    uint4 lo = make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
                    uint4 hi = make_uint4(pack2(v[8], v[9]), pack2(v[10], v[11]), pack2(v[12], v[13]),
                                          pack2(v[14], v[15]));
                    uint8_t *rowp = buf + lane * 128;
                    *reinterpret_cast<uint4 *>(rowp + (((2 * sub) ^ (lane & 7)) * 16)) = lo;
                    *reinterpret_cast<uint4 *>(rowp + (((2 * sub + 1) ^ (lane & 7)) * 16)) = hi;
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_2d(&mapO, cc, (int32_t)(t * kBM + q * 32), buf);
                    tc::bulk_commit();
                }
                ob ^= 1;
            }
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars->tempty[acc]);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
        if (lane == 0) tc::bulk_wait<0>();
        __syncwarp();
    }
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && bars->abort_flag) atomicOr(err, kErrWaitTc);
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, ncols);
    }
}

__global__ void pack_wt_bf16_kernel(const float *__restrict__ Wp, int64_t ldw, int64_t Kp, int64_t N, int64_t K_pad,
                                    int64_t N_pad, __nv_bfloat16 *__restrict__ Wt) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= N_pad * K_pad) return;
    int64_t n = x / K_pad, k = x % K_pad;
    float v = (n < N && k < Kp) ? Wp[k * ldw + n] : 0.f;
    Wt[x] = __float2bfloat16_rn(v);
}

}  // namespace

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

bool make_map_bf16_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_f32_2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                     uint32_t box_inner, uint32_t box_outer) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_map_rows(CUtensorMap *m, bool bf16, const void *base, uint64_t inner, uint64_t outer, uint64_t row_bytes,
                   uint32_t box_inner) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {inner, outer};
    cuuint64_t strides[1] = {row_bytes};
    cuuint32_t box[2] = {box_inner, 1};
    cuuint32_t es[2] = {1, 1};
    return fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base),
              dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
    static int n = 0;
    if (!n) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (n <= 0) n = 148;
    }
    return n;
}

namespace {

// one pass holds all of W (Kp x N) in shared memory next to two Z stages
bool fwd_pass_ok(int64_t Kp, int64_t N) {
    const int64_t N_pad = round_up(N, 16);
    const int64_t KC = ceil_div(Kp, kBK);
    if (N_pad > 256 || KC < 1) return false;
    const size_t w = (size_t)KC * N_pad * 128;
    return w + 2 * kTileBytes + kOutBytes + sizeof(Bars) + 1024 <= kSmemLimit;
}

// output columns per pass: all N, or slices of 128 when W does not fit (the
// passes read Z again; each writes its own columns of the output)
constexpr int64_t kNSlice = 128;
int64_t fwd_slice(int64_t Kp, int64_t N) {
    if (fwd_pass_ok(Kp, N)) return N;
    if (N > kNSlice && fwd_pass_ok(Kp, kNSlice)) return kNSlice;
    return 0;
}

gnn_status fwd_tc_pass(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                       int relu, void *out, int64_t ld_o, void *wt_ws, int *err, cudaStream_t s);

}  // namespace

size_t update_tc_wt_bytes(int64_t Kp, int64_t N) {
    const int64_t ns = fwd_slice(Kp, N);
    return (size_t)round_up(ns > 0 ? ns : N, 16) * (size_t)round_up(Kp, kBK) * 2;
}

bool update_fwd_tc_supported(int64_t Kp, int64_t N) { return fwd_slice(Kp, N) > 0; }

gnn_status launch_update_fwd_tc(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w,
                                int64_t N, int relu, void *out, int64_t ld_o, void *wt_ws, int *err, cudaStream_t s) {
    const int64_t ns = fwd_slice(Kp, N);
    if (ns <= 0) return GNN_EUNSUPPORTED;
    for (int64_t n0 = 0; n0 < N; n0 += ns) {
        const gnn_status st = fwd_tc_pass(Z, ld_z, n, Kp, Wp + n0, ld_w, N - n0 < ns ? N - n0 : ns, relu,
                                          static_cast<__nv_bfloat16 *>(out) + n0, ld_o, wt_ws, err, s);
        if (st != GNN_OK) return st;
    }
    return GNN_OK;
}

namespace {

gnn_status fwd_tc_pass(const void *Z, int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                       int relu, void *out, int64_t ld_o, void *wt_ws, int *err, cudaStream_t s) {
    const int64_t N_pad = round_up(N, 16);
    const int64_t KC = ceil_div(Kp, kBK);
    const int64_t K_pad = KC * kBK;
    __nv_bfloat16 *Wt = static_cast<__nv_bfloat16 *>(wt_ws);
    { pack_wt_bf16_kernel<<<(unsigned)ceil_div(N_pad * K_pad, 256), 256, 0, s>>>(Wp, ld_w, Kp, N, K_pad, N_pad, Wt); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    CUtensorMap mapA, mapB, mapO;
    if (!make_map_bf16_2d(&mapA, Z, (uint64_t)Kp, (uint64_t)n, (uint64_t)ld_z * 2, kBK, kBM)) return GNN_ECUDA;
    if (!make_map_bf16_2d(&mapB, Wt, (uint64_t)K_pad, (uint64_t)N_pad, (uint64_t)K_pad * 2, kBK, (uint32_t)N_pad))
        return GNN_ECUDA;
    if (!make_map_bf16_2d(&mapO, out, (uint64_t)N, (uint64_t)n, (uint64_t)ld_o * 2, 64, 32)) return GNN_ECUDA;
    const size_t w_bytes = (size_t)KC * N_pad * 128;
    int stages = (int)((kSmemLimit - w_bytes - kOutBytes - sizeof(Bars) - 1024) / kTileBytes);
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return GNN_EUNSUPPORTED;
    const size_t smem = w_bytes + (size_t)stages * kTileBytes + kOutBytes + sizeof(Bars) + 1024;
    GNN_CUDA_TRY(cudaFuncSetAttribute(update_fwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem));
    const int64_t n_tiles = ceil_div(n, kBM);
    const int64_t grid = n_tiles < num_sms() ? n_tiles : num_sms();
    { update_fwd_tc_kernel<<<(unsigned)grid, kThreads, smem, s>>>(mapA, mapB, mapO, n, (int)N, (int)N_pad, (int)KC,
                                                                stages, relu, n_tiles, err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace

}  // namespace gnn
