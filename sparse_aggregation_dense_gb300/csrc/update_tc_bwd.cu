// update_tc_bwd.cu - backward of the dense update on the tensor cores (bf16
// storage, fp32 accumulation), by the chain rule of H_out = act(Z W):
//   dY = G * 1[H_out > 0]   (ReLU'(0) = 0; dY = G without ReLU)
//   dZ = dY W^T             dgrad kernel
//   dW = Z^T dY             wgrad kernel: per-CTA partial sums over row tiles,
//                           then a fixed-order sum over CTAs
// Both kernels stream tiles of G (and H_out) with TMA; four "mask" warps apply
// the ReLU mask in place in shared memory (G and H_out tiles share the same
// swizzled layout, so the mask is elementwise on raw bytes) before the MMA
// warp consumes them.
//   warp 0 TMA producer, warp 1 MMA issuer, warps 2..5 epilogue, warps 6..9 mask
// dgrad: K-major operands (dY tile x resident W), accumulator double-buffered.
// wgrad: MN-major operands (Z^T and dY^T straight from the row tiles), one
// accumulator per CTA holding its whole Kp x N partial.
#include <cudaTypedefs.h>

#include "gnn_internal.cuh"
#include "tc_common.cuh"

namespace gnn {

namespace {

constexpr int kThreadsB = 320;
constexpr int kMaxStagesB = 6;
constexpr size_t kSmemLimitB = 227 * 1024;
constexpr int kDRows = 128;  // dgrad rows per tile
constexpr int kWRows = 64;   // wgrad rows per tile
constexpr int kBoxD = kDRows * 128;  // one 64-column bf16 box of a dgrad tile
constexpr int kBoxW = kWRows * 128;  // one 64-column bf16 box of a wgrad tile
constexpr int kStageOut = 32 * 128;           // one 32-row x 128-byte dZ tile (TMA store source)
constexpr int kOutBytes = 4 * 2 * kStageOut;  // 4 epilogue warps x 2 buffers

struct BarsB {
    uint64_t full[kMaxStagesB];
    uint64_t ready[kMaxStagesB];
    uint64_t empty[kMaxStagesB];
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

__device__ __forceinline__ uint32_t mask_pair(uint32_t g, uint32_t h) {
    // keep each bf16 half of g where the matching half of h is > 0
    const float h0 = __uint_as_float(h << 16), h1 = __uint_as_float(h & 0xffff0000u);
    return (h0 > 0.f ? (g & 0x0000ffffu) : 0u) | (h1 > 0.f ? (g & 0xffff0000u) : 0u);
}

// in-place ReLU mask of `bytes` bytes of G by H, by the 128 mask threads
__device__ __forceinline__ void mask_tile(uint8_t *g, const uint8_t *h, int bytes, int tid) {
    uint4 *g4 = reinterpret_cast<uint4 *>(g);
    const uint4 *h4 = reinterpret_cast<const uint4 *>(h);
    for (int i = tid; i < bytes / 16; i += 128) {
        uint4 a = g4[i];
        const uint4 b = h4[i];
        a.x = mask_pair(a.x, b.x);
        a.y = mask_pair(a.y, b.y);
        a.z = mask_pair(a.z, b.z);
        a.w = mask_pair(a.w, b.w);
        g4[i] = a;
    }
}

__device__ __forceinline__ void init_common(BarsB *bars, int stages, uint32_t tempty_count) {
    for (int s = 0; s < stages; ++s) {
        tc::mbar_init(&bars->full[s], 1);
        tc::mbar_init(&bars->ready[s], 4);
        tc::mbar_init(&bars->empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
        tc::mbar_init(&bars->tfull[b], 1);
        tc::mbar_init(&bars->tempty[b], tempty_count);
    }
    tc::mbar_init(&bars->wbar, 1);
    tc::mbar_init(&bars->drain, 1);
    bars->abort_flag = 0;
    tc::fence_mbar_init();
}

// ---------------------------------------------------------------------------
// dgrad: dZ[m][k] = sum_n dY[m][n] W[k][n]; A = dY tile (K-major over n),
// B = W packed as Wk[k][n] (K-major over n), resident; D = 128 x Kp_pad.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsB, 1)
    update_dgrad_tc_kernel(const __grid_constant__ CUtensorMap mapG, const __grid_constant__ CUtensorMap mapH,
                           const __grid_constant__ CUtensorMap mapW, const __grid_constant__ CUtensorMap mapO,
                           int Kp_pad, int NC, int stages, int relu, int out_f32, int64_t n_tiles, int *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int w_chunk = Kp_pad * 128;
    uint8_t *sW = smem;
    uint8_t *sG = sW + NC * w_chunk;
    uint8_t *sH = sG + stages * kBoxD;
    uint8_t *sO = sH + (relu ? stages * kBoxD : 0);  // 1024-aligned: every region above is a multiple of 1 KB
    BarsB *bars = reinterpret_cast<BarsB *>(sO + kOutBytes);
    volatile int *abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t ncols = Kp_pad <= 128 ? 256u : 512u;
    const uint32_t acc_stride = ncols / 2;

    if (threadIdx.x == 0) init_common(bars, stages, 4);
    if (warp == 1) {
        tc::tmem_alloc(&bars->tmem_slot, ncols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&mapG);
        if (relu) tc::prefetch_tmap(&mapH);
        tc::prefetch_tmap(&mapW);
        tc::prefetch_tmap(&mapO);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_slot;
    const uint32_t stage_bytes = (uint32_t)(relu ? 2 * kBoxD : kBoxD);

    if (warp == 0) {
        if (lane == 0) {
            tc::mbar_arrive_expect_tx(&bars->wbar, (uint32_t)(NC * w_chunk));
            for (int nc = 0; nc < NC; ++nc) tc::tma_load_2d(sW + nc * w_chunk, &mapW, nc * 64, 0, &bars->wbar);
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
                for (int nc = 0; nc < NC; ++nc) {
                    if (!tc::mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::mbar_arrive_expect_tx(&bars->full[stage], stage_bytes);
                    tc::tma_load_2d(sG + stage * kBoxD, &mapG, nc * 64, (int32_t)(t * kDRows), &bars->full[stage]);
                    if (relu)
                        tc::tma_load_2d(sH + stage * kBoxD, &mapH, nc * 64, (int32_t)(t * kDRows),
                                        &bars->full[stage]);
                    issued |= 1u << stage;
                    issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                int dummy = 0;
                for (int s = 0; s < stages; ++s)
                    if (issued & (1u << s))
                        tc::mbar_wait(&bars->full[s], (issued_parity >> s) & 1u, (volatile int *)&dummy);
                tc::mbar_wait(&bars->wbar, 0, (volatile int *)&dummy);
            }
        }
    } else if (warp >= 6) {
        const int tid = threadIdx.x - 192;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t t = blockIdx.x; t < n_tiles && ok; t += gridDim.x) {
            for (int nc = 0; nc < NC; ++nc) {
                if (!tc::mbar_wait(&bars->full[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                if (relu) mask_tile(sG + stage * kBoxD, sH + stage * kBoxD, kBoxD, tid);
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars->ready[stage]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(kDRows, Kp_pad, 0, 0);
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
                for (int nc = 0; nc < NC; ++nc) {
                    if (!tc::mbar_wait(&bars->ready[stage], phase, abort_flag)) {
                        ok = false;
                        break;
                    }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(sG + stage * kBoxD);
                    const uint32_t b0 = tc::smem_u32(sW + nc * w_chunk);
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        tc::mma_bf16(d, tc::sw128_desc(a0 + k * 32, 16, 1024), tc::sw128_desc(b0 + k * 32, 16, 1024),
                                     idesc, (nc | k) != 0);
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
            if (!ok) {
                int dummy = 0;
                tc::mma_commit(&bars->drain);
                tc::mbar_wait(&bars->drain, 0, (volatile int *)&dummy);
            }
        }
    } else {
        // epilogue: TMEM -> a swizzled staging tile of 32 rows x 128 bytes (64 bf16
        // or 32 fp32 columns) -> TMA store (rows and columns past dZ's edge are
        // not written)
        const int q = warp & 3;  // TMEM lane quarter this warp may access
        uint8_t *stage_out = sO + (warp - 2) * 2 * kStageOut;
        const int cstep = out_f32 ? 32 : 64;  // columns per 128-byte staging row
        int acc = 0, ob = 0;
        uint32_t acc_phase = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            if (!tc::mbar_wait(&bars->tfull[acc], acc_phase, abort_flag)) break;
            tc::tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + acc * acc_stride;
            for (int cc = 0; cc < Kp_pad; cc += cstep) {
                // the TMA store that last read this buffer must be done with it
                if (lane == 0) tc::bulk_wait_read<1>();
                __syncwarp();
                uint8_t *buf = stage_out + ob * kStageOut;
                uint8_t *rowp = buf + lane * 128;
                if (out_f32) {
#pragma unroll
                    for (int sub = 0; sub < 2; ++sub) {
                        const int c = cc + sub * 16;
                        uint32_t r[16];
                        if (c < Kp_pad) {
                            tc::tmem_ld16(taddr + (uint32_t)c, r);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) r[i] = 0u;
                        }
                        // 16-byte chunks 4*sub .. 4*sub+3 of this thread's row, 128-byte swizzle
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            *reinterpret_cast<uint4 *>(rowp + (((4 * sub + j) ^ (lane & 7)) * 16)) =
                                make_uint4(r[4 * j], r[4 * j + 1], r[4 * j + 2], r[4 * j + 3]);
                    }
                } else {
#pragma unroll
                    for (int sub = 0; sub < 4; ++sub) {
                        const int c = cc + sub * 16;
                        uint32_t r[16];
                        if (c < Kp_pad) {
                            tc::tmem_ld16(taddr + (uint32_t)c, r);
                        } else {
#pragma unroll
                            for (int i = 0; i < 16; ++i) r[i] = 0u;
                        }
                        // 16-byte chunks 2*sub and 2*sub+1 of this thread's 128-byte row, 128-byte swizzle
                        uint4 lo = make_uint4(pack2(__uint_as_float(r[0]), __uint_as_float(r[1])),
                                              pack2(__uint_as_float(r[2]), __uint_as_float(r[3])),
                                              pack2(__uint_as_float(r[4]), __uint_as_float(r[5])),
                                              pack2(__uint_as_float(r[6]), __uint_as_float(r[7])));
                        uint4 hi = make_uint4(pack2(__uint_as_float(r[8]), __uint_as_float(r[9])),
                                              pack2(__uint_as_float(r[10]), __uint_as_float(r[11])),
                                              pack2(__uint_as_float(r[12]), __uint_as_float(r[13])),
                                              pack2(__uint_as_float(r[14]), __uint_as_float(r[15])));
                        *reinterpret_cast<uint4 *>(rowp + (((2 * sub) ^ (lane & 7)) * 16)) = lo;
                        *reinterpret_cast<uint4 *>(rowp + (((2 * sub + 1) ^ (lane & 7)) * 16)) = hi;
                    }
                }
                tc::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tc::tma_store_2d(&mapO, cc, (int32_t)(t * kDRows + q * 32), buf);
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

// ---------------------------------------------------------------------------
// wgrad: partial[cta][k][n] = sum over the CTA's 64-row tiles of Z[m][k] dY[m][n].
// A = Z^T (MN-major: k contiguous within a box, m the reduction), B = dY^T
// (MN-major), D = MB blocks of 128 k-rows x N_pad columns in TMEM.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreadsB, 1)
    update_wgrad_tc_kernel(const __grid_constant__ CUtensorMap mapZ, const __grid_constant__ CUtensorMap mapG,
                           const __grid_constant__ CUtensorMap mapH, float *__restrict__ partial, int64_t M, int Kp,
                           int MB, int N, int N_pad, int NC, int stages, int relu, int64_t n_tiles, int *err) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int zboxes = 2 * MB;
    const int stage_boxes = zboxes + NC * (relu ? 2 : 1);
    const int stage_bytes = stage_boxes * kBoxW;
    BarsB *bars = reinterpret_cast<BarsB *>(smem + stages * stage_bytes);
    volatile int *abort_flag = &bars->abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint32_t ncols = 32;
    while (ncols < (uint32_t)(MB * N_pad)) ncols <<= 1;

    if (threadIdx.x == 0) init_common(bars, stages, 4);
    if (warp == 1) {
        tc::tmem_alloc(&bars->tmem_slot, ncols);
        tc::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tc::prefetch_tmap(&mapZ);
        tc::prefetch_tmap(&mapG);
        if (relu) tc::prefetch_tmap(&mapH);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem_base = bars->tmem_slot;

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, issued = 0, issued_parity = 0;
            bool ok = true;
            for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
                if (!tc::mbar_wait(&bars->empty[stage], phase ^ 1u, abort_flag)) {
                    ok = false;
                    break;
                }
                uint8_t *base = smem + stage * stage_bytes;
                const int32_t y = (int32_t)(t * kWRows);
                tc::mbar_arrive_expect_tx(&bars->full[stage], (uint32_t)stage_bytes);
                for (int b = 0; b < zboxes; ++b) tc::tma_load_2d(base + b * kBoxW, &mapZ, b * 64, y, &bars->full[stage]);
                for (int b = 0; b < NC; ++b)
                    tc::tma_load_2d(base + (zboxes + b) * kBoxW, &mapG, b * 64, y, &bars->full[stage]);
                if (relu)
                    for (int b = 0; b < NC; ++b)
                        tc::tma_load_2d(base + (zboxes + NC + b) * kBoxW, &mapH, b * 64, y, &bars->full[stage]);
                issued |= 1u << stage;
                issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!ok) {
                int dummy = 0;
                for (int s = 0; s < stages; ++s)
                    if (issued & (1u << s))
                        tc::mbar_wait(&bars->full[s], (issued_parity >> s) & 1u, (volatile int *)&dummy);
            }
        }
    } else if (warp >= 6) {
        const int tid = threadIdx.x - 192;
        int stage = 0;
        uint32_t phase = 0;
        for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
            if (!tc::mbar_wait(&bars->full[stage], phase, abort_flag)) break;
            uint8_t *base = smem + stage * stage_bytes;
            if (relu) mask_tile(base + zboxes * kBoxW, base + (zboxes + NC) * kBoxW, NC * kBoxW, tid);
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars->ready[stage]);
            if (++stage == stages) {
                stage = 0;
                phase ^= 1u;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16(128, N_pad, 1, 1);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true, first = true;
            for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x) {
                if (!tc::mbar_wait(&bars->ready[stage], phase, abort_flag)) {
                    ok = false;
                    break;
                }
                tc::tc_fence_after();
                const uint32_t zb = tc::smem_u32(smem + stage * stage_bytes);
                const uint32_t gb = zb + (uint32_t)(zboxes * kBoxW);
                for (int mb = 0; mb < MB; ++mb) {
#pragma unroll
                    for (int kk = 0; kk < kWRows / 16; ++kk) {
                        const uint64_t a = tc::sw128_desc(zb + mb * 2 * kBoxW + kk * 2048, kBoxW, 1024);
                        const uint64_t b = tc::sw128_desc(gb + kk * 2048, kBoxW, 1024);
                        tc::mma_bf16(tmem_base + (uint32_t)(mb * N_pad), a, b, idesc, (first && kk == 0) ? 0u : 1u);
                    }
                }
                first = false;
                tc::mma_commit(&bars->empty[stage]);
                if (++stage == stages) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            tc::mma_commit(ok ? &bars->tfull[0] : &bars->drain);
            if (!ok) {
                int dummy = 0;
                tc::mbar_wait(&bars->drain, 0, (volatile int *)&dummy);
            }
        }
    } else {
        const int q = warp & 3;
        const int64_t cta = blockIdx.x;
        float *P = partial + cta * (int64_t)Kp * N;
        const bool have = (int64_t)blockIdx.x < n_tiles;
        if (have && tc::mbar_wait(&bars->tfull[0], 0, abort_flag)) {
            tc::tc_fence_after();
            for (int mb = 0; mb < MB; ++mb) {
                const int k = mb * 128 + q * 32 + lane;
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(mb * N_pad);
                for (int c = 0; c < N_pad; c += 16) {
                    uint32_t r[16];
                    tc::tmem_ld16(taddr + (uint32_t)c, r);
                    if (k < Kp)
                        for (int i = 0; i < 16 && c + i < N; ++i) P[(int64_t)k * N + c + i] = __uint_as_float(r[i]);
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && bars->abort_flag) atomicOr(err, kErrWaitTc);
    if (warp == 1) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem_base, ncols);
    }
}

__global__ void pack_wk_bf16_kernel(const float *__restrict__ Wp, int64_t ldw, int64_t Kp, int64_t N, int64_t Kp_pad,
                                    int64_t N_pad, __nv_bfloat16 *__restrict__ Wk) {
    // Wk[k][n] = W[k][n]: rows k (the dgrad output columns), n contiguous
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= Kp_pad * N_pad) return;
    int64_t k = x / N_pad, n = x % N_pad;
    Wk[x] = __float2bfloat16_rn((k < Kp && n < N) ? Wp[k * ldw + n] : 0.f);
}

__global__ void sum_partials_kernel(const float *__restrict__ P, int64_t parts, int64_t KN, float *__restrict__ out) {
    int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= KN) return;
    double s = 0.0;
    for (int64_t q = 0; q < parts; ++q) s += (double)P[q * KN + x];
    out[x] = (float)s;
}

// dY = bf16(relu ? G * 1[H_out > 0] : G), eight columns per thread (two 16-byte
// loads of G, one of H_out, one 16-byte store); the group that straddles N
// reads element by element, and columns [N, ld_y) are written as zero.
__global__ void grad_to_bf16_kernel(const float *__restrict__ G, int64_t ld_g, const __nv_bfloat16 *__restrict__ H,
                                    int64_t ld_h, int64_t n, int64_t N, int64_t groups, __nv_bfloat16 *__restrict__ Y,
                                    int64_t ld_y) {
    const int64_t x = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (x >= n * groups) return;
    const int64_t r = x / groups, c0 = (x % groups) * 8;
    const float *g = G + r * ld_g + c0;
    float v[8];
    if (c0 + 8 <= N) {
        const float4 a = *reinterpret_cast<const float4 *>(g), b = *reinterpret_cast<const float4 *>(g + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = c0 + k < N ? g[k] : 0.f;
    }
    if (H) {
        const uint4 h = *reinterpret_cast<const uint4 *>(H + r * ld_h + c0);  // c0 + 8 <= ld_h: ld_h is a multiple of 8
        const uint32_t hw[4] = {h.x, h.y, h.z, h.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            if (!(__uint_as_float(hw[k] << 16) > 0.f)) v[2 * k] = 0.f;
            if (!(__uint_as_float(hw[k] & 0xffff0000u) > 0.f)) v[2 * k + 1] = 0.f;
        }
    }
    *reinterpret_cast<uint4 *>(Y + r * ld_y + c0) =
        make_uint4(pack2(v[0], v[1]), pack2(v[2], v[3]), pack2(v[4], v[5]), pack2(v[6], v[7]));
}

struct BwdPlan {
    int64_t Kp_pad, N_pad, NC, MB;
    int dstages, wstages;
    size_t dsmem, wsmem;
};

bool plan_bwd(int64_t Kp, int64_t N, int relu, BwdPlan *p) {
    p->Kp_pad = round_up(Kp, 16);
    p->N_pad = round_up(N, 16);
    p->NC = ceil_div(N, 64);
    p->MB = ceil_div(Kp, 128);
    if (p->Kp_pad > 256 || p->N_pad > 256 || p->MB * p->N_pad > 512) return false;
    const size_t bars = sizeof(BarsB) + 1024;
    // dgrad: resident W (NC chunks of Kp_pad x 64) + stages of G (+ H)
    const size_t wbytes = (size_t)p->NC * p->Kp_pad * 128;
    const size_t dstage = (size_t)kBoxD * (relu ? 2 : 1);
    if (wbytes + 2 * dstage + kOutBytes + bars > kSmemLimitB) return false;
    int ds = (int)((kSmemLimitB - wbytes - kOutBytes - bars) / dstage);
    p->dstages = ds > kMaxStagesB ? kMaxStagesB : ds;
    p->dsmem = wbytes + p->dstages * dstage + kOutBytes + bars;
    // wgrad: stages of Z (2 MB boxes) + G (NC) (+ H (NC))
    const size_t wstage = (size_t)kBoxW * (2 * p->MB + p->NC * (relu ? 2 : 1));
    if (2 * wstage + bars > kSmemLimitB) return false;
    int ws = (int)((kSmemLimitB - bars) / wstage);
    p->wstages = ws > kMaxStagesB ? kMaxStagesB : ws;
    p->wsmem = p->wstages * wstage + bars;
    return true;
}

}  // namespace

gnn_status launch_grad_to_bf16(const float *G, int64_t ld_g, const void *Hout, int64_t ld_h, int64_t n, int64_t N,
                               void *Y, int64_t ld_y, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    if (ld_y % 8 != 0 || ld_y < N) return GNN_EINVAL;
    const int64_t groups = ld_y / 8;
    { grad_to_bf16_kernel<<<(unsigned)ceil_div(n * groups, 256), 256, 0, s>>>(
        G, ld_g, static_cast<const __nv_bfloat16 *>(Hout), ld_h, n, N, groups, static_cast<__nv_bfloat16 *>(Y),
        ld_y); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

namespace {

// columns of Z (rows of W and dW) per pass: all Kp, or slices of 256 when the
// wgrad accumulator or the dgrad's resident W of the whole Kp does not fit; the
// slices are independent (dZ[:, k0:k1] = dY W[k0:k1]^T, dW[k0:k1] = Z[:, k0:k1]^T dY)
constexpr int64_t kKSlice = 256;
int64_t bwd_slice(int64_t Kp, int64_t N) {
    BwdPlan p;
    if (plan_bwd(Kp, N, 1, &p)) return Kp;
    if (Kp > kKSlice && plan_bwd(kKSlice, N, 1, &p)) return kKSlice;
    return 0;
}

gnn_status bwd_tc_pass(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                       int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N, float *dWp,
                       void *dZ, int64_t ld_dz, bool dz_f32, void *ws, int *err, cudaStream_t s);

}  // namespace

bool update_bwd_tc_supported(int64_t Kp, int64_t N) { return bwd_slice(Kp, N) > 0; }

size_t update_bwd_tc_ws_bytes(int64_t n, int64_t Kp_all, int64_t N) {
    const int64_t ks = bwd_slice(Kp_all, N);
    const int64_t Kp = ks > 0 ? ks : Kp_all;
    const int64_t tiles = ceil_div(n, kWRows);
    const int64_t grid = tiles < num_sms() ? tiles : num_sms();
    const int64_t kpad = round_up(Kp, 16), npad = round_up(N, 16);
    return (size_t)grid * Kp * N * sizeof(float) + 256 + (size_t)kpad * npad * 2;
}

gnn_status launch_update_bwd_tc(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                                int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N,
                                float *dWp, void *dZ, int64_t ld_dz, bool dz_f32, void *ws, int *err, cudaStream_t s) {
    const int64_t ks = bwd_slice(Kp, N);
    if (ks <= 0) return GNN_EUNSUPPORTED;
    const int64_t dzb = dz_f32 ? 4 : 2;
    for (int64_t k0 = 0; k0 < Kp; k0 += ks) {
        const gnn_status st = bwd_tc_pass(
            G, ld_g, Hout, ld_h, relu, Z ? static_cast<const char *>(Z) + k0 * 2 : nullptr, ld_z, n,
            Kp - k0 < ks ? Kp - k0 : ks, Wp + k0 * ld_w, ld_w, N, dWp ? dWp + k0 * N : nullptr,
            dZ ? static_cast<char *>(dZ) + k0 * dzb : nullptr, ld_dz, dz_f32, ws, err, s);
        if (st != GNN_OK) return st;
    }
    return GNN_OK;
}

namespace {

gnn_status bwd_tc_pass(const void *G, int64_t ld_g, const void *Hout, int64_t ld_h, int relu, const void *Z,
                       int64_t ld_z, int64_t n, int64_t Kp, const float *Wp, int64_t ld_w, int64_t N, float *dWp,
                       void *dZ, int64_t ld_dz, bool dz_f32, void *ws, int *err, cudaStream_t s) {
    BwdPlan p;
    if (!plan_bwd(Kp, N, relu, &p)) return GNN_EUNSUPPORTED;
    if (n == 0) {
        if (dWp) GNN_CUDA_TRY(cudaMemsetAsync(dWp, 0, (size_t)Kp * N * sizeof(float), s));
        return GNN_OK;
    }
    const int64_t wtiles = ceil_div(n, kWRows);
    const int64_t wgrid = wtiles < num_sms() ? wtiles : num_sms();
    float *partial = static_cast<float *>(ws);
    __nv_bfloat16 *Wk = reinterpret_cast<__nv_bfloat16 *>(static_cast<char *>(ws) +
                                                          round_up((int64_t)wgrid * Kp * N * 4, 256));
    CUtensorMap mG, mH, mZ, mW;
    // wgrad (skipped when dWp is null: dZ only)
    if (dWp) {
        if (!make_map_bf16_2d(&mZ, Z, (uint64_t)Kp, (uint64_t)n, (uint64_t)ld_z * 2, 64, kWRows)) return GNN_ECUDA;
        if (!make_map_bf16_2d(&mG, G, (uint64_t)N, (uint64_t)n, (uint64_t)ld_g * 2, 64, kWRows)) return GNN_ECUDA;
        if (!make_map_bf16_2d(&mH, relu ? Hout : G, (uint64_t)N, (uint64_t)n, (uint64_t)(relu ? ld_h : ld_g) * 2, 64,
                              kWRows))
            return GNN_ECUDA;
        GNN_CUDA_TRY(cudaFuncSetAttribute(update_wgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          (int)p.wsmem));
        { update_wgrad_tc_kernel<<<(unsigned)wgrid, kThreadsB, p.wsmem, s>>>(mZ, mG, mH, partial, n, (int)Kp, (int)p.MB,
                                                                            (int)N, (int)p.N_pad, (int)p.NC, p.wstages,
                                                                            relu, wtiles, err); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        { sum_partials_kernel<<<(unsigned)ceil_div(Kp * N, 256), 256, 0, s>>>(partial, wgrid, Kp * N, dWp);
          GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
    }
    if (!dZ) return GNN_OK;
    // dgrad
    { pack_wk_bf16_kernel<<<(unsigned)ceil_div(p.Kp_pad * p.N_pad, 256), 256, 0, s>>>(Wp, ld_w, Kp, N, p.Kp_pad,
                                                                                     p.N_pad, Wk); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    if (!make_map_bf16_2d(&mG, G, (uint64_t)N, (uint64_t)n, (uint64_t)ld_g * 2, 64, kDRows)) return GNN_ECUDA;
    if (!make_map_bf16_2d(&mH, relu ? Hout : G, (uint64_t)N, (uint64_t)n, (uint64_t)(relu ? ld_h : ld_g) * 2, 64,
                          kDRows))
        return GNN_ECUDA;
    if (!make_map_bf16_2d(&mW, Wk, (uint64_t)p.N_pad, (uint64_t)p.Kp_pad, (uint64_t)p.N_pad * 2, 64,
                          (uint32_t)p.Kp_pad))
        return GNN_ECUDA;
    CUtensorMap mO;
    if (dz_f32 ? !make_map_f32_2d(&mO, dZ, (uint64_t)Kp, (uint64_t)n, (uint64_t)ld_dz * 4, 32, 32)
               : !make_map_bf16_2d(&mO, dZ, (uint64_t)Kp, (uint64_t)n, (uint64_t)ld_dz * 2, 64, 32))
        return GNN_ECUDA;
    GNN_CUDA_TRY(cudaFuncSetAttribute(update_dgrad_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      (int)p.dsmem));
    const int64_t dtiles = ceil_div(n, kDRows);
    const int64_t dgrid = dtiles < num_sms() ? dtiles : num_sms();
    { update_dgrad_tc_kernel<<<(unsigned)dgrid, kThreadsB, p.dsmem, s>>>(
        mG, mH, mW, mO, (int)p.Kp_pad, (int)p.NC, p.dstages, relu, dz_f32 ? 1 : 0, dtiles, err); GNN_LAUNCHED(1); }
    GNN_CUDA_TRY(cudaGetLastError());
    return GNN_OK;
}

}  // namespace

}  // namespace gnn
