// codec.cu - the low-bit halo codec of the Sylvie page ("Sylvie: 3D-Adaptive
// and Universal System for Large-Scale Graph Neural Network Training",
// Quantizer and Dequantizer), fused into push and pull.
//
// Push side (quantiser): every pushed row h of f values becomes f b-bit codes
// (b = 1, 2, 4 or 8, B = 2^b - 1 bins) plus two fp32 numbers, the scale
// s = (max(h) - min(h)) / B and the zero point min(h).  A code is the
// stochastic rounding of (h[c] - min) / s: floor of that value plus a uniform
// draw u in [0, 1), kept in [0, B]; a row with s = 0 gets code 0 throughout.
// Pull side (dequantiser): the halo row is recovered as code * s + min.
//
// The draws come from a counter-based generator, SplitMix64 (Steele, Lea and
// Flood, OOPSLA 2014): element c of table row r uses output k = r * 2^14 +
// c / 4 + 1 of the stream seeded with the caller's seed, bits 48..63, 32..47,
// 16..31 or 0..15 for c % 4 = 0, 1, 2, 3, as a 16-bit fraction.  All
// arithmetic is IEEE single precision with one rounding per operation
// (explicit _rn intrinsics, nothing fused), the division by s taken as a
// multiplication by the row's rounded reciprocal 1 / s, so the codes depend
// on the inputs and the seed only.
//
// Layout: codes of table row r at codes + r * ld_codes (bytes, a multiple of
// 16), code c in bits [c * b, c * b + b) little-endian, bytes past the last
// code zero; (scale, zero point) at scale_zero[2 r], scale_zero[2 r + 1].
//
// Quantiser: rows of up to 256 values take eight lanes each (four rows per
// warp), lane g owning 8, 16 or 32 consecutive values; wider rows take one
// warp each, lane l owning the 8 consecutive values 8 l + 256 j, so its codes
// of a 256-value chunk are one b-byte word.  Dequantiser: one warp per row
// (the pull's grid of 16 blocks per SM loops over the rows).
#include <algorithm>

#include "gnn_internal.cuh"

namespace gnn {

namespace {

// SplitMix64 (Steele, Lea and Flood): draw k of the stream `seed` is the
// finaliser applied to seed + k * gamma
constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
__device__ __forceinline__ uint64_t splitmix64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// the 8 values c0 .. c0 + 7 of a row as fp32 (exact widening); values at or
// past f are not read and come back as 0
__device__ __forceinline__ void load8(const float *row, int c0, int f, float (&v)[8]) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = a;
    if (c0 < f) a = __ldg(reinterpret_cast<const float4 *>(row + c0));
    if (c0 + 4 < f) b = __ldg(reinterpret_cast<const float4 *>(row + c0 + 4));
    v[0] = a.x, v[1] = a.y, v[2] = a.z, v[3] = a.w, v[4] = b.x, v[5] = b.y, v[6] = b.z, v[7] = b.w;
}
__device__ __forceinline__ void load8(const __nv_bfloat16 *row, int c0, int f, float (&v)[8]) {
    uint4 q = make_uint4(0u, 0u, 0u, 0u);
    if (c0 < f) q = __ldg(reinterpret_cast<const uint4 *>(row + c0));
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        v[2 * k] = __uint_as_float(w[k] << 16);
        v[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
}

// store the values of c0 .. c0 + 7 that lie below f
__device__ __forceinline__ void store8(float *row, int c0, int f, const float (&v)[8]) {
    if (c0 + 8 <= f) {
        reinterpret_cast<float4 *>(row + c0)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(row + c0)[1] = make_float4(v[4], v[5], v[6], v[7]);
    } else {
        for (int k = 0; k < 8 && c0 + k < f; ++k) row[c0 + k] = v[k];
    }
}
__device__ __forceinline__ void store8(__nv_bfloat16 *row, int c0, int f, const float (&v)[8]) {
    if (c0 + 8 <= f) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(row + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    } else {
        for (int k = 0; k < 8 && c0 + k < f; ++k) row[c0 + k] = __float2bfloat16_rn(v[k]);
    }
}

// the b-byte word holding the codes of 8 values (code k in bits k*b ..)
template <int BITS>
struct CodeWord;
template <>
struct CodeWord<1> {
    using type = uint8_t;
};
template <>
struct CodeWord<2> {
    using type = uint16_t;
};
template <>
struct CodeWord<4> {
    using type = uint32_t;
};
template <>
struct CodeWord<8> {
    using type = unsigned long long;
};


// packed IEEE single-precision pairs (two independent roundings, the same
// results as two scalar _rn operations)
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
    return ((unsigned long long)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ unsigned long long sub2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long mul2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// the codes of the 8 values x of a lane's piece (columns c0 .. c0 + 7 of the
// row, the draws of the row starting at z_row): t = (x - mn) * inv, plus a
// 16-bit uniform, floored and kept in [0, B]; codes past column f are 0.
// FINITE: the row's values, its scale and its reciprocal are finite, so every
// sum of a value inside the row is a number >= 0 and the floor needs no test
// (a value past f may give any code; it is cleared).
template <int BITS, bool FINITE>
__device__ __forceinline__ typename CodeWord<BITS>::type encode8(const float (&x)[8], int c0, int f, float mn,
                                                                 float inv, uint64_t z_row) {
    using W = typename CodeWord<BITS>::type;
    constexpr int B = (1 << BITS) - 1;
    const uint64_t zz[2] = {splitmix64_mix(z_row + (uint64_t)(c0 >> 2) * kGamma),
                            splitmix64_mix(z_row + (uint64_t)((c0 >> 2) + 1) * kGamma)};
    const unsigned long long mn2 = pack2(mn, mn), inv2 = pack2(inv, inv), one2 = pack2(1.0f, 1.0f);
    W word = 0;
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        // 16 bits of the draw as the fraction bits of 1.x, minus 1: u16 / 2^16, exact
        const uint32_t w0 = (uint32_t)(zz[e >> 2] >> (48 - 16 * (e & 3))) & 0xffffu;
        const uint32_t w1 = (uint32_t)(zz[e >> 2] >> (32 - 16 * (e & 3))) & 0xffffu;
        const unsigned long long u2 =
            sub2(pack2(__uint_as_float(0x3f800000u | (w0 << 7)), __uint_as_float(0x3f800000u | (w1 << 7))), one2);
        const unsigned long long v2 = add2(mul2(sub2(pack2(x[e], x[e + 1]), mn2), inv2), u2);
        const float v[2] = {__uint_as_float((uint32_t)v2), __uint_as_float((uint32_t)(v2 >> 32))};
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            int q;
            if constexpr (FINITE) {
                q = __float2int_rd(v[k]);
            } else {
                q = v[k] >= 0.f ? __float2int_rd(v[k]) : 0;  // not a number: 0
            }
            q = q > B ? B : q;
            word |= (W)(uint32_t)q << ((e + k) * BITS);
        }
    }
    const int valid = f - c0;
    if (valid < 8) word &= (W)(((W)1 << (valid * BITS)) - 1);
    return word;
}

// quantise one row h into its codes and (scale, zero point); one warp.  x0 is
// the lane's first piece (load8 of columns 8 lane ..; all of a row of up to
// 256 values), loaded by the caller and kept in registers for both passes.
template <typename T, int BITS>
__device__ __forceinline__ void quantize_row(const T *__restrict__ h, const float (&x0)[8], int64_t id,
                                             uint8_t *__restrict__ crow, int64_t ld_codes, float *__restrict__ sz,
                                             int64_t f64, uint64_t seed, int lane) {
    using W = typename CodeWord<BITS>::type;
    constexpr int B = (1 << BITS) - 1;
    const int f = (int)f64;  // a row's width fits 32 bits
    // min and max of the row
    float mn = INFINITY, mx = -INFINITY;
    if (lane * 8 + 8 <= f) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            mn = fminf(mn, x0[k]);
            mx = fmaxf(mx, x0[k]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (lane * 8 + k < f) {
                mn = fminf(mn, x0[k]);
                mx = fmaxf(mx, x0[k]);
            }
    }
    for (int c0 = lane * 8 + 256; c0 < f; c0 += 256) {
        float x[8];
        load8(h, c0, f, x);
#pragma unroll
        for (int k = 0; k < 8; ++k)
            if (c0 + k < f) {
                mn = fminf(mn, x[k]);
                mx = fmaxf(mx, x[k]);
            }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)B);
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;  // the rounded reciprocal 1 / s
    const int used = (f + 7) / 8 * BITS;             // code bytes of the row (whole 8-value words)
    // value c of the row takes bits of draw (id << 14) + c / 4 + 1
    const uint64_t z_row = seed + (((uint64_t)id << 14) + 1u) * kGamma;
    const bool finite = isfinite(mn) && isfinite(mx) && isfinite(inv);  // the same for the whole warp
    auto encode = [&](const float (&x)[8], int c0) -> W {
        if (!(s > 0.f)) return (W)0;
        return finite ? encode8<BITS, true>(x, c0, f, mn, inv, z_row) : encode8<BITS, false>(x, c0, f, mn, inv, z_row);
    };
    if (lane * 8 < f) *reinterpret_cast<W *>(crow + lane * BITS) = encode(x0, lane * 8);
    for (int c0 = lane * 8 + 256; c0 < f; c0 += 256) {
        float x[8];
        load8(h, c0, f, x);
        *reinterpret_cast<W *>(crow + c0 / 8 * BITS) = encode(x, c0);
    }
    // bytes past the codes are zero
    for (int64_t b = used + lane; b < ld_codes; b += 32) crow[b] = 0;
    if (lane == 0) {
        sz[0] = s;
        sz[1] = mn;
    }
}

// Quantise pushed rows: row v of H goes to table row ids[v] if the push checks
// passed it (id in range and seen once; else the row is skipped).
template <typename T, int BITS>
__global__ void __launch_bounds__(256) codec_push_kernel(const T *__restrict__ H, int64_t ld_h,
                                                         const int64_t *__restrict__ ids, int64_t n,
                                                         const uint8_t *__restrict__ ok, uint8_t *__restrict__ codes,
                                                         int64_t ld_codes, float *__restrict__ scale_zero, int64_t f,
                                                         uint64_t seed) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t v = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; v < n; v += nw) {
        // the row's values do not depend on its id: their load overlaps the id and claim-word loads
        float x0[8];
        load8(H + v * ld_h, lane * 8, (int)f, x0);
        if (!ok[v]) continue;  // id out of range or repeated (reported by the checks)
        const int64_t id = ids[v];
        quantize_row<T, BITS>(H + v * ld_h, x0, id, codes + id * ld_codes, ld_codes, scale_zero + 2 * id, f, seed,
                              lane);
    }
}

// ---- rows of at most 256 values: eight lanes per row ----------------------
// A group of 8 lanes quantises one row, so a warp takes four rows at once and
// the per-row work (the min / max reduction, the scale and its reciprocal, the
// id and draw offset) is shared by four rows.  Lane g of a group owns the
// R = 8 NC consecutive values g R .. g R + R - 1 (NC = 1, 2, 4: rows of up to
// 64, 128, 256 values) and their R b-bit codes, R b / 8 contiguous bytes.

// 2^23: for 0 <= v < 2^23, v + 2^23 rounded toward -inf is 2^23 + floor(v),
// whose bits are kFloorBias + floor(v)
constexpr uint32_t kFloorBias = 0x4B000000u;

__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b, unsigned long long c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}
__device__ __forceinline__ unsigned long long add2_rm(unsigned long long a, unsigned long long b) {
    unsigned long long d;
    asm("add.rm.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
// three-input minimum / maximum (NaN inputs ignored, as fminf / fmaxf)
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float d;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

template <int BITS, int NC>
struct LaneCodes {
    static constexpr int R = 8 * NC;                          // values of a lane
    static constexpr int NBYTES = R * BITS / 8;               // their code bytes
    static constexpr int NW = NBYTES >= 4 ? NBYTES / 4 : 1;   // 32-bit words holding them
};

// sum over the codes in word w of kFloorBias << (code's bit offset), mod 2^32
__host__ __device__ constexpr uint32_t floor_bias_word(int w, int bits, int r) {
    uint32_t b = 0;
    for (int i = 0; i < r; ++i)
        if ((i * bits) >> 5 == w) b += kFloorBias << ((i * bits) & 31);
    return b;
}

// codes of a lane's R values x (columns c0 .. c0 + R - 1 of the row) when the
// row's values, scale and reciprocal are finite and s > 0: every
// t = (x - mn) * inv and v = t + u then lies in [0, 2^23), so floor(v) is the
// low mantissa of v + 2^23 rounded down; the words accumulate
// (kFloorBias + min(floor(v), B)) << offset and start at minus the biases
template <int BITS, int NC>
__device__ __forceinline__ void encode_lane(const float (&x)[8 * NC], int c0, float mn, float inv, uint64_t z_row,
                                            uint32_t (&acc)[LaneCodes<BITS, NC>::NW]) {
    constexpr int B = (1 << BITS) - 1;
    constexpr int R = LaneCodes<BITS, NC>::R;
#pragma unroll
    for (int w = 0; w < LaneCodes<BITS, NC>::NW; ++w) acc[w] = 0u - floor_bias_word(w, BITS, R);
    const unsigned long long mn2 = pack2(mn, mn), inv2 = pack2(inv, inv);
    const unsigned long long big2 = pack2(8388608.0f, 8388608.0f), frac2 = pack2(1.0f / 65536.0f, 1.0f / 65536.0f);
#pragma unroll
    for (int d = 0; d < 2 * NC; ++d) {
        // draw d serves values 4d .. 4d + 3 through its bits 48..63, 32..47,
        // 16..31, 0..15; each 16-bit w is placed as the float 2^23 + w
        const uint64_t z = splitmix64_mix(z_row + (uint64_t)((c0 >> 2) + d) * kGamma);
        const uint32_t half[2] = {(uint32_t)(z >> 32), (uint32_t)z};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int i = 4 * d + 2 * h;
            const unsigned long long w2 = sub2(pack2(__uint_as_float(__byte_perm(half[h], kFloorBias, 0x7632)),
                                                     __uint_as_float(__byte_perm(half[h], kFloorBias, 0x7610))),
                                               big2);                          // the draws w, exact
            const unsigned long long t2 = mul2(sub2(pack2(x[i], x[i + 1]), mn2), inv2);
            const unsigned long long v2 = fma2(w2, frac2, t2);             // t + w / 2^16, one rounding
            const unsigned long long r2 = add2_rm(v2, big2);               // 2^23 + floor(v)
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const uint32_t qb = min(k ? (uint32_t)(r2 >> 32) : (uint32_t)r2, kFloorBias + (uint32_t)B);
                const int p = (i + k) * BITS;
                acc[p >> 5] += qb << (p & 31);
            }
        }
    }
}

// the NBYTES code bytes of a lane, one aligned store
template <int NBYTES, int NW>
__device__ __forceinline__ void store_lane_codes(uint8_t *p, const uint32_t (&acc)[NW]) {
    if constexpr (NBYTES == 1) {
        *p = (uint8_t)acc[0];
    } else if constexpr (NBYTES == 2) {
        *reinterpret_cast<uint16_t *>(p) = (uint16_t)acc[0];
    } else if constexpr (NBYTES == 4) {
        *reinterpret_cast<uint32_t *>(p) = acc[0];
    } else if constexpr (NBYTES == 8) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(acc[0], acc[1]);
    } else {
#pragma unroll
        for (int q = 0; q < NBYTES / 16; ++q)
            reinterpret_cast<uint4 *>(p)[q] = make_uint4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    }
}

// the lane's R values of row h (zeros for a row that is not there)
template <typename T, int NC>
__device__ __forceinline__ void load_lane(const T *h, bool in, int c0, int f, float (&x)[8 * NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        float y[8];
        if (in) {
            load8(h, c0 + 8 * j, f, y);
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) y[k] = 0.f;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) x[8 * j + k] = y[k];
    }
}

// quantise the row of this lane's group (x: the lane's values, loaded by
// load_lane); every lane of the warp calls it, `live` says whether the
// group's row is quantised and stored
template <int BITS, int NC, int G>
__device__ __forceinline__ void quantize_row_group(float (&x)[8 * NC], bool live, int64_t id,
                                                   uint8_t *__restrict__ crow, int64_t ld_codes,
                                                   float *__restrict__ sz, int f, uint64_t seed, int g) {
    using L = LaneCodes<BITS, NC>;
    constexpr int B = (1 << BITS) - 1;
    constexpr int R = L::R;
    const int c0 = g * R;
    const bool full = c0 + R <= f;
    float mn = INFINITY, mx = -INFINITY;
    if (full) {
#pragma unroll
        for (int k = 0; k + 1 < R; k += 2) {
            mn = min3f(mn, x[k], x[k + 1]);
            mx = max3f(mx, x[k], x[k + 1]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < R; ++k)
            if (c0 + k < f) {
                mn = fminf(mn, x[k]);
                mx = fmaxf(mx, x[k]);
            }
    }
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) {
        mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if (!live) return;
    const float s = __fdiv_rn(__fsub_rn(mx, mn), (float)B);
    const float inv = s > 0.f ? __frcp_rn(s) : 0.f;  // the rounded reciprocal 1 / s
    if (c0 < f) {
        uint32_t acc[L::NW];
        if (s > 0.f) {
            // value c of the row takes bits of draw (id << 14) + c / 4 + 1
            const uint64_t z_row = seed + (((uint64_t)id << 14) + 1u) * kGamma;
            if (isfinite(mn) && isfinite(mx) && isfinite(s) && isfinite(inv)) {
                if (!full) {
#pragma unroll
                    for (int k = 0; k < R; ++k) x[k] = c0 + k < f ? x[k] : mn;  // code 0 past the row
                }
                encode_lane<BITS, NC>(x, c0, mn, inv, z_row, acc);
            } else {
#pragma unroll
                for (int w = 0; w < L::NW; ++w) acc[w] = 0u;
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    if (c0 + 8 * j >= f) break;
                    float y[8];
#pragma unroll
                    for (int k = 0; k < 8; ++k) y[k] = x[8 * j + k];
                    const unsigned long long word =
                        (unsigned long long)encode8<BITS, false>(y, c0 + 8 * j, f, mn, inv, z_row);
                    const int p = j * 8 * BITS;  // a chunk's 8 b bits never straddle a word unless b = 8
                    acc[p >> 5] |= (uint32_t)word << (p & 31);
                    if constexpr (BITS == 8) acc[(p >> 5) + 1] = (uint32_t)(word >> 32);
                }
            }
        } else {
#pragma unroll
            for (int w = 0; w < L::NW; ++w) acc[w] = 0u;
        }
        if (full) {
            store_lane_codes<L::NBYTES, L::NW>(crow + g * L::NBYTES, acc);
        } else {
            // the bytes of the chunks that hold values of the row
            const int nb = ((f - c0 + 7) / 8) * BITS;
#pragma unroll
            for (int b = 0; b < L::NBYTES; ++b)
                if (b < nb) crow[g * L::NBYTES + b] = (uint8_t)(acc[b >> 2] >> ((b & 3) * 8));
        }
    }
    // bytes past the codes are zero
    for (int64_t b = (f + 7) / 8 * BITS + g; b < ld_codes; b += G) crow[b] = 0;
    if (g == 0) {
        sz[0] = s;
        sz[1] = mn;
    }
}

// resident blocks of 256 threads per SM the grouped kernels are compiled for
// (at most 64 registers: the loads of four rows per warp are latency-bound,
// and 116 registers with two blocks per SM took 2.95 ms instead of 1.84)
constexpr int kGroupBlocks = 4;

// The quantising push with G lanes per row (rows of at most 8 NC G values).
template <typename T, int BITS, int NC, int G>
__global__ void __launch_bounds__(256, kGroupBlocks) codec_push_group_kernel(const T *__restrict__ H, int64_t ld_h,
                                                                             const int64_t *__restrict__ ids, int64_t n,
                                                                             const uint8_t *__restrict__ ok,
                                                                             uint8_t *__restrict__ codes,
                                                                             int64_t ld_codes,
                                                                             float *__restrict__ scale_zero, int64_t f,
                                                                             uint64_t seed) {
    constexpr int RW = 32 / G;  // rows per warp
    const int lane = threadIdx.x & 31, g = lane & (G - 1);
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    // the loop is uniform over the warp (its shuffles need all 32 lanes)
    for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * RW; base < n; base += nw * RW) {
        const int64_t v = base + lane / G;
        const bool in = v < n;
        float x[8 * NC];
        load_lane<T, NC>(H + (in ? v : 0) * ld_h, in, g * 8 * NC, (int)f, x);
        // the flag and the id are loaded together (the id is read even where the flag will skip it)
        const bool live = in && ok[v];  // id in range and seen once (reported by the checks)
        const int64_t id_any = in ? ids[v] : 0;
        const int64_t id = live ? id_any : 0;
        quantize_row_group<BITS, NC, G>(x, live, id, codes + id * ld_codes, ld_codes, scale_zero + 2 * id, (int)f,
                                        seed, g);
    }
}

// Message rows with G lanes per row: row i of X into codes row i, keyed by keys[i].
template <typename T, int BITS, int NC, int G>
__global__ void __launch_bounds__(256, kGroupBlocks) quantize_rows_group_kernel(const T *__restrict__ X, int64_t ld_x,
                                                                                const int64_t *__restrict__ keys,
                                                                                int64_t n, uint8_t *__restrict__ codes,
                                                                                int64_t ld_codes,
                                                                                float *__restrict__ scale_zero,
                                                                                int64_t f, uint64_t seed) {
    constexpr int RW = 32 / G;
    const int lane = threadIdx.x & 31, g = lane & (G - 1);
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t base = (((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5) * RW; base < n; base += nw * RW) {
        const int64_t i = base + lane / G;
        const bool in = i < n;
        float x[8 * NC];
        load_lane<T, NC>(X + (in ? i : 0) * ld_x, in, g * 8 * NC, (int)f, x);
        const int64_t r = in ? i : 0;
        quantize_row_group<BITS, NC, G>(x, in, in ? keys[i] : 0, codes + r * ld_codes, ld_codes, scale_zero + 2 * r,
                                        (int)f, seed, g);
    }
}

// shape (NC values per lane / 8, G lanes per row) of the grouped kernels for
// a row width: 0 above 256 values
// (sixteen lanes per row for 256 values measured slower: 2.12 against
// 1.84 ms for 8.4M rows, the per-row work shared by two rows instead of four)
inline int group_shape(int64_t f) { return f <= 64 ? 1 : f <= 128 ? 2 : f <= 256 ? 4 : 0; }
inline int group_rows_per_warp(int) { return 4; }

template <typename F>
gnn_status dispatch_shape(int shape, F &&fn) {
    switch (shape) {
        case 1: return fn(std::integral_constant<int, 1>(), std::integral_constant<int, 8>());
        case 2: return fn(std::integral_constant<int, 2>(), std::integral_constant<int, 8>());
        case 4: return fn(std::integral_constant<int, 4>(), std::integral_constant<int, 8>());
    }
    return GNN_EINVAL;
}

// Dequantise halo rows: H[row0 + i] = code * scale + zero of table row ids[i].
template <typename T, int BITS>
__global__ void __launch_bounds__(256) codec_pull_kernel(const uint8_t *__restrict__ codes, int64_t ld_codes,
                                                         const float *__restrict__ scale_zero, int64_t n_table,
                                                         const int64_t *__restrict__ ids, int64_t n, T *__restrict__ H,
                                                         int64_t ld_h, int64_t row0, int64_t f, int *err) {
    using W = typename CodeWord<BITS>::type;
    constexpr int B = (1 << BITS) - 1;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        const int64_t id = ids[i];
        if (id < 0 || id >= n_table) {
            if (lane == 0) atomicOr(err, 1);
            continue;
        }
        const float s = __ldg(scale_zero + 2 * id), z = __ldg(scale_zero + 2 * id + 1);
        const uint8_t *crow = codes + id * ld_codes;
        T *out = H + (row0 + i) * ld_h;
        for (int c0 = lane * 8; c0 < (int)f; c0 += 256) {
            const W word = __ldg(reinterpret_cast<const W *>(crow + c0 / 8 * BITS));
            float y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int q = (int)((word >> (k * BITS)) & (W)B);
                y[k] = __fadd_rn(__fmul_rn((float)q, s), z);
            }
            store8(out, c0, (int)f, y);
        }
    }
}

// Rows as a message between processes: row i of X is quantised into codes row
// i, its draws keyed by keys[i] (the vertex's global id) as a table row would be
template <typename T, int BITS>
__global__ void __launch_bounds__(256) quantize_rows_kernel(const T *__restrict__ X, int64_t ld_x,
                                                            const int64_t *__restrict__ keys, int64_t n,
                                                            uint8_t *__restrict__ codes, int64_t ld_codes,
                                                            float *__restrict__ scale_zero, int64_t f, uint64_t seed) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        float x0[8];
        load8(X + i * ld_x, lane * 8, (int)f, x0);
        quantize_row<T, BITS>(X + i * ld_x, x0, keys[i], codes + i * ld_codes, ld_codes, scale_zero + 2 * i, f, seed,
                              lane);
    }
}

// dst[ids[i]] (+)= code * scale + zero of codes row i (ids null: row i); the
// ids of one launch are distinct; the sum is fp32, stored as T
template <typename T, int BITS>
__global__ void __launch_bounds__(256) dequantize_rows_kernel(const uint8_t *__restrict__ codes, int64_t ld_codes,
                                                              const float *__restrict__ scale_zero, int64_t n,
                                                              const int64_t *__restrict__ ids, T *__restrict__ dst,
                                                              int64_t ld_dst, int64_t n_dst, int64_t f, int add,
                                                              int *err) {
    using W = typename CodeWord<BITS>::type;
    constexpr int B = (1 << BITS) - 1;
    const int lane = threadIdx.x & 31;
    const int64_t nw = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; i < n; i += nw) {
        const int64_t r = ids ? ids[i] : i;
        if (r < 0 || r >= n_dst) {
            if (lane == 0 && err) atomicOr(err, kErrIndex);
            continue;
        }
        const float s = __ldg(scale_zero + 2 * i), z = __ldg(scale_zero + 2 * i + 1);
        const uint8_t *crow = codes + i * ld_codes;
        T *out = dst + r * ld_dst;
        for (int c0 = lane * 8; c0 < (int)f; c0 += 256) {
            const W word = __ldg(reinterpret_cast<const W *>(crow + c0 / 8 * BITS));
            float y[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int q = (int)((word >> (k * BITS)) & (W)B);
                y[k] = __fadd_rn(__fmul_rn((float)q, s), z);
            }
            if (add) {
                float o[8];
                load8(out, c0, (int)f, o);
#pragma unroll
                for (int k = 0; k < 8; ++k) y[k] = __fadd_rn(o[k], y[k]);
            }
            store8(out, c0, (int)f, y);
        }
    }
}

template <typename F>
gnn_status dispatch_bits(int bits, F &&fn) {
    switch (bits) {
        case 1: return fn(std::integral_constant<int, 1>());
        case 2: return fn(std::integral_constant<int, 2>());
        case 4: return fn(std::integral_constant<int, 4>());
        case 8: return fn(std::integral_constant<int, 8>());
    }
    return GNN_EINVAL;
}

}  // namespace

gnn_status launch_codec_push(gnn_graph *g, const void *H, int64_t ld_h, int64_t n_rows, int64_t f, const int64_t *ids,
                             uint8_t *codes, int64_t ld_codes, float *scale_zero, int64_t n_table, int bits,
                             uint64_t seed, gnn_dtype dt, cudaStream_t s) {
    if (n_rows == 0) return GNN_OK;
    gnn_status st = launch_push_checks(g, ids, n_rows, n_table, s);
    if (st != GNN_OK) return st;
    // one warp per row (eight lanes per row up to 256 values): the
    // quantisation is arithmetic-heavy and a bounded grid looping over the
    // rows measured slower
    const int shape = group_shape(f);
    const unsigned blocks =
        (unsigned)ceil_div(shape ? ceil_div(n_rows, group_rows_per_warp(shape)) * 32 : n_rows * 32, 256);
    return dispatch_bits(bits, [&](auto Bc) -> gnn_status {
        constexpr int BITS = decltype(Bc)::value;
        if (shape)
            return dispatch_shape(shape, [&](auto Cc, auto Gc) -> gnn_status {
                constexpr int NC = decltype(Cc)::value, G = decltype(Gc)::value;
                if (dt == GNN_BF16)
                    { codec_push_group_kernel<__nv_bfloat16, BITS, NC, G><<<blocks, 256, 0, s>>>(
                        static_cast<const __nv_bfloat16 *>(H), ld_h, ids, n_rows, g->push_ok, codes, ld_codes,
                        scale_zero, f, seed); GNN_LAUNCHED(1); }
                else
                    { codec_push_group_kernel<float, BITS, NC, G><<<blocks, 256, 0, s>>>(
                        static_cast<const float *>(H), ld_h, ids, n_rows, g->push_ok, codes, ld_codes, scale_zero, f,
                        seed); GNN_LAUNCHED(1); }
                GNN_CUDA_TRY(cudaGetLastError());
                return GNN_OK;
            });
        if (dt == GNN_BF16)
            { codec_push_kernel<__nv_bfloat16, BITS><<<blocks, 256, 0, s>>>(
                static_cast<const __nv_bfloat16 *>(H), ld_h, ids, n_rows, g->push_ok, codes, ld_codes, scale_zero, f,
                seed); GNN_LAUNCHED(1); }
        else
            { codec_push_kernel<float, BITS><<<blocks, 256, 0, s>>>(static_cast<const float *>(H), ld_h, ids, n_rows,
                                                                   g->push_ok, codes, ld_codes, scale_zero, f, seed); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

gnn_status launch_quantize_rows(const void *X, int64_t ld_x, int64_t n, int64_t f, const int64_t *keys, int bits,
                                uint64_t seed, uint8_t *codes, int64_t ld_codes, float *scale_zero, gnn_dtype dt,
                                cudaStream_t s) {
    if (n == 0) return GNN_OK;
    const int shape = group_shape(f);
    const unsigned blocks = (unsigned)ceil_div(shape ? ceil_div(n, group_rows_per_warp(shape)) * 32 : n * 32, 256);
    return dispatch_bits(bits, [&](auto Bc) -> gnn_status {
        constexpr int BITS = decltype(Bc)::value;
        if (shape)
            return dispatch_shape(shape, [&](auto Cc, auto Gc) -> gnn_status {
                constexpr int NC = decltype(Cc)::value, G = decltype(Gc)::value;
                if (dt == GNN_BF16)
                    { quantize_rows_group_kernel<__nv_bfloat16, BITS, NC, G><<<blocks, 256, 0, s>>>(
                        static_cast<const __nv_bfloat16 *>(X), ld_x, keys, n, codes, ld_codes, scale_zero, f, seed);
                      GNN_LAUNCHED(1); }
                else
                    { quantize_rows_group_kernel<float, BITS, NC, G><<<blocks, 256, 0, s>>>(
                        static_cast<const float *>(X), ld_x, keys, n, codes, ld_codes, scale_zero, f, seed);
                      GNN_LAUNCHED(1); }
                GNN_CUDA_TRY(cudaGetLastError());
                return GNN_OK;
            });
        if (dt == GNN_BF16)
            { quantize_rows_kernel<__nv_bfloat16, BITS><<<blocks, 256, 0, s>>>(
                static_cast<const __nv_bfloat16 *>(X), ld_x, keys, n, codes, ld_codes, scale_zero, f, seed); GNN_LAUNCHED(1); }
        else
            { quantize_rows_kernel<float, BITS><<<blocks, 256, 0, s>>>(static_cast<const float *>(X), ld_x, keys, n,
                                                                      codes, ld_codes, scale_zero, f, seed); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

gnn_status launch_dequantize_rows(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n,
                                  int64_t f, int bits, const int64_t *ids, void *dst, int64_t ld_dst, int64_t n_dst,
                                  int add, gnn_dtype dt, int *err, cudaStream_t s) {
    if (n == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n * 32, 256), (int64_t)num_sms() * 16);
    return dispatch_bits(bits, [&](auto Bc) -> gnn_status {
        constexpr int BITS = decltype(Bc)::value;
        if (dt == GNN_BF16)
            { dequantize_rows_kernel<__nv_bfloat16, BITS><<<blocks, 256, 0, s>>>(
                codes, ld_codes, scale_zero, n, ids, static_cast<__nv_bfloat16 *>(dst), ld_dst, n_dst, f, add, err); GNN_LAUNCHED(1); }
        else
            { dequantize_rows_kernel<float, BITS><<<blocks, 256, 0, s>>>(codes, ld_codes, scale_zero, n, ids,
                                                                        static_cast<float *>(dst), ld_dst, n_dst, f,
                                                                        add, err); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

gnn_status launch_codec_pull(const uint8_t *codes, int64_t ld_codes, const float *scale_zero, int64_t n_table,
                             int bits, const int64_t *ids, int64_t n_ids, void *H, int64_t ld_h, int64_t row0,
                             int64_t f, gnn_dtype dt, int *err, cudaStream_t s) {
    if (n_ids == 0) return GNN_OK;
    const unsigned blocks = (unsigned)std::min<int64_t>(ceil_div(n_ids * 32, 256), (int64_t)num_sms() * 16);
    return dispatch_bits(bits, [&](auto Bc) -> gnn_status {
        constexpr int BITS = decltype(Bc)::value;
        if (dt == GNN_BF16)
            { codec_pull_kernel<__nv_bfloat16, BITS><<<blocks, 256, 0, s>>>(
                codes, ld_codes, scale_zero, n_table, ids, n_ids, static_cast<__nv_bfloat16 *>(H), ld_h, row0, f,
                err); GNN_LAUNCHED(1); }
        else
            { codec_pull_kernel<float, BITS><<<blocks, 256, 0, s>>>(codes, ld_codes, scale_zero, n_table, ids, n_ids,
                                                                   static_cast<float *>(H), ld_h, row0, f, err); GNN_LAUNCHED(1); }
        GNN_CUDA_TRY(cudaGetLastError());
        return GNN_OK;
    });
}

}  // namespace gnn
