// qsa_prep: query RMS-norm + RoPE and K/V int8 quantisation.
//
// "Round 36 Track C: qsa_prep Single-Barrier norm_rope & w == 128 tg_sum +
// qsa_score_mm Loop Unrolling", section "Summary & Decision": the prep pass is
// memory-bound on the query and K/V rows; norm_rope reduces the row's squares,
// scales by rs and the weight g, and rotates dims below QROT with partner
// tid ^ 32.
//
// One CTA per token.  Each of the first ceil(Hq/3) warps owns three of the
// token's query rows, the next warp the K row and the last the V row.  With
// head_dim 128 every lane holds four consecutive elements, so a row is one
// coalesced 512-byte load and a sum of squares is five xor-shuffles.  The token's rotation angles are computed once
// per CTA (the product p * inv_freq exactly in double, reduced modulo 2*pi,
// then an fp32 sincos) because a single fp32 product p * inv_freq is off by up
// to 2e-3 rad at p ~ 32k.  The frequency table itself is computed once per
// call on the host (GB300's fp64 rate makes a per-CTA pow expensive).
#include <cuda_fp16.h>

#include <cmath>

#include "check.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int D = 128;
constexpr int G = 32;

struct PrepParams {
    PrepLaunch a;
};

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

constexpr int MAXQH = 30;  // query heads per token (the launcher's limit)

// HPW query heads per warp: warps 0 .. ceil(Hq/HPW)-1 own the query rows,
// the next two the K and the V row.  Three heads per warp keeps a token's
// CTA at 6 warps for 12 heads (at most 384 threads for the launcher's 30),
// so eight tokens' CTAs fit on an SM at 40 registers; prep is bound by each
// token's latency chain, and more tokens in flight hide it.  (One head per
// warp, 14 warps per token: 14.4 us at the 1984-token workload; three: 12.9.)
constexpr int HPW = 3;

__global__ void __launch_bounds__(384, 4) prep_kernel(PrepParams P) {
    const PrepLaunch &a = P.a;
    allow_dependent_launch();  // a programmatic dependent may be scheduled once every CTA has started
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (t >= a.ntok) {  // padding rows of the score's head sum
        if (!QSA_IN(t, a.ntok_pad)) return;
        for (int i = threadIdx.x; i < 2 * D; i += blockDim.x) a.qbar[(size_t)t * 2 * D + i] = 0;
        if (threadIdx.x == 0) a.qexp[t] = 0;
        return;
    }
    __shared__ float4 qrows[MAXQH][D / 4];  // rotated query rows, for the head sum
    __shared__ float2 cs[D / 2];
    __shared__ float2 kcs[D / 2];  // fp32 of double-precision (cos, sin), for the key rotation
    const int half = a.rope_dims >> 1;

    // Issue this warp's row loads before the angle table is built.
    const int nqw = (a.n_q_heads + HPW - 1) / HPW;
    const bool is_q = warp < nqw, is_kv = !is_q && warp < nqw + 2;
    const bool is_v = warp == nqw + 1;
    float4 xs[HPW], g = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < HPW; ++j) xs[j] = g;
    if (is_q) {
        g = __ldg(reinterpret_cast<const float4 *>(a.norm_w) + lane);
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
            const int h = HPW * warp + j;
            if (h < a.n_q_heads && QSA_IN(((size_t)t * a.n_q_heads + h) * D + D - 1, (size_t)a.ntok * a.n_q_heads * D))
                xs[j] = __ldg(reinterpret_cast<const float4 *>(a.q_in + ((size_t)t * a.n_q_heads + h) * D) + lane);
        }
    } else if (is_kv) {
        xs[0] = __ldg(reinterpret_cast<const float4 *>((is_v ? a.v_in : a.k_in) + (size_t)t * D) + lane);
    }
    const float4 x = xs[0];

    if ((int)threadIdx.x < half) {
        const int i = threadIdx.x;
        const double ang = (double)(a.pos0 + t) * (double)a.inv_freq[i];  // exact: 24-bit x < 2^29
        const double two_pi = 6.283185307179586;
        const double k = rint(ang * (1.0 / two_pi));
        const float r = (float)fma(-k, two_pi, ang);
        float s, c;
        sincosf(r, &s, &c);
        cs[i] = make_float2(c, s);
        if (a.rope_k) {
            double sd, cd;
            sincos(ang, &sd, &cd);
            kcs[i] = make_float2((float)cd, (float)sd);
        }
    }
    __syncthreads();

    if (is_q) {
        // The warp's rows side by side: their shuffle chains interleave.
        float y[HPW][4];
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
            const float4 xj = xs[j];
            float ss = xj.x * xj.x + xj.y * xj.y + xj.z * xj.z + xj.w * xj.w;
            ss = warp_sum(ss);
            const float rs = __frsqrt_rn(ss / (float)D + a.eps);
            y[j][0] = (rs * xj.x) * g.x;
            y[j][1] = (rs * xj.y) * g.y;
            y[j][2] = (rs * xj.z) * g.z;
            y[j][3] = (rs * xj.w) * g.w;
        }
        if (half > 0) {
            const int sh = half >> 2;  // lanes between partners (half is a multiple of 4)
            const int i0 = lane * 4;
#pragma unroll
            for (int j = 0; j < HPW; ++j) {
                float up[4], dn[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    up[e] = __shfl_down_sync(0xffffffffu, y[j][e], sh);
                    dn[e] = __shfl_up_sync(0xffffffffu, y[j][e], sh);
                }
                if (i0 < half) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 c = cs[i0 + e];
                        y[j][e] = y[j][e] * c.x - up[e] * c.y;
                    }
                } else if (i0 < 2 * half) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 c = cs[i0 - half + e];
                        y[j][e] = y[j][e] * c.x + dn[e] * c.y;
                    }
                }
            }
        }
#pragma unroll
        for (int j = 0; j < HPW; ++j) {
            const int h = HPW * warp + j;
            if (h >= a.n_q_heads) continue;
            const size_t row = ((size_t)t * a.n_q_heads + h) * D;
            if (!QSA_IN(row + D - 1, (size_t)a.ntok * a.n_q_heads * D)) continue;
            if (a.qbar) qrows[h][lane] = make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
            const __half2 h01 = __floats2half2_rn(y[j][0], y[j][1]);
            const __half2 h23 = __floats2half2_rn(y[j][2], y[j][3]);
            uint2 hv;
            hv.x = *reinterpret_cast<const uint32_t *>(&h01);
            hv.y = *reinterpret_cast<const uint32_t *>(&h23);
            reinterpret_cast<uint2 *>(a.q_out + row)[lane] = hv;
            if (a.q_out_f32)
                reinterpret_cast<float4 *>(a.q_out_f32 + row)[lane] = make_float4(y[j][0], y[j][1], y[j][2], y[j][3]);
        }
    } else if (is_kv) {
        if (!QSA_IN(a.pos0 + t, a.cache_cells)) return;
        int8_t *dst = (is_v ? a.vq : a.kq) + (size_t)(a.pos0 + t) * D;
        uint16_t *sdst = (is_v ? a.vsc : a.ksc) + (size_t)(a.pos0 + t) * (D / G);
        float xv[4] = {x.x, x.y, x.z, x.w};
        if (a.rope_k && !is_v && half > 0) {
            // Key rotation in explicit round-to-nearest fp32 steps (no fused
            // multiply-add), the order the oracle defines, since the rotated
            // values decide the codes.
            const int sh = half >> 2;
            float up[4], dn[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                up[e] = __shfl_down_sync(0xffffffffu, xv[e], sh);
                dn[e] = __shfl_up_sync(0xffffffffu, xv[e], sh);
            }
            const int i0 = lane * 4;
            if (i0 < half) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 c = kcs[i0 + e];
                    xv[e] = __fsub_rn(__fmul_rn(xv[e], c.x), __fmul_rn(up[e], c.y));
                }
            } else if (i0 < 2 * half) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 c = kcs[i0 - half + e];
                    xv[e] = __fadd_rn(__fmul_rn(xv[e], c.x), __fmul_rn(dn[e], c.y));
                }
            }
        }
        float amax = fmaxf(fmaxf(fabsf(xv[0]), fabsf(xv[1])), fmaxf(fabsf(xv[2]), fabsf(xv[3])));
#pragma unroll
        for (int o = 1; o < 8; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        const __half sh = __float2half_rn(__fdiv_rn(amax, 127.0f));
        const float sf = __half2float(sh);
        uint32_t packed = 0;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float c = 0.0f;
            if (sf != 0.0f) c = fminf(fmaxf(rintf(__fdiv_rn(xv[e], sf)), -127.0f), 127.0f);
            packed |= ((uint32_t)(uint8_t)(int8_t)(int)c) << (8 * e);
        }
        reinterpret_cast<uint32_t *>(dst)[lane] = packed;
        if ((lane & 7) == 0) sdst[lane >> 3] = __half_as_ushort(sh);
    }
    if (a.qbar) {
        // The score's head sum: fp32, heads in order (as the score's own
        // head-sum pass adds the fp32 rows), scaled by the token's power of
        // two and split into an fp16 hi/lo pair.  A block has at least 96
        // threads, so each thread sums at most two of the 128 dims.
        __shared__ float wmax[12];
        __syncthreads();
        const float *rows = reinterpret_cast<const float *>(qrows);
        float sums[2] = {0.0f, 0.0f}, m = 0.0f;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int d = threadIdx.x + i * blockDim.x;
            if (d < D) {
                float sum = 0.0f;
                for (int h = 0; h < a.n_q_heads; ++h) sum += rows[h * D + d];
                sums[i] = sum;
                m = fmaxf(m, fabsf(sum));
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) wmax[warp] = m;
        __syncthreads();
        m = wmax[0];
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) m = fmaxf(m, wmax[w]);
        const int e = head_sum_exponent(m);
        if (!QSA_IN(t, a.ntok_pad)) return;
        const float f = exp2i(e);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int d = threadIdx.x + i * blockDim.x;
            if (d < D) {
                const float v = sums[i] * f;
                const __half hi = __float2half_rn(v);
                const __half lo = __float2half_rn(v - __half2float(hi));
                a.qbar[(size_t)t * 2 * D + d] = __half_as_ushort(hi);
                a.qbar[(size_t)t * 2 * D + D + d] = __half_as_ushort(lo);
            }
        }
        if (threadIdx.x == 0) a.qexp[t] = e;
    }
}

}  // namespace

cudaError_t launch_prep(const PrepLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    PrepParams P{a};
    for (int i = 0; i < a.rope_dims / 2; ++i)
        P.a.inv_freq[i] = (float)std::pow((double)a.rope_theta, -2.0 * (double)i / (double)a.rope_dims);
    const int threads = 32 * ((a.n_q_heads + HPW - 1) / HPW + 2);  // <= 384 for n_q_heads <= 30
    prep_kernel<<<a.qbar ? a.ntok_pad : a.ntok, threads, 0, s>>>(P);
    return cudaGetLastError();
}

}  // namespace qsa

QSA_DEFINE_CHECK_READER(take_check_word_prep)

