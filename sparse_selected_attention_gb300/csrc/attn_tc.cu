// qsa_attn fused path on the 5th-generation tensor cores (tcgen05).
//
// Same computation as attn.cu's fused path (see there for the pages' passages:
// per-token selected ids with -1 padding, per-chunk maxima and denominators,
// max-first merge, one value load per dimension per cell shared by all heads).
//
// One persistent CTA per SM walks a stream of tokens; each token's id list is
// cut into 128-cell tiles.  Warp roles:
//  * converter warps 4..11 gather the tile's int8 K and V rows (prefetched one
//    tile ahead into registers) and write them as fp16 into shared memory in
//    the 128-byte-swizzled layout: K exact (codes), V dequantised by its group
//    scale.  The same bytes serve as the K-major A operand of Q.K^T
//    (rows = cells) and as the MN-major A operand of P.V (rows = cells,
//    M = head dims contiguous), so no transposition is needed.  Warp 4 also
//    stages each token's Q rows (the B operand of Q.K^T).
//  * one thread of warp 12 issues the MMAs: S_g = K_g Q_g^T for the four
//    32-dim scale groups into four TMEM accumulators (M = 128 cells, N = 16
//    heads), and O += V^T P^T into a TMEM accumulator (M = 128 dims, N = 16).
//  * softmax warps 0..3 (thread = cell = TMEM lane) combine the groups with
//    the cell's key scales, take the tile maximum per head across the CTA,
//    rescale O in tensor memory when a head's running maximum grows, write
//    P (fp16) as the K-major B operand of P.V, and at the end of a token read
//    O back (thread = head dim), divide by the denominator and store fp16.
// Every hand-off is an mbarrier with a bounded wait; on expiry the kernel
// records QSA_DEVERR_TIMEOUT, all roles stop, tensor memory is freed and the
// kernel returns.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "qsa.h"
#include "qsa_internal.h"
#include "tc_common.cuh"

namespace qsa {
namespace {

using namespace tc;

constexpr int D = 128;
constexpr int NG = 4;     // 32-dim scale groups
constexpr int HP = 16;    // heads padded to the MMA's N
constexpr int TC = 128;   // cells per tile
constexpr int NSM = 4;    // softmax warps 0..3
constexpr int NCV = 8;    // converter warps 4..11
constexpr int MMA_W = NSM + NCV;
constexpr int THREADS = 32 * (MMA_W + 1);
constexpr int CV = NCV * 32;
constexpr uint32_t TMEM_COLS = 256;
constexpr uint32_t OCOL = 128;  // O accumulators at columns 128.. (2 x 16)

constexpr uint32_t Q_BYTES = HP * D * 2;  // 2 K-blocks x 16 rows x 128 B
constexpr uint32_t Q_KB = HP * 128;
constexpr uint32_t T_BYTES = TC * D * 2;  // one fp16 K or V tile
constexpr uint32_t T_KB = TC * 128;       // 64-dim block of a tile (= MN atom stride for V)
constexpr uint32_t P_BYTES = HP * TC * 2; // 2 K-blocks (64 cells) x 16 rows x 128 B
constexpr uint32_t P_KB = HP * 128;
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + 2 * Q_BYTES;
constexpr uint32_t OFF_V = OFF_K + 2 * T_BYTES;
constexpr uint32_t OFF_P = OFF_V + 2 * T_BYTES;
constexpr uint32_t OFF_RED = OFF_P + 2 * P_BYTES;  // [4][16] per-warp + [16] final, floats
constexpr uint32_t OFF_BAR = OFF_RED + 512;
constexpr int NBAR = 20;
constexpr uint32_t OFF_FLAG = OFF_BAR + NBAR * 8;
constexpr uint32_t SMEM_USED = OFF_FLAG + 16;
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;
static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory layout");

constexpr uint32_t IDESC_QK = idesc_f16(128, HP, false, false);
constexpr uint32_t IDESC_PV = idesc_f16(128, HP, true, false);
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_SLACK = 8.0f;  // log2 units: P <= 256 between rescales

__device__ __forceinline__ void sm_sync() { asm volatile("bar.sync 2, %0;" ::"n"(NSM * 32) : "memory"); }

// Barrier among the softmax threads that also ORs a flag across them.
__device__ __forceinline__ bool sm_sync_or(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 3, %2, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(NSM * 32)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// Byte offset of 16-byte chunk `ch16` (0..15 over the 128 head dims) of row
// `row` in a 128-row tile stored as two 64-dim blocks of 128-byte-swizzled rows.
__device__ __forceinline__ uint32_t tile_off(int row, int ch16) {
    return (uint32_t)(ch16 >> 3) * T_KB + (uint32_t)(row >> 3) * 1024 + (uint32_t)(row & 7) * 128 +
           (uint32_t)(((ch16 & 7) ^ (row & 7)) << 4);
}

// Transpose-reduce 16 per-lane values across the warp: afterwards lane l holds
// the reduction for head 8*b4 + 4*b3 + 2*b2 + b1 (b_k = bit k of l).
template <bool MAX>
__device__ __forceinline__ float warp_head_reduce(float (&x)[16]) {
    const int lane = threadIdx.x & 31;
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool up = lane & 16;
        const float send = up ? x[i] : x[i + 8], keep = up ? x[i + 8] : x[i];
        x[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 16));
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const bool up = lane & 8;
        const float send = up ? x[i] : x[i + 4], keep = up ? x[i + 4] : x[i];
        x[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 8));
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const bool up = lane & 4;
        const float send = up ? x[i] : x[i + 2], keep = up ? x[i + 2] : x[i];
        x[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, 4));
    }
    {
        const bool up = lane & 2;
        const float send = up ? x[0] : x[1], keep = up ? x[1] : x[0];
        x[0] = op(keep, __shfl_xor_sync(0xffffffffu, send, 2));
    }
    return op(x[0], __shfl_xor_sync(0xffffffffu, x[0], 1));
}

__device__ __forceinline__ int lane_head(int lane) {
    return 8 * ((lane >> 4) & 1) + 4 * ((lane >> 3) & 1) + 2 * ((lane >> 2) & 1) + ((lane >> 1) & 1);
}

// Cross-warp combination of the per-warp head reductions of the 4 softmax
// warps; returns all 16 results to every softmax thread.
template <bool MAX>
__device__ __forceinline__ void cta_head_reduce(float (&x)[16], float *red, float (&out)[16]) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const float v = warp_head_reduce<MAX>(x);
    if ((lane & 1) == 0) red[warp * 16 + lane_head(lane)] = v;
    sm_sync();
    if (warp == 0 && lane < 16) {
        float m = red[lane];
#pragma unroll
        for (int w = 1; w < NSM; ++w) m = MAX ? fmaxf(m, red[w * 16 + lane]) : m + red[w * 16 + lane];
        red[64 + lane] = m;
    }
    sm_sync();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4 f = reinterpret_cast<const float4 *>(red + 64)[i];
        out[4 * i] = f.x;
        out[4 * i + 1] = f.y;
        out[4 * i + 2] = f.z;
        out[4 * i + 3] = f.w;
    }
}

struct TcArgs {
    AttnLaunch a;
    int nt;  // tiles per token
};

// 13 warps: the busiest SM sub-partition holds 4 of them, so its 16 K-register
// file caps the kernel at 128 registers per thread.
__global__ void __launch_bounds__(THREADS, 1) attn_tc_kernel(TcArgs P) {
    const AttnLaunch &a = P.a;
    const int NT = P.nt;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gen = smem_raw + (base - raw);
    const uint32_t sQ = base + OFF_Q, sK = base + OFF_K, sV = base + OFF_V, sP = base + OFF_P;
    float *red = reinterpret_cast<float *>(gen + OFF_RED);
    const uint32_t bar = base + OFF_BAR;
    const uint32_t q_full = bar, q_empty = bar + 16, k_full = bar + 32, k_empty = bar + 48, v_full = bar + 64,
                   pv_done = bar + 80, s_full = bar + 96, s_empty = bar + 112, p_full = bar + 128,
                   o_free = bar + 144;
    volatile int *abort = reinterpret_cast<volatile int *>(gen + OFF_FLAG);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gen + OFF_FLAG + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(q_full + 8 * i, 32);
            mbar_init(q_empty + 8 * i, 1);
            mbar_init(k_full + 8 * i, CV);
            mbar_init(k_empty + 8 * i, 1);
            mbar_init(v_full + 8 * i, CV);
            mbar_init(pv_done + 8 * i, 1);
            mbar_init(s_full + 8 * i, 1);
            mbar_init(s_empty + 8 * i, NSM * 32);
            mbar_init(p_full + 8 * i, NSM * 32);
            mbar_init(o_free + 8 * i, NSM * 32);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MMA_W) tmem_alloc(smem_u32((const void *)tslot), TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;

    // Tokens of this CTA: t_i = ntok-1 - (blockIdx.x + i*gridDim.x).
    const int ntoks = (int)blockIdx.x < a.ntok ? (a.ntok - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int ntiles = ntoks * NT;
    auto token_of = [&](int ti) { return a.ntok - 1 - ((int)blockIdx.x + ti * (int)gridDim.x); };

    if (warp >= NSM && warp < MMA_W) {
        // ---------------- converters ----------------
        const int ct = tid - NSM * 32, ch = ct & 7, c0 = ct >> 3;  // chunk of 16 dims; cells c0 + 32*it
        bool bad = false;
        auto load_ids = [&](int k, int (&id)[4]) {
#pragma unroll
            for (int it = 0; it < 4; ++it) id[it] = -1;
            if (k >= ntiles) return;
            const int t = token_of(k / NT), slot0 = (k % NT) * TC;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int slot = slot0 + c0 + 32 * it;
                int v = slot < a.width ? __ldg(a.ids + (size_t)t * a.width + slot) : -1;
                bad |= (v < -1) || (v >= a.cache_cells);
                id[it] = (v >= 0 && v < a.cache_cells) ? v : -1;
            }
        };
        struct Raw {
            uint4 k[4], v[4];
            uint32_t vs[4];
        };
        auto load_raw = [&](const int (&id)[4], Raw &r) {
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                if (id[it] >= 0) {
                    const size_t row = (size_t)id[it] * D;
                    r.k[it] = __ldg(reinterpret_cast<const uint4 *>(a.kq + row) + ch);
                    r.v[it] = __ldg(reinterpret_cast<const uint4 *>(a.vq + row) + ch);
                    r.vs[it] = __ldg(a.vsc + (size_t)id[it] * NG + (ch >> 1));
                } else {
                    r.k[it] = r.v[it] = make_uint4(0u, 0u, 0u, 0u);
                    r.vs[it] = 0u;
                }
            }
        };
        int idA[4], idB[4];
        Raw cur, nxt;
        load_ids(0, idA);
        load_ids(1, idB);
        load_raw(idA, cur);
        bool failed = false;
        for (int k = 0; k < ntiles && !failed; ++k) {
            const int ti = k / NT, j = k % NT, kb = k & 1;
            // Prefetch: raw rows of tile k+1 (ids known), ids of tile k+2.
            load_raw(idB, nxt);
            load_ids(k + 2, idA);
            if (j == 0 && warp == NSM) {
                // Stage this token's Q rows (zeros past n_q_heads).
                const int qb = ti & 1, t = token_of(ti);
                if (ti >= 2 && !mbar_wait_or_abort(q_empty + 8 * qb, ((ti >> 1) - 1) & 1, abort)) {
                    failed = true;
                    break;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int q = i * 32 + lane, row = q >> 4, ci = q & 15;
                    uint4 v = make_uint4(0u, 0u, 0u, 0u);
                    if (row < a.n_q_heads)
                        v = __ldg(reinterpret_cast<const uint4 *>(a.q + ((size_t)t * a.n_q_heads + row) * D) + ci);
                    const uint32_t p = sQ + qb * Q_BYTES + (ci >> 3) * Q_KB + (row >> 3) * 1024 + (row & 7) * 128 +
                                       (((ci & 7) ^ (row & 7)) << 4);
                    asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                                 "r"(v.w));
                }
                fence_async_smem();
                mbar_arrive(q_full + 8 * qb);
            }
            if (k >= 2 && !mbar_wait_or_abort(k_empty + 8 * kb, ((k >> 1) - 1) & 1, abort)) {
                failed = true;
                break;
            }
            // K: exact fp16 codes.
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int c = c0 + 32 * it;
                uint32_t h[8];
                codes_to_h2(cur.k[it].x ^ 0x80808080u, h[0], h[1]);
                codes_to_h2(cur.k[it].y ^ 0x80808080u, h[2], h[3]);
                codes_to_h2(cur.k[it].z ^ 0x80808080u, h[4], h[5]);
                codes_to_h2(cur.k[it].w ^ 0x80808080u, h[6], h[7]);
                const uint32_t dst = sK + kb * T_BYTES;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + tile_off(c, 2 * ch)), "r"(h[0]),
                             "r"(h[1]), "r"(h[2]), "r"(h[3]));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + tile_off(c, 2 * ch + 1)),
                             "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]));
            }
            fence_async_smem();
            mbar_arrive(k_full + 8 * kb);
            if (k >= 2 && !mbar_wait_or_abort(pv_done + 8 * kb, ((k >> 1) - 1) & 1, abort)) {
                failed = true;
                break;
            }
            // V: codes times their group scale.
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int c = c0 + 32 * it;
                const __half2 sc = __half2half2(__ushort_as_half((unsigned short)cur.vs[it]));
                uint32_t h[8];
                codes_to_h2(cur.v[it].x ^ 0x80808080u, h[0], h[1]);
                codes_to_h2(cur.v[it].y ^ 0x80808080u, h[2], h[3]);
                codes_to_h2(cur.v[it].z ^ 0x80808080u, h[4], h[5]);
                codes_to_h2(cur.v[it].w ^ 0x80808080u, h[6], h[7]);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    __half2 x = __hmul2(*reinterpret_cast<__half2 *>(&h[e]), sc);
                    h[e] = *reinterpret_cast<uint32_t *>(&x);
                }
                const uint32_t dst = sV + kb * T_BYTES;
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + tile_off(c, 2 * ch)), "r"(h[0]),
                             "r"(h[1]), "r"(h[2]), "r"(h[3]));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(dst + tile_off(c, 2 * ch + 1)),
                             "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]));
            }
            fence_async_smem();
            mbar_arrive(v_full + 8 * kb);
            cur = nxt;
#pragma unroll
            for (int it = 0; it < 4; ++it) {
                const int tmp = idB[it];
                idB[it] = idA[it];
                idA[it] = tmp;
            }
        }
        if (__any_sync(0xffffffffu, bad) && lane == 0 && a.err) atomicOr(a.err, QSA_DEVERR_BAD_ID);
    } else if (warp == MMA_W) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            auto pv = [&](int k) -> bool {
                const int ti = k / NT, j = k % NT, kb = k & 1, ob = ti & 1;
                if (!mbar_wait_or_abort(v_full + 8 * kb, (k >> 1) & 1, abort)) return false;
                if (!mbar_wait_or_abort(p_full + 8 * kb, (k >> 1) & 1, abort)) return false;
                if (j == 0 && ti >= 2 && !mbar_wait_or_abort(o_free + 8 * ob, ((ti >> 1) - 1) & 1, abort))
                    return false;
                fence_after();
                // A = V^T: MN-major, 64-dim atoms T_KB apart, 8-cell groups 1024
                // apart; only the 14-bit start-address field moves per k-step.
                const uint64_t ad0 = smem_desc(sV + kb * T_BYTES, T_KB, 1024, 2);
                const uint64_t bd0 = sw128_kmajor(sP + kb * P_BYTES);
#pragma unroll
                for (int ks = 0; ks < TC / 16; ++ks)
                    mma_f16(tmem + OCOL + ob * HP, ad0 + (uint64_t)((ks * 2048) >> 4),
                            bd0 + (uint64_t)(((ks >> 2) * P_KB + (ks & 3) * 32) >> 4), IDESC_PV,
                            (j > 0 || ks > 0) ? 1u : 0u);
                mma_commit(pv_done + 8 * kb);
                return true;
            };
            bool ok = true;
            for (int k = 0; k < ntiles && ok; ++k) {
                const int ti = k / NT, j = k % NT, kb = k & 1, qb = ti & 1;
                if (j == 0 && !mbar_wait_or_abort(q_full + 8 * qb, (ti >> 1) & 1, abort)) break;
                if (!mbar_wait_or_abort(k_full + 8 * kb, (k >> 1) & 1, abort)) break;
                if (k >= 2 && !mbar_wait_or_abort(s_empty + 8 * kb, ((k >> 1) - 1) & 1, abort)) break;
                fence_after();
                const uint64_t ad0 = sw128_kmajor(sK + kb * T_BYTES), bd0 = sw128_kmajor(sQ + qb * Q_BYTES);
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
                    for (int g = 0; g < NG; ++g) {
                        // Groups interleaved so consecutive MMAs target different accumulators.
                        const int ksx = 2 * g + s2, kb2 = ksx >> 2;
                        const uint32_t koff = (ksx & 3) * 32;
                        mma_f16(tmem + kb * (NG * HP) + g * HP, ad0 + (uint64_t)((kb2 * T_KB + koff) >> 4),
                                bd0 + (uint64_t)((kb2 * Q_KB + koff) >> 4), IDESC_QK, s2 ? 1u : 0u);
                    }
                mma_commit(k_empty + 8 * kb);
                mma_commit(s_full + 8 * kb);
                if (j == NT - 1) mma_commit(q_empty + 8 * qb);
                if (k >= 1) ok = pv(k - 1);
            }
            if (ok && ntiles > 0) pv(ntiles - 1);
        }
    } else {
        // ---------------- softmax (thread = cell of the tile = TMEM lane) ----------------
        const float sl2 = a.softmax_scale * LOG2E;
        float M[HP], L[HP];
        // This thread's cell id (two tiles ahead) and key scales (one tile
        // ahead), so neither load sits on a tile's critical path.
        auto raw_id = [&](int k) -> int {
            if (k >= ntiles) return -1;
            const int t = token_of(k / NT), slot = (k % NT) * TC + tid;
            const int v = slot < a.width ? __ldg(a.ids + (size_t)t * a.width + slot) : -1;
            return (v >= 0 && v < a.cache_cells) ? v : -1;
        };
        auto scales_of = [&](int id) -> uint2 {
            return id >= 0 ? __ldg(reinterpret_cast<const uint2 *>(a.ksc + (size_t)id * NG)) : make_uint2(0u, 0u);
        };
        int id_cur = raw_id(0), id_nxt = raw_id(1);
        uint2 kv_cur = scales_of(id_cur);
        for (int k = 0; k < ntiles; ++k) {
            const int ti = k / NT, j = k % NT, kb = k & 1, ob = ti & 1;
            const bool valid = id_cur >= 0;
            const uint2 kv = kv_cur;
            kv_cur = scales_of(id_nxt);
            id_cur = id_nxt;
            id_nxt = raw_id(k + 2);
            if (j == 0) {
#pragma unroll
                for (int h = 0; h < HP; ++h) {
                    M[h] = -CUDART_INF_F;
                    L[h] = 0.0f;
                }
            }
            bool fail = !mbar_wait_or_abort(s_full + 8 * kb, (k >> 1) & 1, abort);
            if (sm_sync_or(fail)) break;
            fence_after();
            // Combine the four group accumulators one TMEM load at a time:
            // s_h = sum_g (scale * log2 e * ksc[g]) * S_g[h].
            const float kg[NG] = {sl2 * __half2float(__ushort_as_half((unsigned short)(kv.x & 0xFFFF))),
                                  sl2 * __half2float(__ushort_as_half((unsigned short)(kv.x >> 16))),
                                  sl2 * __half2float(__ushort_as_half((unsigned short)(kv.y & 0xFFFF))),
                                  sl2 * __half2float(__ushort_as_half((unsigned short)(kv.y >> 16)))};
            uint64_t s2[HP / 2];
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                uint32_t acc[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + kb * (NG * HP) + g * HP, acc);
                tmem_wait_ld();
                const uint64_t K2 = pack2(kg[g], kg[g]);
#pragma unroll
                for (int i = 0; i < HP / 2; ++i)
                    s2[i] = fma2(K2, pack2(__uint_as_float(acc[2 * i]), __uint_as_float(acc[2 * i + 1])),
                                 g == 0 ? 0ull : s2[i]);
            }
            fence_before();
            mbar_arrive(s_empty + 8 * kb);
            float s[HP];
#pragma unroll
            for (int i = 0; i < HP / 2; ++i) {
                s[2 * i] = valid ? __uint_as_float((uint32_t)s2[i]) : -CUDART_INF_F;
                s[2 * i + 1] = valid ? __uint_as_float((uint32_t)(s2[i] >> 32)) : -CUDART_INF_F;
            }
            // Lazy rescaling: keep each head's reference maximum M unless a
            // score exceeds it by more than RESCALE_SLACK (log2 units), so P
            // stays <= 2^RESCALE_SLACK and fits fp16; the final O / L is exact
            // for any reference.  The tile maximum (and a rescale of O) is
            // only needed on a token's first tile and when the slack is
            // exceeded.
            bool over = false;
#pragma unroll
            for (int h = 0; h < HP; ++h) over |= s[h] > M[h] + RESCALE_SLACK;
            if (sm_sync_or(over)) {
                float x[HP], tmax[HP];
#pragma unroll
                for (int h = 0; h < HP; ++h) x[h] = s[h];
                cta_head_reduce<true>(x, red, tmax);
                float alpha[HP];
                bool grow = false;
#pragma unroll
                for (int h = 0; h < HP; ++h) {
                    const float mn = fmaxf(M[h], tmax[h]);
                    alpha[h] = mn == -CUDART_INF_F ? 1.0f : exp2f(M[h] - mn);
                    grow |= alpha[h] != 1.0f;
                    M[h] = mn;
                }
                if (j > 0 && grow) {
                    // Rescale O (which holds tiles up to k-1) before P.V of tile k.
                    fail = !mbar_wait_or_abort(pv_done + 8 * ((k - 1) & 1), ((k - 1) >> 1) & 1, abort);
                    if (sm_sync_or(fail)) break;
                    fence_after();
                    uint32_t o[16];
                    const uint32_t oaddr = tmem + ((uint32_t)(warp * 32) << 16) + OCOL + ob * HP;
                    tmem_ld16(oaddr, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int h = 0; h < HP; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * alpha[h]);
                    tmem_st16(oaddr, o);
                    tmem_wait_st();
#pragma unroll
                    for (int h = 0; h < HP; ++h) L[h] *= alpha[h];
                }
            }
            __half p16[HP];
#pragma unroll
            for (int h = 0; h < HP; ++h) {
                const float p = (valid && M[h] != -CUDART_INF_F) ? exp2f(s[h] - M[h]) : 0.0f;
                L[h] += p;
                p16[h] = __float2half_rn(p);
            }
            fail = k >= 2 && !mbar_wait_or_abort(pv_done + 8 * kb, ((k >> 1) - 1) & 1, abort);
            if (sm_sync_or(fail)) break;
            {
                // P row h, column (cell) tid of the K-major B operand.
                const int c = tid;
                const uint32_t pb = sP + kb * P_BYTES + (c >> 6) * P_KB + (c & 7) * 2;
#pragma unroll
                for (int h = 0; h < HP; ++h) {
                    const uint32_t adr = pb + (h >> 3) * 1024 + (h & 7) * 128 + ((((c & 63) >> 3) ^ (h & 7)) << 4);
                    asm volatile("st.shared.b16 [%0], %1;" ::"r"(adr), "h"(__half_as_ushort(p16[h])));
                }
            }
            fence_async_smem();
            fence_before();
            mbar_arrive(p_full + 8 * kb);

            if (j == NT - 1) {
                // End of token: O / L -> fp16 out (thread = head dim).
                float lx[HP], Lt[HP];
#pragma unroll
                for (int h = 0; h < HP; ++h) lx[h] = L[h];
                cta_head_reduce<false>(lx, red, Lt);
                fail = !mbar_wait_or_abort(pv_done + 8 * kb, (k >> 1) & 1, abort);
                if (sm_sync_or(fail)) break;
                fence_after();
                uint32_t o[16];
                tmem_ld16(tmem + ((uint32_t)(warp * 32) << 16) + OCOL + ob * HP, o);
                tmem_wait_ld();
                fence_before();
                mbar_arrive(o_free + 8 * ob);
                const int t = token_of(ti);
                for (int h = 0; h < a.n_q_heads; ++h) {
                    const float r = Lt[h] > 0.0f ? __uint_as_float(o[h]) / Lt[h] : 0.0f;
                    a.out[((size_t)t * a.n_q_heads + h) * D + tid] = __half_as_ushort(__float2half_rn(r));
                }
            }
        }
    }

    fence_before();
    __syncthreads();
    if (tid == 0 && *abort && a.err) atomicOr(a.err, QSA_DEVERR_TIMEOUT);
    if (warp == MMA_W) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_attn_tc(const AttnLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    int dev = 0, sms = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC)) !=
        cudaSuccess)
        return e;
    TcArgs P{a, (a.width + TC - 1) / TC};
    const int grid = a.ntok < sms ? a.ntok : sms;
    attn_tc_kernel<<<grid, THREADS, SMEM_ALLOC, s>>>(P);
    return cudaGetLastError();
}

}  // namespace qsa
