// qsa_attn: chunked attention over per-token selected cache cells.
//
// "round 11 track b: qsa attention and score", section "implementation and
// evaluator": per-token selected ids with -1 padding, 64-cell chunks (the last
// one possibly incomplete), K row pointers and the four scale groups resolved
// once per step, V pointers and scales once per run of cells.
// "round 5 track b: cached residual norms and fused mtp attention", sections
// "mtp attention" and "preflight / ownership": per-chunk maxima and
// denominators, a max-first chunk merge, and value accumulation for all 12
// heads together so each value is loaded once per dimension per cell.
//
// GB300 design.  The 12 query heads share one KV row, so a cell's K and V
// codes are gathered once and used for every head: the head dimension is the
// M side (padded 12 -> 16) of m16n8k16 tensor-core products, cells are N for
// Q.K^T and the contraction for P.V.  A permutation of the contraction index d
// makes each thread's part of a K row one contiguous 32-byte span (group r of
// the row for quad lane r) and its part of a V row one contiguous 16-byte span,
// so fragments are read with 16-byte shared-memory loads.  Codes are turned
// into exact fp16 integers with a byte-permute bias trick (0x64xx - 1152) and
// scaled by their fp16 group scale in the same registers.  Padding slots are
// never dereferenced: cp.async zero-fills them, scores are -inf, values zero.
//
// Fused path (part == NULL): one CTA per token, four warps; each warp streams
// its share of 32-cell units through a private two-stage shared-memory ring
// filled by cp.async (rows swizzled by 16-byte chunk so fragment reads are
// bank-conflict free), with an online max / denominator, and the warps' states
// are merged max-first in shared memory.  Split path (part != NULL): one warp
// per 64-cell chunk writes that chunk's (o_c, m_c, l_c); a second kernel merges
// the chunks max-first exactly as the definition states.
//
// Several KV heads ("round 5 track b ...", section "mtp attention": a grid of
// two KV heads per token, 12 query heads on each) become a second grid
// dimension: a CTA serves one (token, KV head).  The pages' head_dim 256 with
// per-64 scales keeps four scale groups per row; two warps share each unit,
// each staging, converting and multiplying only its 128-dim half of every K
// and V row.  Their partial Q.K^T sums meet in shared memory (one 64-thread
// named barrier per unit), and both warps add them, so they hold identical
// scores and softmax state; each then accumulates P.V for its half of the
// dims.  An optional sigmoid output gate multiplies the merged result.
#include <cuda_fp16.h>
#include <math_constants.h>

#include "check.cuh"
#include "qsa.h"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int D = 128;     // dims one warp handles (the whole row when head_dim is 128)
constexpr int UNIT = 32;   // cells per warp step
constexpr int CHUNK = 64;  // cells per chunk of the definition
constexpr float LN2 = 0.6931471805599453f;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_SLACK = 8.0f;  // fused path: probabilities below 2^8 (exact in fp16 range)

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 2^x by the SFU's approximate base-2 exponential (relative error about
// 2^-22; results below the normal range flush to zero, where a probability
// is negligible against the running maximum's 1).
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<uint32_t *>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<__half2 *>(&u); }

// Bytes 0..3 of w are int8 codes already xor'ed with 0x80 (i.e. code + 128).
// 0x64xx is the fp16 value 1024 + xx, so (byte | 0x6400) - 1152 is the code,
// exactly.  lo = (code0, code1), hi = (code2, code3).
__device__ __forceinline__ void codes_to_h2(uint32_t wx, __half2 &lo, __half2 &hi) {
    const uint32_t m = 0x64646464u;
    const __half2 bias = u2h(0x64806480u);  // 1152.0 in both halves
    lo = __hsub2(u2h(prmt(wx, m, 0x4140)), bias);
    hi = __hsub2(u2h(prmt(wx, m, 0x4342)), bias);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

// Where a warp's data lives.  KV head kvh serves query heads h0 .. h0+per-1;
// with S warps sharing a unit, warp part `half` owns dims [128 half, 128 half
// + 128) of rows of S * 128 dims.  Scales are four fp16 per (cell, KV head).
struct Geom {
    int kvh, h0, per, half;
    int kstride, koff;  // code row of cell c starts at c * kstride + koff
    int sstride, soff;  // its four scales at c * sstride + soff
};

template <int S>
__device__ __forceinline__ Geom make_geom(const AttnLaunch &a, int half) {
    Geom g;
    g.kvh = blockIdx.y;
    g.per = a.n_q_heads / a.n_kv_heads;
    g.h0 = g.kvh * g.per;
    g.half = half;
    g.kstride = a.n_kv_heads * D * S;
    g.koff = g.kvh * D * S + D * half;
    g.sstride = a.n_kv_heads * 4;
    g.soff = g.kvh * 4;
    return g;
}

template <int S>
__device__ __forceinline__ size_t kv_row(const AttnLaunch &, const Geom &g, int c) {
    return (size_t)c * g.kstride + g.koff;
}
__device__ __forceinline__ size_t scale_row(const AttnLaunch &, const Geom &g, int c) {
    return (size_t)c * g.sstride + g.soff;
}
// Scale group of quad lane r's 32 K dims and of lane group g's 16 V dims.
template <int S>
__device__ __forceinline__ int kgroup(int r, int half) {
    return S == 1 ? r : 2 * half + (r >> 1);
}
template <int S>
__device__ __forceinline__ int vgroup(int g, int half) {
    return S == 1 ? (g >> 1) : 2 * half + (g >> 2);
}

// With S == 2 the two warps of a unit (warps 2p, 2p+1) each hold Q.K^T over
// their half of the contraction; after this both hold the full sums, equal
// bit for bit (floating-point addition commutes).  `xch` holds two parity
// slots of 16 floats x 32 lanes per warp; one named barrier per unit suffices
// because a slot is rewritten only after the partner passed the next barrier.
template <int S>
__device__ __forceinline__ void exchange_s(float (&s)[4][4], float *xch, int parity) {
    if constexpr (S == 2) {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        float *mine = xch + (warp * 2 + parity) * 16 * 32 + lane;
        const float *other = xch + ((warp ^ 1) * 2 + parity) * 16 * 32 + lane;
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) mine[(4 * j + e) * 32] = s[j][e];
        asm volatile("bar.sync %0, 64;" ::"r"(1 + (warp >> 1)) : "memory");
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) s[j][e] += other[(4 * j + e) * 32];
    }
}

__device__ __forceinline__ float gated(const AttnLaunch &a, size_t idx, float v) {
    return a.gate ? v * (1.0f / (1.0f + expf(-__ldg(a.gate + idx)))) : v;
}

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Per-warp running state of one token: rows g and g+8 of the 16-head tile.
struct State {
    float o[16][4];  // o[jd][0..1]: row g, d = 32r + jd (+16); o[jd][2..3]: row g+8
    float m[2];      // running maximum, base-2 logits
    float l[2];      // running denominator, this thread's columns only
};

__device__ __forceinline__ void state_init(State &st) {
#pragma unroll
    for (int j = 0; j < 16; ++j)
#pragma unroll
        for (int e = 0; e < 4; ++e) st.o[j][e] = 0.0f;
    st.m[0] = st.m[1] = -CUDART_INF_F;
    st.l[0] = st.l[1] = 0.0f;
}

// Q fragments of token t for the permuted contraction: slot 2r+e of k-step ks
// holds d = 32r + 4ks + e, slot 2r+8+e holds d = 32r + 4ks + 2 + e.  `neg`
// flips every sign (exact), for a kernel that runs a negative softmax scale
// as its absolute value.
template <int S>
__device__ __forceinline__ void load_q(const AttnLaunch &a, int t, const Geom &geo, uint32_t (&qa)[8][4],
                                       bool neg = false) {
    const int lane = threadIdx.x & 31, g = lane >> 2, r = lane & 3;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int h = g + 8 * half;
        uint32_t w[16];
        const size_t qoff = ((size_t)t * a.n_q_heads + geo.h0 + h) * (D * S) + D * geo.half + 32 * r;
        if (h < geo.per && QSA_IN(qoff + 31, (size_t)a.ntok * a.n_q_heads * D * S)) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.q + qoff);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = __ldg(src + i);
                w[4 * i + 0] = v.x;
                w[4 * i + 1] = v.y;
                w[4 * i + 2] = v.z;
                w[4 * i + 3] = v.w;
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) w[i] = 0u;
        }
        const uint32_t flip = neg ? 0x80008000u : 0u;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][half] = w[2 * ks] ^ flip;
            qa[ks][2 + half] = w[2 * ks + 1] ^ flip;
        }
    }
}

// Q fragments held in registers for the whole token.
struct QRegs {
    uint32_t qa[8][4];
    __device__ __forceinline__ void get(int k, uint32_t (&f)[4]) const {
        f[0] = qa[k][0];
        f[1] = qa[k][1];
        f[2] = qa[k][2];
        f[3] = qa[k][3];
    }
};

// Q fragments in shared memory in fragment order: k-step k's four registers
// for lane l at 16 (32 k + l) bytes, so each k-step is one conflict-free
// 16-byte load per lane.  The warps that work on the same dims of the same
// token share one copy.
struct QSmem {
    const uint4 *base;  // this lane's k-step 0
    __device__ __forceinline__ void get(int k, uint32_t (&f)[4]) const {
        const uint4 v = base[32 * k];
        f[0] = v.x;
        f[1] = v.y;
        f[2] = v.z;
        f[3] = v.w;
    }
};
constexpr int QFRAG_BYTES = 8 * 32 * 16;  // one copy of a token's Q fragments (128 dims)

// One 32-cell unit (id slots slot0 .. slot0+31, lane's id already loaded)
// folded into the warp's state.  sl2 = softmax_scale * log2(e).  Sets `bad`
// if an id was < -1 or >= cache_cells.
template <int S, class Q>
__device__ __forceinline__ void process_unit(const AttnLaunch &a, int id, const Q &qsrc, State &st, float sl2,
                                             bool &bad, const Geom &geo, float *xch, int parity) {
    const int lane = threadIdx.x & 31, g = lane >> 2, r = lane & 3;
    const bool valid = id >= 0 && id < a.cache_cells;
    bad |= (id < -1) || (id >= a.cache_cells);
    const unsigned vmask = __ballot_sync(0xffffffffu, valid);
    if (vmask == 0u) return;
    if (!valid) id = -1;

    // Gather: K rows of cells 8j+g (this thread's bytes 32r..32r+31, group r)
    // and V rows of cells 16kk + 2r + {0,1,8,9} (bytes 16g..16g+15, group g/2).
    uint4 kd[4][2];
    __half ks[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int c = __shfl_sync(0xffffffffu, id, 8 * j + g);
        if (c >= 0 && QSA_IN(kv_row<S>(a, geo, c) + 32 * r + 31, (size_t)a.cache_cells * geo.kstride) &&
            QSA_IN(scale_row(a, geo, c) + 3, (size_t)a.cache_cells * geo.sstride)) {
            const uint4 *src = reinterpret_cast<const uint4 *>(a.kq + kv_row<S>(a, geo, c) + 32 * r);
            kd[j][0] = __ldg(src);
            kd[j][1] = __ldg(src + 1);
            ks[j] = __ushort_as_half(__ldg(a.ksc + scale_row(a, geo, c) + kgroup<S>(r, geo.half)));
        } else {
            kd[j][0] = kd[j][1] = make_uint4(0u, 0u, 0u, 0u);
            ks[j] = __ushort_as_half(0);
        }
    }
    uint4 vd[2][4];
    __half vs[2][4];
#pragma unroll
    for (int kk = 0; kk < 2; ++kk)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int c = __shfl_sync(0xffffffffu, id, 16 * kk + 2 * r + (e & 1) + 8 * (e >> 1));
            if (c >= 0 && QSA_IN(kv_row<S>(a, geo, c) + 16 * g + 15, (size_t)a.cache_cells * geo.kstride) &&
                QSA_IN(scale_row(a, geo, c) + 3, (size_t)a.cache_cells * geo.sstride)) {
                vd[kk][e] = __ldg(reinterpret_cast<const uint4 *>(a.vq + kv_row<S>(a, geo, c) + 16 * g));
                vs[kk][e] = __ushort_as_half(__ldg(a.vsc + scale_row(a, geo, c) + vgroup<S>(g, geo.half)));
            } else {
                vd[kk][e] = make_uint4(0u, 0u, 0u, 0u);
                vs[kk][e] = __ushort_as_half(0);
            }
        }

    // S = Q K^T for the 32 cells (4 n-tiles of 8), K dequantised in registers.
    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        uint32_t qf[4];
        qsrc.get(k, qf);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            __half2 lo, hi;
            const __half2 sc = __half2half2(ks[j]);
            codes_to_h2(word_of(kd[j][k >> 2], k & 3) ^ 0x80808080u, lo, hi);
            mma16816(s[j], qf, h2u(__hmul2(lo, sc)), h2u(__hmul2(hi, sc)));
        }
    }
    exchange_s<S>(s, xch, parity);

    // Online softmax in base 2 over this unit's valid cells.
    float mx0 = -CUDART_INF_F, mx1 = -CUDART_INF_F;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const bool v = (vmask >> (8 * j + 2 * r + e)) & 1u;
            s[j][e] = v ? s[j][e] * sl2 : -CUDART_INF_F;
            s[j][e + 2] = v ? s[j][e + 2] * sl2 : -CUDART_INF_F;
            mx0 = fmaxf(mx0, s[j][e]);
            mx1 = fmaxf(mx1, s[j][e + 2]);
        }
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    const float al0 = exp2f(st.m[0] - mn0), al1 = exp2f(st.m[1] - mn1);
    st.m[0] = mn0;
    st.m[1] = mn1;
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            s[j][e] = exp2f(s[j][e] - mn0);
            s[j][e + 2] = exp2f(s[j][e + 2] - mn1);
            ps0 += s[j][e];
            ps1 += s[j][e + 2];
        }
    st.l[0] = st.l[0] * al0 + ps0;
    st.l[1] = st.l[1] * al1 + ps1;
    if (__any_sync(0xffffffffu, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
        for (int jd = 0; jd < 16; ++jd) {
            st.o[jd][0] *= al0;
            st.o[jd][1] *= al0;
            st.o[jd][2] *= al1;
            st.o[jd][3] *= al1;
        }
    }

    // O += P V: P from the S accumulators (the mma C layout is the A layout),
    // V transposed by byte permutes and dequantised by its group scale.
#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4];
        pa[0] = h2u(__floats2half2_rn(s[2 * kk][0], s[2 * kk][1]));
        pa[1] = h2u(__floats2half2_rn(s[2 * kk][2], s[2 * kk][3]));
        pa[2] = h2u(__floats2half2_rn(s[2 * kk + 1][0], s[2 * kk + 1][1]));
        pa[3] = h2u(__floats2half2_rn(s[2 * kk + 1][2], s[2 * kk + 1][3]));
        const __half2 v01 = __halves2half2(vs[kk][0], vs[kk][1]);
        const __half2 v89 = __halves2half2(vs[kk][2], vs[kk][3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w0 = word_of(vd[kk][0], i) ^ 0x80808080u, w1 = word_of(vd[kk][1], i) ^ 0x80808080u;
            const uint32_t w8 = word_of(vd[kk][2], i) ^ 0x80808080u, w9 = word_of(vd[kk][3], i) ^ 0x80808080u;
            __half2 a0, a1, a2, a3, c0, c1, c2, c3;
            codes_to_h2(prmt(w0, w1, 0x5140), a0, a1);  // d = 16g + 4i + {0, 1}
            codes_to_h2(prmt(w0, w1, 0x7362), a2, a3);  // d = 16g + 4i + {2, 3}
            codes_to_h2(prmt(w8, w9, 0x5140), c0, c1);
            codes_to_h2(prmt(w8, w9, 0x7362), c2, c3);
            mma16816(st.o[4 * i + 0], pa, h2u(__hmul2(a0, v01)), h2u(__hmul2(c0, v89)));
            mma16816(st.o[4 * i + 1], pa, h2u(__hmul2(a1, v01)), h2u(__hmul2(c1, v89)));
            mma16816(st.o[4 * i + 2], pa, h2u(__hmul2(a2, v01)), h2u(__hmul2(c2, v89)));
            mma16816(st.o[4 * i + 3], pa, h2u(__hmul2(a3, v01)), h2u(__hmul2(c3, v89)));
        }
    }
}

__device__ __forceinline__ void quad_sum_l(State &st) {
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        st.l[0] += __shfl_xor_sync(0xffffffffu, st.l[0], o);
        st.l[1] += __shfl_xor_sync(0xffffffffu, st.l[1], o);
    }
}

#ifndef QSA_ATTN_MINB
#define QSA_ATTN_MINB 3
#endif

// ---------------------------------------------------------------------------
// Fused kernel: each warp streams its 32-cell units through a private ring
// of NS shared-memory stages filled by cp.async, NS-1 units ahead of the one
// it computes, so the gathers' latency overlaps the tensor-core work without
// holding the rows in registers.  Stage layout per unit: K codes [32][128]
// with 16-byte chunk q of cell c at q ^ (c & 1); V codes [32][128] with chunk
// q at q ^ (2 * ((c >> 1) & 3)) (both keep the fragment reads on distinct
// banks); then ksc [32][4] and vsc [32][4] fp16.
// ---------------------------------------------------------------------------
constexpr int STAGE_BYTES = 2 * UNIT * D + 2 * UNIT * 8;

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool pred) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(pred ? 16 : 0));
}
__device__ __forceinline__ void cp_async8(uint32_t dst, const void *src, bool pred) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8, %2;\n" ::"r"(dst), "l"(src), "r"(pred ? 8 : 0));
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// Issue the copies of one unit into stage `st` (shared address).  `id` is the
// lane's id slot (already mapped to -1 when invalid).
template <int S>
__device__ __forceinline__ void issue_unit(const AttnLaunch &a, int id, uint32_t st, const Geom &geo) {
    const int lane = threadIdx.x & 31, q = lane & 7;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int cell = (lane >> 3) + 4 * i;
        const int c = __shfl_sync(0xffffffffu, id, cell);
        const bool ok = c >= 0 && QSA_IN(kv_row<S>(a, geo, c) + 16 * q + 15, (size_t)a.cache_cells * geo.kstride);
        const size_t off = kv_row<S>(a, geo, ok ? c : 0) + 16 * q;
        cp_async16(st + cell * D + ((q ^ (cell & 1)) << 4), a.kq + off, ok);
        cp_async16(st + UNIT * D + cell * D + ((q ^ (2 * ((cell >> 1) & 3))) << 4), a.vq + off, ok);
    }
    const bool ok = id >= 0 && QSA_IN(scale_row(a, geo, id) + 3, (size_t)a.cache_cells * geo.sstride);
    const size_t so = scale_row(a, geo, ok ? id : 0);
    cp_async8(st + 2 * UNIT * D + lane * 8, a.ksc + so, ok);
    cp_async8(st + 2 * UNIT * D + UNIT * 8 + lane * 8, a.vsc + so, ok);
}

// Compute one staged unit.  vmask: valid cells of the unit.
template <int S, class Q>
__device__ __forceinline__ void compute_staged(const uint8_t *stp, unsigned vmask, const Q &qsrc, State &st,
                                               float sl2, int dhalf, float *xch, int parity) {
    const int lane = threadIdx.x & 31, g = lane >> 2, r = lane & 3;
    const uint8_t *K = stp, *V = stp + UNIT * D;
    const __half *KS = reinterpret_cast<const __half *>(stp + 2 * UNIT * D);
    const __half *VS = KS + UNIT * 4;

    float s[4][4];
#pragma unroll
    for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        uint4 kd[4];
        __half2 sc[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int cell = 8 * j + g;
            kd[j] = *reinterpret_cast<const uint4 *>(K + cell * D + (((2 * r + half) ^ (cell & 1)) << 4));
            sc[j] = __half2half2(KS[cell * 4 + kgroup<S>(r, dhalf)]);
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            uint32_t qf[4];
            qsrc.get(4 * half + kk, qf);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                __half2 lo, hi;
                codes_to_h2(word_of(kd[j], kk) ^ 0x80808080u, lo, hi);
                mma16816(s[j], qf, h2u(__hmul2(lo, sc[j])), h2u(__hmul2(hi, sc[j])));
            }
        }
    }
    exchange_s<S>(s, xch, parity);

    // Online softmax in base 2.  sl2 > 0 (the launch folds a negative scale
    // into the sign of q), so the maximum of the scaled logits is sl2 times
    // the maximum of the raw sums, and each probability is one fused
    // multiply-subtract and one ex2.  Padding cells are masked only in units
    // that hold some.
    if (vmask != 0xffffffffu) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const bool v = (vmask >> (8 * j + 2 * r + e)) & 1u;
                s[j][e] = v ? s[j][e] : -CUDART_INF_F;
                s[j][e + 2] = v ? s[j][e + 2] : -CUDART_INF_F;
            }
    }
    float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
    mx0 = fmaxf(mx0, fmaxf(fmaxf(s[2][0], s[2][1]), fmaxf(s[3][0], s[3][1])));
    mx1 = fmaxf(mx1, fmaxf(fmaxf(s[2][2], s[2][3]), fmaxf(s[3][2], s[3][3])));
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
    }
    mx0 *= sl2;
    mx1 *= sl2;
    // Lazy rescale: the reference maximum moves only when a unit's maximum
    // exceeds it by more than RESCALE_SLACK (base-2 logits), so the
    // probabilities stay below 2^RESCALE_SLACK and the values are rarely
    // rescaled; the max-first merge only needs a consistent reference.
    const float mn0 = mx0 > st.m[0] + RESCALE_SLACK ? mx0 : st.m[0];
    const float mn1 = mx1 > st.m[1] + RESCALE_SLACK ? mx1 : st.m[1];
    const float al0 = ex2(st.m[0] - mn0), al1 = ex2(st.m[1] - mn1);
    st.m[0] = mn0;
    st.m[1] = mn1;
    float ps0 = 0.0f, ps1 = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            s[j][e] = ex2(fmaf(s[j][e], sl2, -mn0));
            s[j][e + 2] = ex2(fmaf(s[j][e + 2], sl2, -mn1));
            ps0 += s[j][e];
            ps1 += s[j][e + 2];
        }
    st.l[0] = st.l[0] * al0 + ps0;
    st.l[1] = st.l[1] * al1 + ps1;
    if (__any_sync(0xffffffffu, al0 != 1.0f || al1 != 1.0f)) {
#pragma unroll
        for (int jd = 0; jd < 16; ++jd) {
            st.o[jd][0] *= al0;
            st.o[jd][1] *= al0;
            st.o[jd][2] *= al1;
            st.o[jd][3] *= al1;
        }
    }

#pragma unroll
    for (int kk = 0; kk < 2; ++kk) {
        uint32_t pa[4];
        pa[0] = h2u(__floats2half2_rn(s[2 * kk][0], s[2 * kk][1]));
        pa[1] = h2u(__floats2half2_rn(s[2 * kk][2], s[2 * kk][3]));
        pa[2] = h2u(__floats2half2_rn(s[2 * kk + 1][0], s[2 * kk + 1][1]));
        pa[3] = h2u(__floats2half2_rn(s[2 * kk + 1][2], s[2 * kk + 1][3]));
        uint4 vd[4];
        __half vs[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int cell = 16 * kk + 2 * r + (e & 1) + 8 * (e >> 1);
            vd[e] = *reinterpret_cast<const uint4 *>(V + cell * D + ((g ^ (2 * ((cell >> 1) & 3))) << 4));
            vs[e] = VS[cell * 4 + vgroup<S>(g, dhalf)];
        }
        const __half2 v01 = __halves2half2(vs[0], vs[1]);
        const __half2 v89 = __halves2half2(vs[2], vs[3]);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t w0 = word_of(vd[0], i) ^ 0x80808080u, w1 = word_of(vd[1], i) ^ 0x80808080u;
            const uint32_t w8 = word_of(vd[2], i) ^ 0x80808080u, w9 = word_of(vd[3], i) ^ 0x80808080u;
            __half2 a0, a1, a2, a3, c0, c1, c2, c3;
            codes_to_h2(prmt(w0, w1, 0x5140), a0, a1);
            codes_to_h2(prmt(w0, w1, 0x7362), a2, a3);
            codes_to_h2(prmt(w8, w9, 0x5140), c0, c1);
            codes_to_h2(prmt(w8, w9, 0x7362), c2, c3);
            mma16816(st.o[4 * i + 0], pa, h2u(__hmul2(a0, v01)), h2u(__hmul2(c0, v89)));
            mma16816(st.o[4 * i + 1], pa, h2u(__hmul2(a1, v01)), h2u(__hmul2(c1, v89)));
            mma16816(st.o[4 * i + 2], pa, h2u(__hmul2(a2, v01)), h2u(__hmul2(c2, v89)));
            mma16816(st.o[4 * i + 3], pa, h2u(__hmul2(a3, v01)), h2u(__hmul2(c3, v89)));
        }
    }
}

#ifndef QSA_ATTN_NS
#define QSA_ATTN_NS 2
#endif

// Exchange slots for S == 2: per warp, two parities of 16 floats x 32 lanes.
template <int NW, int S>
__host__ __device__ constexpr int xch_bytes() {
    return S == 2 ? NW * 2 * 16 * 32 * (int)sizeof(float) : 0;
}

template <int NW, int NS, int S>
__global__ void __launch_bounds__(NW * 32, QSA_ATTN_MINB) attn_staged_kernel(AttnLaunch a) {
    extern __shared__ __align__(16) uint8_t smem8[];
    wait_for_previous_grid();  // launched as a programmatic dependent: inputs may come from the previous kernel
    constexpr int NP = NW / S;  // unit groups per CTA
    const int t = a.ntok - 1 - (int)blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, r = lane & 3;
    const int pw = warp / S, half = warp % S;
    const Geom geo = make_geom<S>(a, half);
    // |scale| in base 2, floored at the smallest normal float: a zero scale
    // then still gives exactly uniform weights (every logit rounds to 0) while
    // a masked -inf stays -inf instead of becoming -inf * 0.
    const float sl2 = fmaxf(fabsf(a.softmax_scale) * LOG2E, 1.17549435e-38f);
    const int32_t *idrow = a.ids + (size_t)t * a.width;
    const int nunits = a.width / UNIT;
    uint8_t *ring = smem8 + warp * NS * STAGE_BYTES;
    const uint32_t ring_s = static_cast<uint32_t>(__cvta_generic_to_shared(ring));
    float *xch = reinterpret_cast<float *>(smem8 + NW * NS * STAGE_BYTES);
    // One copy of the Q fragments per dim half, written by the first group.
    uint4 *qfrag = reinterpret_cast<uint4 *>(smem8 + NW * NS * STAGE_BYTES + xch_bytes<NW, S>());
    if (pw == 0) {
        uint32_t qa[8][4];
        load_q<S>(a, t, geo, qa, a.softmax_scale < 0.0f);
        uint4 *dst = qfrag + half * (QFRAG_BYTES / 16) + lane;
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[32 * k] = make_uint4(qa[k][0], qa[k][1], qa[k][2], qa[k][3]);
    }
    __syncthreads();
    QSmem qsrc{qfrag + half * (QFRAG_BYTES / 16) + lane};
    State st;
    state_init(st);
    bool bad = false;

    // My group's units are u_i = pw + i*NP, i = 0 .. n-1.  A unit's ids are
    // loaded one whole unit before its copies are issued (a ring of NS + 1
    // registers), so the load's latency hides behind a unit of compute; they
    // are validated when the copies are issued.
    const int n = pw < nunits ? (nunits - pw + NP - 1) / NP : 0;
    auto raw_id = [&](int i) -> int {
        return i < n && QSA_IN((size_t)t * a.width + (pw + i * NP) * UNIT + lane, (size_t)a.ntok * a.width)
                   ? __ldg(idrow + (pw + i * NP) * UNIT + lane)
                   : -1;
    };
    auto check_id = [&](int id) -> int {
        bad |= (id < -1) || (id >= a.cache_cells);
        return (id >= 0 && id < a.cache_cells) ? id : -1;
    };
    constexpr int NQ = NS + 1;
    int idq[NQ];  // ids of units i .. i+NS (validated once issued)
#pragma unroll
    for (int k = 0; k < NQ; ++k) idq[k] = raw_id(k);
#pragma unroll
    for (int k = 0; k < NS - 1; ++k) {
        idq[k] = check_id(idq[k]);
        if (__any_sync(0xffffffffu, idq[k] >= 0)) issue_unit<S>(a, idq[k], ring_s + k * STAGE_BYTES, geo);
        cp_commit();
    }
    int nx = 0;   // exchanges so far: their parity picks the slot (skipped units exchange nothing)
    for (int i = 0; i < n; ++i) {
        const int sI = i % NS;
        const int sN = (i + NS - 1) % NS;
        const int qI = i % NQ, qN = (i + NS - 1) % NQ, qL = (i + NS) % NQ;
        int id_i = 0, id_n = 0;
#pragma unroll
        for (int k = 0; k < NQ; ++k) {
            if (k == qI) id_i = idq[k];
            if (k == qN) id_n = idq[k];
        }
        if (i + NS - 1 < n) {
            id_n = check_id(id_n);
            if (__any_sync(0xffffffffu, id_n >= 0)) issue_unit<S>(a, id_n, ring_s + sN * STAGE_BYTES, geo);
#pragma unroll
            for (int k = 0; k < NQ; ++k)
                if (k == qN) idq[k] = id_n;
        }
        cp_commit();
        // Unit i + NS's ids, used when its copies are issued next iteration;
        // kept in their own register until this unit is computed, so that
        // nothing waits for the load before then.
        const int nid = raw_id(i + NS);
        cp_wait<NS - 1>();
        __syncwarp();
        const unsigned vmask = __ballot_sync(0xffffffffu, id_i >= 0);  // the same in both warps of a group
        if (vmask) compute_staged<S>(ring + sI * STAGE_BYTES, vmask, qsrc, st, sl2, half, xch, nx++ & 1);
        __syncwarp();
#pragma unroll
        for (int k = 0; k < NQ; ++k)
            if (k == qL) idq[k] = nid;
    }
    cp_wait<0>();
    if (__any_sync(0xffffffffu, bad) && lane == 0 && a.err) atomicOr(a.err, QSA_DEVERR_BAD_ID);
    quad_sum_l(st);
    __syncthreads();

    // Merge: reuse the rings (all copies have landed) for the groups' states.
    // Value (h, d) of group w sits at (16 w + h) DR + (d ^ 4 x), x = 2 (d / 32)
    // + (h & 1).  A 16-byte store is served eight lanes at a time, and the
    // eight lanes (g, r) with g in {2k, 2k+1} then hit eight different
    // 16-byte bank groups: four wavefronts per store instruction, the fewest
    // 512 bytes allow.  The XOR stays inside each 32-float block, so the
    // reads of consecutive d are conflict-free.
    constexpr int DR = D * S;  // row length
    float *so = reinterpret_cast<float *>(smem8);
    float *sm = so + NP * 16 * DR;
    float *sl = sm + NP * 16;
    float *ow = so + pw * 16 * DR + D * half;
    const int sw = 4 * ((2 * r + (g & 1)) & 7);
#pragma unroll
    for (int jd = 0; jd < 16; jd += 4) {
        const int d0 = (32 * r + jd) ^ sw, d1 = (32 * r + 16 + jd) ^ sw;
        *reinterpret_cast<float4 *>(ow + g * DR + d0) =
            make_float4(st.o[jd][0], st.o[jd + 1][0], st.o[jd + 2][0], st.o[jd + 3][0]);
        *reinterpret_cast<float4 *>(ow + g * DR + d1) =
            make_float4(st.o[jd][1], st.o[jd + 1][1], st.o[jd + 2][1], st.o[jd + 3][1]);
        *reinterpret_cast<float4 *>(ow + (g + 8) * DR + d0) =
            make_float4(st.o[jd][2], st.o[jd + 1][2], st.o[jd + 2][2], st.o[jd + 3][2]);
        *reinterpret_cast<float4 *>(ow + (g + 8) * DR + d1) =
            make_float4(st.o[jd][3], st.o[jd + 1][3], st.o[jd + 2][3], st.o[jd + 3][3]);
    }
    if (r == 0 && half == 0) {
        sm[pw * 16 + g] = st.m[0];
        sm[pw * 16 + g + 8] = st.m[1];
        sl[pw * 16 + g] = st.l[0];
        sl[pw * 16 + g + 8] = st.l[1];
    }
    __syncthreads();
    // Per head: M = max over the groups, and group w's weight 2^(m_w - M) / L
    // with L = sum_w 2^(m_w - M) l_w (0 for a head with no valid cell, whose
    // output is then +0), computed once rather than per output element.
    float *sf = sl + NP * 16;
    if (threadIdx.x < 16) {
        const int h = threadIdx.x;
        float M = -CUDART_INF_F;
#pragma unroll
        for (int w = 0; w < NP; ++w) M = fmaxf(M, sm[w * 16 + h]);
        float f[NP], L = 0.0f;
#pragma unroll
        for (int w = 0; w < NP; ++w) {
            const float mw = sm[w * 16 + h];
            f[w] = mw == -CUDART_INF_F ? 0.0f : exp2f(mw - M);
            L += f[w] * sl[w * 16 + h];
        }
        const float inv = M == -CUDART_INF_F ? 0.0f : 1.0f / L;
#pragma unroll
        for (int w = 0; w < NP; ++w) sf[w * 16 + h] = f[w] * inv;
    }
    __syncthreads();
    // Two adjacent dims per thread: d and d + 1 sit next to each other under
    // the swizzle (it moves 4-float blocks), and their outputs are one half2.
    for (int idx = threadIdx.x; idx < geo.per * (DR / 2); idx += NW * 32) {
        const int h = idx / (DR / 2), d = 2 * (idx % (DR / 2));
        const int pd = d ^ (4 * ((2 * (d >> 5) + (h & 1)) & 7));
        float r0 = 0.0f, r1 = 0.0f;
#pragma unroll
        for (int w = 0; w < NP; ++w) {
            const float fw = sf[w * 16 + h];
            const float2 o = *reinterpret_cast<const float2 *>(so + (w * 16 + h) * DR + pd);
            r0 = fmaf(fw, o.x, r0);
            r1 = fmaf(fw, o.y, r1);
        }
        const size_t oi = ((size_t)t * a.n_q_heads + geo.h0 + h) * DR + d;
        if (!QSA_IN(oi + 1, (size_t)a.ntok * a.n_q_heads * DR)) continue;
        const __half2 hv = __floats2half2_rn(gated(a, oi, r0), gated(a, oi + 1, r1));
        *reinterpret_cast<__half2 *>(a.out + oi) = hv;
    }
}

// Split path, part 1: one group of S warps per (token, KV head, 64-cell
// chunk) writes the chunk's unnormalised values, maximum (natural-log units)
// and denominator.
template <int NW, int S>
__global__ void __launch_bounds__(NW * 32) attn_chunk_kernel(AttnLaunch a) {
    constexpr int NP = NW / S;
    constexpr int DR = D * S;
    __shared__ float xch[S == 2 ? NW * 2 * 16 * 32 : 1];
    wait_for_previous_grid();  // launched as a programmatic dependent: q and ids may come from the kernel before
    allow_dependent_launch();  // the merge may be scheduled; it waits for this grid's completion
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, r = lane & 3;
    const int pw = warp / S, half = warp % S;
    const Geom geo = make_geom<S>(a, half);
    const int nch = a.width / CHUNK;
    const int c = blockIdx.z * NP + pw;
    if (c >= nch) return;  // both warps of a group leave together
    const float sl2 = a.softmax_scale * LOG2E;
    const int32_t *idrow = a.ids + (size_t)t * a.width;
    QRegs qsrc;
    load_q<S>(a, t, geo, qsrc.qa);
    State st;
    state_init(st);
    bool bad = false;
    const bool idok = QSA_IN((size_t)t * a.width + c * CHUNK + UNIT + lane, (size_t)a.ntok * a.width);
    const int id0 = idok ? __ldg(idrow + c * CHUNK + lane) : -1, id1 = idok ? __ldg(idrow + c * CHUNK + UNIT + lane) : -1;
    process_unit<S>(a, id0, qsrc, st, sl2, bad, geo, xch, 0);
    process_unit<S>(a, id1, qsrc, st, sl2, bad, geo, xch, 1);
    if (__any_sync(0xffffffffu, bad) && lane == 0 && a.err) atomicOr(a.err, QSA_DEVERR_BAD_ID);
    quad_sum_l(st);
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
        const int h = g + 8 * hf;
        if (h >= geo.per) continue;
        const size_t pbase = (((size_t)t * nch + c) * a.n_q_heads + geo.h0 + h) * (DR + 2);
        if (!QSA_IN(pbase + DR + 1, (size_t)a.ntok * nch * a.n_q_heads * (DR + 2))) continue;
        float *dst = a.part + pbase;
#pragma unroll
        for (int jd = 0; jd < 16; ++jd) {
            dst[D * half + 32 * r + jd] = st.o[jd][2 * hf];
            dst[D * half + 32 * r + 16 + jd] = st.o[jd][2 * hf + 1];
        }
        if (r == 0 && half == 0) {
            const float mm = st.m[hf];
            dst[DR] = mm == -CUDART_INF_F ? mm : mm * LN2;
            dst[DR + 1] = st.l[hf];
        }
    }
}

// Split path, part 2: max-first merge of the chunk partials of one (token,
// query head); a token's heads merge in parallel blocks (grid y, striding
// when there are more heads than grid rows).
template <int S>
__global__ void __launch_bounds__(D * S) attn_merge_kernel(AttnLaunch a) {
    constexpr int DR = D * S;
    wait_for_previous_grid();  // the chunk partials of the grid before
    const int t = blockIdx.x, d = threadIdx.x;
    const int nch = a.width / CHUNK;
    for (int h = blockIdx.y; h < a.n_q_heads; h += gridDim.y) {
        if (!QSA_IN(((size_t)t * nch * a.n_q_heads + h) * (DR + 2) + (size_t)(nch - 1) * a.n_q_heads * (DR + 2) + DR + 1,
                    (size_t)a.ntok * nch * a.n_q_heads * (DR + 2)))
            continue;
        const float *base = a.part + ((size_t)t * nch * a.n_q_heads + h) * (DR + 2);
        const size_t cstride = (size_t)a.n_q_heads * (DR + 2);
        float M = -CUDART_INF_F;
        for (int c = 0; c < nch; ++c) M = fmaxf(M, base[c * cstride + DR]);
        float res = 0.0f;
        if (M != -CUDART_INF_F) {
            float L = 0.0f, O = 0.0f;
            for (int c = 0; c < nch; ++c) {
                const float mc = base[c * cstride + DR];
                if (mc == -CUDART_INF_F) continue;
                const float w = expf(mc - M);
                L += w * base[c * cstride + DR + 1];
                O += w * base[c * cstride + d];
            }
            res = O / L;
        }
        const size_t oi = ((size_t)t * a.n_q_heads + h) * DR + d;
        if (QSA_IN(oi, (size_t)a.ntok * a.n_q_heads * DR)) a.out[oi] = __half_as_ushort(__float2half_rn(gated(a, oi, res)));
    }
}

template <int NW, int NS, int S>
cudaError_t launch_staged(const AttnLaunch &a, cudaStream_t s) {
    size_t smem = (size_t)NW * NS * STAGE_BYTES + xch_bytes<NW, S>() + (size_t)S * QFRAG_BYTES;
    const size_t merge = (size_t)(NW / S) * (16 * D * S + 48) * sizeof(float);
    if (smem < merge) smem = merge;
    cudaError_t e = cudaFuncSetAttribute(attn_staged_kernel<NW, NS, S>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    return launch_dependent(attn_staged_kernel<NW, NS, S>, dim3(a.ntok, a.n_kv_heads), dim3(NW * 32), smem, s, a);
}

template <int S>
cudaError_t launch_split(const AttnLaunch &a, cudaStream_t s) {
    constexpr int NW = 4;
    const int nch = a.width / CHUNK;
    const dim3 grid(a.ntok, a.n_kv_heads, (nch + NW / S - 1) / (NW / S));
    cudaError_t e = launch_dependent(attn_chunk_kernel<NW, S>, grid, dim3(NW * 32), 0, s, a);
    if (e != cudaSuccess) return e;
    return launch_dependent(attn_merge_kernel<S>, dim3(a.ntok, a.n_q_heads < 65535 ? a.n_q_heads : 65535), dim3(D * S),
                            0, s, a);
}

}  // namespace

cudaError_t launch_attn(const AttnLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    const bool wide = a.head_dim == 2 * D;
    if (a.part) return wide ? launch_split<2>(a, s) : launch_split<1>(a, s);
#ifndef QSA_ATTN_NW
#define QSA_ATTN_NW 4
#endif
    return wide ? launch_staged<QSA_ATTN_NW, QSA_ATTN_NS, 2>(a, s) : launch_staged<QSA_ATTN_NW, QSA_ATTN_NS, 1>(a, s);
}

}  // namespace qsa

QSA_DEFINE_CHECK_READER(take_check_word_attn)
