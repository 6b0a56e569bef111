// qsa_score: head-reduced fp32 scores of every causal cache cell.
//
// "Round 36 Track C: qsa_prep Single-Barrier norm_rope & w == 128 tg_sum +
// qsa_score_mm Loop Unrolling", section "Summary & Decision": the score pass
// is a 64x64x128 tile matmul of the queries against the int8 key cache, bound
// by the tensor op and by DRAM reads/writes.  "round 11 track b: qsa attention
// and score", section "score: valid negative result": the tile output is
// reduced over heads; the comparison covers a dead-key tail and untouched
// beyond-causal cells.
//
// The score is linear in q, so
//   S[t,c] = sum_g ksc[c,g] * sum_{d in g} (sum_h q[t,h,d]) * kq[c,d].
// A first kernel forms qbar[t,d] = sum_h q[t,h,d] in fp32 (heads in order) and
// stores it as an fp16 pair hi + lo (hi = fp16(qbar), lo = fp16(qbar - hi)),
// which carries ~22 significant bits.
//
// The key side folds each cell's group scales into its codes.  With e_c the
// power of two that puts 127 * max_g |ksc[c,g]| into [2^14, 2^15), the scaled
// key p[c,d] = kq[c,d] * ksc[c,g] * 2^e_c is exact in fp32 (an 8-bit integer
// times an 11-bit significand) and below 2^15, and it splits exactly-enough
// into fp16 hi = fp16(p), lo = fp16(p - hi) (the remainder has at most 7
// significant bits; it is exact unless it falls below fp16's normal range).
// Then
//   S[t,c] = 2^-e_c * sum_d (hi + lo)[c,d] * (hi + lo)[t,d]
// and dropping lo x lo (below 2^-22 of each product) leaves three fp16
// products per 16-deep k-step, all into ONE fp32 accumulator per output:
// there is no per-group accumulator, and the epilogue is one multiply by
// 2^-e_c (exact) per value.
//
// Kernel layout: one persistent CTA per SM owns a contiguous range of
// (token tile, cell tile) pairs, 128 x 128 each, and runs it as a
// warp-specialised pipeline:
//  - eight producer warps turn a cell tile's int8 codes and scales into the
//    hi and lo key planes of one of two A stages in TENSOR memory (lane =
//    cell, two fp16 per 32-bit column, written with tcgen05.st), and copy
//    qbar hi/lo of 128 tokens into one of two shared-memory B buffers
//    (128-byte-swizzled K-major) when the token tile changes;
//  - one thread issues 8 k-steps x 3 tcgen05.mma (M = 128 cells, N = 128
//    tokens, K = 16; A read from tensor memory, B through a shared-memory
//    descriptor) into one of two accumulators in tensor memory (2 x 128
//    columns);
//  - eight epilogue warps drain the other accumulator: each thread holds one
//    cell and 64 token columns, so every store instruction writes 32
//    consecutive cells of one score row (128 bytes).
// Every mbarrier wait is bounded; on expiry the kernel records
// QSA_DEVERR_TIMEOUT and all roles stop; the MMA thread then waits (bounded)
// for the MMAs it has issued, and only then is tensor memory freed and the
// kernel returns.
#include <cuda_fp16.h>

#include <mutex>

#include "check.cuh"
#include "qsa.h"
#include "qsa_internal.h"
#include "tc_common.cuh"

namespace qsa {
namespace {

constexpr int D = 128;
constexpr int TM = 128;      // cells per tile (MMA M)
constexpr int TN = 128;      // tokens per tile (MMA N)
constexpr int NEPI = 8;      // epilogue warps 0..7 (TMEM lane quarter w % 4, token half w / 4)
constexpr int NPROD = 8;     // producer warps 8..15
constexpr int MMA_WARP = 16; // TMEM owner / MMA issuer
constexpr int THREADS = 32 * 17;
constexpr int PT = NPROD * 32;  // producer threads
constexpr int NA = 2;        // A stages (in tensor memory)
// Tensor memory: two fp32 accumulators of TN columns, then NA key stages of
// D/2 hi columns and D/2 lo columns (two fp16 per 32-bit column, lane = cell).
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_COL = 2 * TN;
constexpr uint32_t A_STAGE_COLS = D;
static_assert(A_COL + NA * A_STAGE_COLS <= TMEM_COLS, "tensor memory layout");
constexpr uint32_t PLANE = TN * D * 2;          // one fp16 qbar plane (hi or lo) in shared memory: 32 KB
constexpr uint32_t KBLOCK = TN * 128;           // bytes of one 64-wide K block of a plane
constexpr uint32_t B_PAIR = 2 * PLANE;          // qbar hi + lo of one token tile
constexpr uint32_t OFF_BAR = 2 * B_PAIR;        // two token tiles in flight
constexpr uint32_t OFF_FLAG = OFF_BAR + (2 * NA + 9) * 8;
constexpr uint32_t SMEM_USED = OFF_FLAG + 16;
// All 512 tensor-memory columns and more than half of the shared memory: one
// CTA per SM.
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;

static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory layout");
// A second CTA on the SM would wait for tensor-memory columns the first holds.
static_assert(2 * SMEM_ALLOC > 227 * 1024, "one CTA per SM");

using namespace tc;

// Instruction descriptor of the score tile: M = 128 cells, N = 128 tokens,
// fp16 operands (both K-major), fp32 accumulation.
constexpr uint32_t IDESC = idesc_f16(TM, TN, false, false);

// D (tensor memory) (+)= A (tensor memory, lane = row, two fp16 of K per
// 32-bit column) x B (shared-memory descriptor).
__device__ __forceinline__ void mma_f16_ts(uint32_t dtmem, uint32_t atmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(dtmem),
        "r"(atmem), "l"(bdesc), "r"(idesc), "r"(acc));
}

// --- kernels ----------------------------------------------------------------

// qbar = sum over heads, split into fp16 hi/lo rows; rows >= ntok are zero.
template <bool F16>
__global__ void __launch_bounds__(D) qsum_kernel(ScoreLaunch a) {
    const int t = blockIdx.x, d = threadIdx.x;
    // Heads added in order from +0 (the order qsa_prep's head sum uses too);
    // the loads are issued sixteen heads at a time so that a token's rows
    // cost one memory round trip per sixteen heads, not one per head.
    constexpr int HB = 16;
    float s = 0.0f;
    if (t < a.ntok) {
        for (int h0 = 0; h0 < a.n_q_heads; h0 += HB) {
            float v[HB];
#pragma unroll
            for (int i = 0; i < HB; ++i) {
                const int h = h0 + i;
                const size_t off = ((size_t)t * a.n_q_heads + h) * D + d;
                v[i] = h >= a.n_q_heads || !QSA_IN(off, (size_t)a.ntok * a.n_q_heads * D) ? 0.0f
                       : F16          ? __half2float(__ldg(reinterpret_cast<const __half *>(a.q) + off))
                                      : __ldg(reinterpret_cast<const float *>(a.q) + off);
            }
#pragma unroll
            for (int i = 0; i < HB; ++i)
                if (h0 + i < a.n_q_heads) s += v[i];
        }
    }
    // The token's power of two (the same rule and order as qsa_prep's head
    // sum, so both write the same workspace bit for bit).
    __shared__ float wmax[D / 32];
    float m = fabsf(s);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((d & 31) == 0) wmax[d >> 5] = m;
    __syncthreads();
    m = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    const int e = head_sum_exponent(m);
    const float v = s * exp2i(e);
    const __half hi = __float2half_rn(v);
    const __half lo = __float2half_rn(v - __half2float(hi));
    if (!QSA_IN(t, (a.ntok + 63) / 64 * 64)) return;
    a.qsum[(size_t)t * 2 * D + d] = __half_as_ushort(hi);
    a.qsum[(size_t)t * 2 * D + D + d] = __half_as_ushort(lo);
    if (d == 0) a.qexp[t] = e;
}

__device__ __forceinline__ int cell_tiles(const ScoreLaunch &a, int tt) {
    const int tl = min(a.ntok - 1, tt * TN + TN - 1);
    return (a.pos0 + tl) / TM + 1;
}

// A cell's power-of-two exponent e_c: 127 * max_g |ksc[c,g]| * 2^e_c lies in
// [2^14, 2^15), so every scaled key kq * ksc * 2^e_c is below 2^15 (fp16 holds
// it) and the largest ones keep fp16's full 11-bit significand.  A cell whose
// scales are all zero gets e_c = 0; one with an infinite or NaN scale too (its
// scores are then not finite either way).
__device__ __forceinline__ int cell_exponent(uint2 kv) {
    const uint32_t m01 = max(kv.x & 0x7FFFu, (kv.x >> 16) & 0x7FFFu);
    const uint32_t m23 = max(kv.y & 0x7FFFu, (kv.y >> 16) & 0x7FFFu);
    const uint32_t mb = max(m01, m23);  // |fp16| bit patterns order like their values
    if (mb == 0u || mb >= 0x7C00u) return 0;
    const float f = 127.0f * __half2float(__ushort_as_half((unsigned short)mb));  // exact, normal in fp32
    return 14 - ((int)((__float_as_uint(f) >> 23) & 0xFFu) - 127);
}
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }

// Scaled scale ksc * 2^e of one group as an fp16 pair (both halves equal).
__device__ __forceinline__ __half2 scaled_scale(uint32_t raw16, float p2) {
    const __half h = __float2half_rn(__half2float(__ushort_as_half((unsigned short)raw16)) * p2);
    return __halves2half2(h, h);
}

// Eight consecutive 32-bit columns of tensor memory for the warp's 32 lanes.
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&v)[8]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};\n" ::"r"(taddr), "r"(v[0]),
                 "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7])
                 : "memory");
}

__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes));
}

struct Walker {
    int tt, ct, ncur;
};

__device__ __forceinline__ void walk_next(const ScoreLaunch &a, Walker &w) {
    if (++w.ct >= w.ncur) {
        w.ct = 0;
        ++w.tt;
        w.ncur = cell_tiles(a, w.tt);
    }
}

// Byte offset of 16-byte unit `u` (0..15 along the 128 dims) of row `r` in a
// 128-row fp16 plane laid out K-major with the 128-byte swizzle.
__device__ __forceinline__ uint32_t plane_off(int r, int u) {
    return (uint32_t)((u >> 3) * KBLOCK + (r >> 3) * 1024 + (r & 7) * 128 + (((u & 7) ^ (r & 7)) << 4));
}

// Warp roles: warps 0-7 drain the accumulators (epilogue; warp w owns TMEM
// lanes 32(w%4).. i.e. cells 32(w%4).. of the tile, and token columns
// 64(w/4)..+63), warps 8-15 produce the operands (scaled key planes into the
// A stages, qbar hi/lo into the B buffer by cp.async), warp 16 allocates
// tensor memory and one of its threads issues the MMAs.  Stages are handed
// over with mbarriers: a_full / a_empty (NA A stages), b_full / b_empty (the
// B buffer), acc_full / acc_empty (2 TMEM accumulators).
// 72 registers a thread (544 x 72 = 39 K a CTA, no spills): a score CTA then
// leaves room on its SM for one attention CTA.
__global__ void __maxnreg__(72) score_kernel(ScoreLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gen = smem_raw + (base - raw);
    const uint32_t sB = base, bar = base + OFF_BAR;
    const uint32_t a_full = bar, a_empty = bar + 8 * NA, b_full = bar + 16 * NA, b_empty = b_full + 16,
                   acc_full = b_empty + 16, acc_empty = acc_full + 16, drain = acc_empty + 16;
    volatile int *abort = reinterpret_cast<volatile int *>(gen + OFF_FLAG);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gen + OFF_FLAG + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    wait_for_previous_grid();  // launched as a programmatic dependent: the head sum may come from qsa_prep
    allow_dependent_launch();

    if (tid == 0) {
        for (int i = 0; i < NA; ++i) {
            mbar_init(a_full + 8 * i, PT);
            mbar_init(a_empty + 8 * i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(b_full + 8 * i, PT);  // one cp.async-tracked arrival per producer thread
            mbar_init(b_empty + 8 * i, 1);
            mbar_init(acc_full + 8 * i, 1);
            mbar_init(acc_empty + 8 * i, NEPI * 32);
        }
        mbar_init(drain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == MMA_WARP) tmem_alloc(smem_u32((const void *)tslot), TMEM_COLS);
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = *tslot;

    // This CTA's contiguous share of the (token tile, cell tile) sequence.
    const int ntt = (a.ntok + TN - 1) / TN;
    long long total = 0;
    for (int tt = 0; tt < ntt; ++tt) total += cell_tiles(a, tt);
    const long long begin = total * blockIdx.x / gridDim.x;
    const long long end = total * (blockIdx.x + 1) / gridDim.x;
    const int n = (int)(end - begin);
    Walker w0{0, 0, 0};
    {
        long long k = begin;
        while (w0.tt < ntt && k >= cell_tiles(a, w0.tt)) {
            k -= cell_tiles(a, w0.tt);
            ++w0.tt;
        }
        w0.ct = (int)k;
        w0.ncur = cell_tiles(a, w0.tt);
    }

    if (warp >= NEPI && warp < NEPI + NPROD) {
        // ---- producers ----
        // Producer warp p (0..7) owns tensor-memory lane quarter p % 4 and
        // dims 64(p / 4) .. +63: each thread converts one cell's 64 codes
        // (two scale groups) into 32 hi and 32 lo columns of the A stage.
        const int pt = tid - NEPI * 32, pw = warp - NEPI, quarter = pw & 3, kh = pw >> 2;
        const int row = quarter * 32 + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        Walker w = w0;
        int nb = 0, cur_tt = -1;
        uint4 pre[4];
        uint2 psc;
        auto load_a = [&](int ct) {
            const int c = ct * TM + row;
            const bool ok = c < a.cache_cells && QSA_IN((size_t)c * D + kh * 64 + 63, (size_t)a.cache_cells * D);
            const uint4 *src = reinterpret_cast<const uint4 *>(a.kq + (size_t)c * D + kh * 64);
#pragma unroll
            for (int i = 0; i < 4; ++i) pre[i] = ok ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
            psc = ok ? __ldg(reinterpret_cast<const uint2 *>(a.ksc + (size_t)c * 4)) : make_uint2(0u, 0u);
        };
        if (n > 0) load_a(w.ct);
        for (int k = 0; k < n; ++k) {
            if (w.tt != cur_tt) {
                // qbar hi/lo rows of the new token tile (rows past ntok read
                // as zero) into one of two B buffers, completing on b_full.
                const int bs = nb & 1;
                if (nb >= 2 && !mbar_wait_or_abort(b_empty + 8 * bs, ((nb >> 1) - 1) & 1, abort)) break;
                const uint32_t dstB = sB + bs * B_PAIR;
#pragma unroll 4
                for (int it = 0; it < 2 * TN * 16 / PT; ++it) {
                    const int q = it * PT + pt, part = q / (TN * 16), r = (q / 16) % TN, u = q & 15;
                    const int t = w.tt * TN + r;
                    const bool ok = t < a.ntok && QSA_IN(t, (a.ntok + 63) / 64 * 64);
                    cp_async16_zfill(dstB + part * PLANE + plane_off(r, u),
                                     reinterpret_cast<const uint4 *>(a.qsum + ((size_t)(ok ? t : 0) * 2 + part) * D) + u,
                                     ok ? 16u : 0u);
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(b_full + 8 * bs)
                             : "memory");
                ++nb;
                cur_tt = w.tt;
            }
            const int st = k % NA;
            if (k >= NA && !mbar_wait_or_abort(a_empty + 8 * st, ((k / NA) - 1) & 1, abort)) break;
            fence_after();
            const float p2 = pow2f(cell_exponent(psc));
            const uint32_t graw = kh ? psc.y : psc.x;  // this thread's two scale groups
            const __half2 sg[2] = {scaled_scale(graw & 0xFFFFu, p2), scaled_scale(graw >> 16, p2)};
            const uint32_t col = lane_base + A_COL + st * A_STAGE_COLS + kh * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) {  // 16 codes (half a scale group): 8 hi and 8 lo columns
                uint32_t h[8], hi[8], lo[8];
                codes_to_h2(pre[i].x ^ 0x80808080u, h[0], h[1]);
                codes_to_h2(pre[i].y ^ 0x80808080u, h[2], h[3]);
                codes_to_h2(pre[i].z ^ 0x80808080u, h[4], h[5]);
                codes_to_h2(pre[i].w ^ 0x80808080u, h[6], h[7]);
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    // hi = fp16(k * s); lo = fp16(k * s - hi), one rounding (fused).
                    const __half2 kk = *reinterpret_cast<const __half2 *>(&h[j]);
                    const __half2 vh = __hmul2(kk, sg[i >> 1]);
                    const __half2 vl = __hfma2(kk, sg[i >> 1], __hneg2(vh));
                    hi[j] = *reinterpret_cast<const uint32_t *>(&vh);
                    lo[j] = *reinterpret_cast<const uint32_t *>(&vl);
                }
                tmem_st8(col + 8 * i, hi);
                tmem_st8(col + D / 2 + 8 * i, lo);
            }
            tmem_wait_st();
            fence_before();
            mbar_arrive(a_full + 8 * st);
            walk_next(a, w);
            if (k + 1 < n) load_a(w.ct);
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == MMA_WARP) {
        // ---- MMA issuer ----
        if (lane == 0) {
            Walker w = w0;
            int nb = 0, cur_tt = -1, bs = 0;
            bool issued = false;
            for (int k = 0; k < n; ++k) {
                if (w.tt != cur_tt) {
                    bs = nb & 1;
                    if (!mbar_wait_or_abort(b_full + 8 * bs, (nb >> 1) & 1, abort)) break;
                    ++nb;
                    cur_tt = w.tt;
                }
                const int st = k % NA, b = k & 1;
                if (!mbar_wait_or_abort(a_full + 8 * st, (k / NA) & 1, abort)) break;
                if (k >= 2 && !mbar_wait_or_abort(acc_empty + 8 * b, ((k >> 1) - 1) & 1, abort)) break;
                fence_after();
                const uint32_t ah = tmem + A_COL + st * A_STAGE_COLS, al = ah + D / 2;
                const uint64_t bh = sw128_kmajor(sB + bs * B_PAIR), bl = sw128_kmajor(sB + bs * B_PAIR + PLANE);
                const uint32_t dt = tmem + (uint32_t)(b * TN);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    // k-step ks: dims 16ks..16ks+15 -- A columns 8ks..8ks+7, B K block
                    // ks / 4 at byte 32 (ks % 4).
                    const uint64_t koff = (uint64_t)(((ks >> 2) * KBLOCK + (ks & 3) * 32) >> 4);
                    mma_f16_ts(dt, ah + 8 * ks, bh + koff, IDESC, ks ? 1u : 0u);
                    mma_f16_ts(dt, ah + 8 * ks, bl + koff, IDESC, 1u);
                    mma_f16_ts(dt, al + 8 * ks, bh + koff, IDESC, 1u);
                }
                issued = true;
                mma_commit(a_empty + 8 * st);
                mma_commit(acc_full + 8 * b);
                Walker nx = w;
                walk_next(a, nx);
                if (k + 1 == n || nx.tt != w.tt) mma_commit(b_empty + 8 * bs);
                w = nx;
            }
            // Whether the loop finished or another role gave up, every MMA this
            // thread issued must be complete before the tensor memory it
            // writes is freed: one more commit tracks all of them.
            if (issued) {
                mma_commit(drain);
                if (!mbar_wait_bounded(drain, 0, DRAIN_LIMIT)) *abort = 1;
            }
        }
    } else if (warp < NEPI) {
        // ---- epilogue ----
        // Thread (warp w, lane l) holds cell c0 + 32(w % 4) + l and token
        // columns 64(w / 4) .. +63, loaded as two 32-column pieces, scales
        // them by 2^-e_c and stores them.  Fully causal tiles store without
        // per-element tests.  For a fixed column the warp's 32
        // lanes store 32 consecutive cells of one score row.
        const int quarter = warp & 3, half = warp >> 2;
        const int ntok_pad = (a.ntok + 63) / 64 * 64;  // rows of the workspace
        auto cell_scales = [&](const Walker &wk) {
            const int c = wk.ct * TM + quarter * 32 + lane;
            return c < a.cache_cells ? __ldg(reinterpret_cast<const uint2 *>(a.ksc + (size_t)c * 4))
                                     : make_uint2(0u, 0u);
        };
        Walker w = w0;
        uint2 kv = n > 0 ? cell_scales(w) : make_uint2(0u, 0u);
        for (int k = 0; k < n; ++k) {
            const int b = k & 1;
            const int c0 = w.ct * TM, t0 = w.tt * TN;
            const int cell = c0 + quarter * 32 + lane;
            const float inv = pow2f(-cell_exponent(kv));
            // The next tile's scales, loaded now so that their latency hides
            // behind this tile.
            Walker nx = w;
            walk_next(a, nx);
            const uint2 kv_next = k + 1 < n ? cell_scales(nx) : make_uint2(0u, 0u);
            const int tw = t0 + half * (TN / 2);       // first token of this warp's columns
            const bool full = c0 + TM - 1 <= a.pos0 + t0 && t0 + TN <= a.ntok;
            const int tmin = cell - a.pos0;            // first token whose causal range reaches `cell`
            float *col = a.scores + (size_t)tw * a.ld + cell;
            // The head-sum exponents of this warp's 64 token columns, two per
            // lane (tokens past the workspace's rows are never stored).
            const int te = tw + 2 * lane;
            const int2 ex = te < ntok_pad ? __ldg(reinterpret_cast<const int2 *>(a.qexp + te)) : make_int2(0, 0);
            if (!mbar_wait_or_abort(acc_full + 8 * b, (k >> 1) & 1, abort)) break;
            fence_after();
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * TN + half * (TN / 2));
            uint32_t va[16], vb[16];
            auto wait16 = [&]() {
                tmem_wait_ld();
                // Each loaded register passes through an empty volatile
                // statement, so no use of it can move above the wait.
#pragma unroll
                for (int j = 0; j < 16; ++j) asm volatile("" : "+r"(va[j]), "+r"(vb[j]));
            };
            // Tokens whose head sum was scaled (exponent != 0) need their own
            // factor 2^-e_t; in the common case no token of the warp's 64 was.
            const bool unit = __all_sync(0xffffffffu, (ex.x | ex.y) == 0);
            // Streaming stores: the scores are not read again by this pass.
            auto store16 = [&](const uint32_t (&v)[16], int j0) {
                float *p = col + (size_t)j0 * a.ld;
                if (!unit) {
#pragma unroll
                    for (int j = 0; j < 16; ++j, p += a.ld) {
                        const int c = j0 + j, t = tw + c;
                        const float f = exp2i(-__shfl_sync(0xffffffffu, (c & 1) ? ex.y : ex.x, c >> 1));
                        if ((full || (t < a.ntok && t >= tmin)) && QSA_IN((size_t)t * a.ld + cell, (size_t)a.ntok * a.ld) &&
                            QSA_IN(cell, a.ld))
                            __stcs(p, fmaf(__uint_as_float(v[j]), inv, 0.0f) * f);
                    }
                } else if (full) {
#pragma unroll
                    for (int j = 0; j < 16; ++j, p += a.ld)
                        if (QSA_IN((size_t)(tw + j0 + j) * a.ld + cell, (size_t)a.ntok * a.ld) && QSA_IN(cell, a.ld))
                            __stcs(p, fmaf(__uint_as_float(v[j]), inv, 0.0f));
                } else {
#pragma unroll
                    for (int j = 0; j < 16; ++j, p += a.ld) {
                        const int t = tw + j0 + j;
                        if (t < a.ntok && t >= tmin && QSA_IN((size_t)t * a.ld + cell, (size_t)a.ntok * a.ld) &&
                            QSA_IN(cell, a.ld))
                            __stcs(p, fmaf(__uint_as_float(v[j]), inv, 0.0f));
                    }
                }
            };
            tmem_ld16(tbase, va);
            tmem_ld16(tbase + 16, vb);
            wait16();
            store16(va, 0);
            store16(vb, 16);
            tmem_ld16(tbase + 32, va);
            tmem_ld16(tbase + 48, vb);
            wait16();
            fence_before();
            mbar_arrive(acc_empty + 8 * b);
            store16(va, 32);
            store16(vb, 48);
            w = nx;
            kv = kv_next;
        }
    }

    fence_before();
    __syncthreads();
    if (tid == 0 && *abort && a.err) atomicOr(a.err, QSA_DEVERR_TIMEOUT);
    if (warp == MMA_WARP) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

cudaError_t launch_score(const ScoreLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    const int ntok_pad = (a.ntok + 63) / 64 * 64;  // rows of the workspace
    if (!a.qsum_ready) {  // otherwise qsa_prep has written the head sum into the workspace
        if (a.q_f16)
            qsum_kernel<true><<<ntok_pad, D, 0, s>>>(a);
        else
            qsum_kernel<false><<<ntok_pad, D, 0, s>>>(a);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    long long total = 0;
    for (int tt = 0; tt * TN < a.ntok; ++tt) {
        const int tl = (tt * TN + TN - 1 < a.ntok - 1) ? tt * TN + TN - 1 : a.ntok - 1;
        total += (a.pos0 + tl) / TM + 1;
    }
    int grid = (int)(total < sms ? total : sms);
    if (a.max_ctas > 0 && a.max_ctas < grid) grid = a.max_ctas;
    e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    return launch_dependent(score_kernel, dim3(grid), dim3(THREADS), SMEM_ALLOC, s, a);
}

// --- allocation-free variant --------------------------------------------------
//
// For callers that may not allocate device memory when they score (an engine
// that owns all device memory, a loop that must not hit cudaMalloc's device
// synchronisation), the q-bar workspace can instead live in this fixed array,
// which the CUDA module reserves on each device that loads the library and
// keeps until the process exits.  Host code must not pass the symbol itself to
// a kernel (on the host it names a stand-in, not device memory): the device
// address is looked up once per device with that device current.  Calls share
// the array, so calls whose kernels overlap on the GPU race on it.
namespace {

// One workspace of QSA_SCORE_NOALLOC_MAX_TOKENS rows: fp16 hi/lo rows, then
// the per-token exponents.
constexpr size_t kNoAllocBytes = (size_t)QSA_SCORE_NOALLOC_MAX_TOKENS * kScoreWsBytesPerTok;
static __device__ __align__(256) uint8_t g_noalloc_qsum[kNoAllocBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

}  // namespace

cudaError_t launch_score_noalloc(const ScoreLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!g_noalloc_addr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_noalloc_qsum);
            if (e != cudaSuccess) return e;
            g_noalloc_addr[dev] = p;
        }
        scratch = g_noalloc_addr[dev];
    }
    ScoreLaunch b = a;
    const size_t pad = (size_t)(a.ntok + kScoreTokTile - 1) / kScoreTokTile * kScoreTokTile;
    b.qsum = static_cast<uint16_t *>(scratch);
    b.qexp = reinterpret_cast<int *>(static_cast<uint8_t *>(scratch) + pad * kScoreRowBytes);
    return launch_score(b, s);
}

}  // namespace qsa

QSA_DEFINE_CHECK_READER(take_check_word_score)

