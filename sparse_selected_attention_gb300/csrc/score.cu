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
// which carries ~22 significant bits.  The int8 codes are exact in fp16, so
// the second kernel is one 128-cell x 64-token x 128-dim tensor-core tile per
// output block, issued as tcgen05.mma kind::f16 with fp32 accumulators in
// tensor memory: one accumulator per 32-dim scale group (the group scale
// varies along the contraction), each fed by two 16-deep k-steps of hi and of
// lo.  The epilogue combines the four groups with the cell's scales and stores
// the causal cells; the others are never written.  Summing heads first cuts
// the contraction twelvefold, so the pass is bound by its fp32 output writes.
//
// Kernel layout: one persistent CTA per SM owns a contiguous range of
// (token tile, cell tile) pairs and runs it as a warp-specialised pipeline:
// four producer warps convert int8 codes to fp16 into a ring of three A stages
// (and copy qbar hi/lo into one of two B buffers when the token tile
// changes), one thread issues the tcgen05 MMAs into one of two accumulator
// sets in tensor memory (2 x 4 groups x 64 columns = 512 columns), and four
// eight epilogue warps drain the other set to global memory.  Operands use the
// 128-byte-swizzled K-major layout read through shared-memory descriptors.
// Every mbarrier wait is bounded; on expiry the kernel records
// QSA_DEVERR_TIMEOUT, all roles stop, tensor memory is freed and the kernel
// returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>

#include <cstring>
#include <mutex>

#include "qsa.h"
#include "qsa_internal.h"
#include "tc_common.cuh"

namespace qsa {
namespace {

constexpr int D = 128;
constexpr int NG = 4;        // 32-dim scale groups
constexpr int TM = 128;      // cells per tile (MMA M)
constexpr int TN = 64;       // tokens per tile (MMA N)
constexpr int NEPI = 8;      // epilogue warps 0..7 (TMEM lane quarter w % 4, token half w / 4)
constexpr int NPROD = 4;     // producer warps 8..11
constexpr int MMA_WARP = 12; // TMEM owner / MMA issuer
constexpr int THREADS = 32 * 13;
constexpr int PT = NPROD * 32;  // producer threads
constexpr int NA = 3;        // A stages
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_BYTES = TM * D * 2;        // fp16, two 64-wide K blocks
constexpr uint32_t A_KBLOCK = TM * 128;         // bytes of one 64-wide K block
constexpr uint32_t B_BYTES = TN * D * 2;        // one of qbar hi / lo
constexpr uint32_t B_KBLOCK = TN * 128;
constexpr uint32_t B_PAIR = 2 * B_BYTES;        // hi + lo of one token tile
constexpr uint32_t C_BYTES = TN * TM * 4;       // fp32 output tile, token-major
constexpr uint32_t OFF_B = NA * A_BYTES;
constexpr uint32_t OFF_C = OFF_B + 2 * B_PAIR;
constexpr uint32_t OFF_BAR = OFF_C + 2 * C_BYTES;
constexpr uint32_t OFF_FLAG = OFF_BAR + (2 * NA + 8) * 8;
constexpr uint32_t SMEM_USED = OFF_FLAG + 16;
// The layout needs more than half of an SM's shared memory, so exactly one
// CTA (and one 512-column tensor-memory allocation) lives on each SM.
constexpr uint32_t SMEM_ALLOC = SMEM_USED + 1024;

static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory layout");


using namespace tc;

// Instruction descriptor of the score tile: M = 128 cells, N = 64 tokens,
// fp16 operands (both K-major), fp32 accumulation.
constexpr uint32_t IDESC = idesc_f16(TM, TN, false, false);

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
                v[i] = h >= a.n_q_heads ? 0.0f
                       : F16          ? __half2float(__ldg(reinterpret_cast<const __half *>(a.q) + off))
                                      : __ldg(reinterpret_cast<const float *>(a.q) + off);
            }
#pragma unroll
            for (int i = 0; i < HB; ++i)
                if (h0 + i < a.n_q_heads) s += v[i];
        }
    }
    const __half hi = __float2half_rn(s);
    const __half lo = __float2half_rn(s - __half2float(hi));
    a.qsum[(size_t)t * 2 * D + d] = __half_as_ushort(hi);
    a.qsum[(size_t)t * 2 * D + D + d] = __half_as_ushort(lo);
}

struct TileWalk {
    int tt, ct;
};

__device__ __forceinline__ int cell_tiles(const ScoreLaunch &a, int tt) {
    const int tl = min(a.ntok - 1, tt * TN + TN - 1);
    return (a.pos0 + tl) / TM + 1;
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}
// Two fp32 fused multiply-adds in one instruction: (a.lo*b.lo + c.lo, a.hi*b.hi + c.hi).
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ void named_sync_epilogue() { asm volatile("bar.sync 1, %0;" ::"n"(NEPI * 32) : "memory"); }

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(dst), "l"(src));
}

// Eight consecutive 32-bit columns of tensor memory for the warp's 32 lanes.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, uint32_t (&v)[8]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7])
                 : "r"(taddr));
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, int x, int y, uint32_t src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(src)
                 : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
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

// Warp roles: warps 0-7 drain the accumulators (epilogue; warp w owns TMEM
// lanes 32(w%4).. i.e. cells 32(w%4).. of the tile, and token columns
// 32(w/4)..+31), warps 8-11 produce the operands (int8 codes -> fp16 A
// stages, qbar hi/lo -> B buffers by cp.async), warp 12 allocates tensor
// memory and one of its threads issues the MMAs.  Stages
// are handed over with mbarriers: a_full / a_empty (NA A stages), b_full /
// b_empty (2 B buffers, one per token tile in flight), acc_full / acc_empty
// (2 TMEM accumulator sets).
__global__ void __launch_bounds__(THREADS, 1) score_kernel(ScoreLaunch a, const __grid_constant__ CUtensorMap tmap,
                                                            int use_tma) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *gen = smem_raw + (base - raw);
    const uint32_t sA = base, sB = base + OFF_B, sC = base + OFF_C, bar = base + OFF_BAR;
    const uint32_t a_full = bar, a_empty = bar + 8 * NA, b_full = bar + 16 * NA, b_empty = b_full + 16,
                   acc_full = b_empty + 16, acc_empty = acc_full + 16;
    volatile int *abort = reinterpret_cast<volatile int *>(gen + OFF_FLAG);
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gen + OFF_FLAG + 8);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

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
        const int pt = tid - NEPI * 32;
        Walker w = w0;
        int nb = 0, cur_tt = -1;
        uint4 pre[8];
        auto load_a = [&](int ct) {
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int q = it * PT + pt, m = q >> 3, dc = q & 7;
                const int c = ct * TM + m;
                pre[it] = c < a.cache_cells ? __ldg(reinterpret_cast<const uint4 *>(a.kq + (size_t)c * D) + dc)
                                            : make_uint4(0u, 0u, 0u, 0u);
            }
        };
        if (n > 0) load_a(w.ct);
        for (int k = 0; k < n; ++k) {
            if (w.tt != cur_tt) {
                // qbar hi/lo rows of the new token tile: asynchronous copies
                // into the swizzled B buffer, completing on b_full.
                const int bs = nb & 1;
                if (nb >= 2 && !mbar_wait_or_abort(b_empty + 8 * bs, ((nb >> 1) - 1) & 1, abort)) break;
                const uint32_t dstB = sB + bs * B_PAIR;
#pragma unroll
                for (int it = 0; it < 2048 / PT; ++it) {
                    const int q = it * PT + pt, part = q >> 10, row = (q & 1023) >> 4, ci = q & 15;
                    const int kb = ci >> 3, cc = ci & 7;
                    cp_async16(dstB + part * B_BYTES + kb * B_KBLOCK + (row >> 3) * 1024 + (row & 7) * 128 +
                                   ((cc ^ (row & 7)) << 4),
                               reinterpret_cast<const uint4 *>(a.qsum + ((size_t)(w.tt * TN + row) * 2 + part) * D) +
                                   ci);
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(b_full + 8 * bs)
                             : "memory");
                ++nb;
                cur_tt = w.tt;
            }
            const int st = k % NA;
            if (k >= NA && !mbar_wait_or_abort(a_empty + 8 * st, ((k / NA) - 1) & 1, abort)) break;
            const uint32_t dstA = sA + st * A_BYTES;
#pragma unroll
            for (int it = 0; it < 8; ++it) {
                const int q = it * PT + pt, m = q >> 3, dc = q & 7;
                uint32_t h[8];
                codes_to_h2(pre[it].x ^ 0x80808080u, h[0], h[1]);
                codes_to_h2(pre[it].y ^ 0x80808080u, h[2], h[3]);
                codes_to_h2(pre[it].z ^ 0x80808080u, h[4], h[5]);
                codes_to_h2(pre[it].w ^ 0x80808080u, h[6], h[7]);
                const int kb = dc >> 2, cc = 2 * (dc & 3);
                const uint32_t row = dstA + kb * A_KBLOCK + (m >> 3) * 1024 + (m & 7) * 128;
                const uint32_t p0 = row + ((cc ^ (m & 7)) << 4), p1 = row + (((cc + 1) ^ (m & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p0), "r"(h[0]), "r"(h[1]), "r"(h[2]),
                             "r"(h[3]));
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p1), "r"(h[4]), "r"(h[5]), "r"(h[6]),
                             "r"(h[7]));
            }
            fence_async_smem();
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
                const uint64_t ad0 = sw128_kmajor(sA + st * A_BYTES), bd0 = sw128_kmajor(sB + bs * B_PAIR);
#pragma unroll
                for (int s2 = 0; s2 < 2; ++s2)
#pragma unroll
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int g = 0; g < NG; ++g) {
                            // Groups innermost: consecutive MMAs target different
                            // accumulators; only the descriptors' address field moves.
                            const int ksx = 2 * g + s2, kb = ksx >> 2;
                            const uint32_t koff = (ksx & 3) * 32;
                            const uint32_t dt = tmem + (uint32_t)(b * NG * TN + g * TN);
                            mma_f16(dt, ad0 + (uint64_t)((kb * A_KBLOCK + koff) >> 4),
                                    bd0 + (uint64_t)((part * B_BYTES + kb * B_KBLOCK + koff) >> 4), IDESC,
                                    (s2 | part) ? 1u : 0u);
                        }
                mma_commit(a_empty + 8 * st);
                mma_commit(acc_full + 8 * b);
                Walker nx = w;
                walk_next(a, nx);
                if (k + 1 == n || nx.tt != w.tt) mma_commit(b_empty + 8 * bs);
                w = nx;
            }
        }
    } else if (warp < NEPI) {
        // ---- epilogue ----
        // Fully causal tiles are combined into a token-major fp32 tile in
        // shared memory and written by one TMA bulk-tensor store; tiles that
        // cross the causal boundary are stored element-wise under the mask.
        // A warp drains its 32 cells x 32 tokens in four 8-token pieces, the
        // tensor-memory loads of each piece issued before the previous piece
        // is combined and stored, so their latency hides behind that work.
        Walker w = w0;
        int nfull = 0;
        for (int k = 0; k < n; ++k) {
            const int b = k & 1;
            const int c0 = w.ct * TM, t0 = w.tt * TN;
            const bool full = use_tma && (c0 + TM - 1 <= a.pos0 + t0);
            const int quarter = warp & 3, half = warp >> 2;
            const int cell = c0 + quarter * 32 + lane;
            uint2 kv = make_uint2(0u, 0u);
            if (cell < a.cache_cells) kv = __ldg(reinterpret_cast<const uint2 *>(a.ksc + (size_t)cell * NG));
            if (!mbar_wait_or_abort(acc_full + 8 * b, (k >> 1) & 1, abort)) break;
            fence_after();
            const float ks0 = __half2float(__ushort_as_half((unsigned short)(kv.x & 0xFFFF)));
            const float ks1 = __half2float(__ushort_as_half((unsigned short)(kv.x >> 16)));
            const float ks2 = __half2float(__ushort_as_half((unsigned short)(kv.y & 0xFFFF)));
            const float ks3 = __half2float(__ushort_as_half((unsigned short)(kv.y >> 16)));
            const uint64_t k0 = pack2(ks0, ks0), k1 = pack2(ks1, ks1), k2 = pack2(ks2, ks2), k3 = pack2(ks3, ks3);
            const uint32_t cbuf = sC + (nfull & 1) * C_BYTES;
            const uint32_t tbase = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * NG * TN + half * (TN / 2));
            const int tmin = cell - a.pos0;  // first token whose causal range reaches `cell`
            const int tw = t0 + half * (TN / 2);  // first token of this warp's 32 columns
            uint32_t va[NG][8], vb[NG][8];
            auto load8 = [&](uint32_t (&v)[NG][8], int j0) {
#pragma unroll
                for (int g = 0; g < NG; ++g) tmem_ld8(tbase + g * TN + j0, v[g]);
            };
            // After the wait: each loaded register passes through an empty
            // volatile statement, so no use of it can move above the wait.
            auto wait8 = [&](uint32_t (&v)[NG][8]) {
                tmem_wait_ld();
#pragma unroll
                for (int g = 0; g < NG; ++g)
#pragma unroll
                    for (int j = 0; j < 8; ++j) asm volatile("" : "+r"(v[g][j]));
            };
            auto drain8 = [&](const uint32_t (&v)[NG][8], int j0) {
                float o[8];
#pragma unroll
                for (int j = 0; j < 8; j += 2) {
                    uint64_t acc = fma2(k0, pack2(__uint_as_float(v[0][j]), __uint_as_float(v[0][j + 1])), 0ull);
                    acc = fma2(k1, pack2(__uint_as_float(v[1][j]), __uint_as_float(v[1][j + 1])), acc);
                    acc = fma2(k2, pack2(__uint_as_float(v[2][j]), __uint_as_float(v[2][j + 1])), acc);
                    acc = fma2(k3, pack2(__uint_as_float(v[3][j]), __uint_as_float(v[3][j + 1])), acc);
                    o[j] = __uint_as_float((uint32_t)acc);
                    o[j + 1] = __uint_as_float((uint32_t)(acc >> 32));
                }
                const int tj = tw + j0;
                if (full) {
                    const uint32_t dst = cbuf + (uint32_t)((tj - t0) * TM + quarter * 32 + lane) * 4;
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        asm volatile("st.shared.f32 [%0], %1;" ::"r"(dst + j * TM * 4), "f"(o[j]) : "memory");
                } else {
                    float *dst = a.scores + (size_t)tj * a.ld + cell;
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const int t = tj + j;
                        if (t < a.ntok && t >= tmin) dst[(size_t)j * a.ld] = o[j];
                    }
                }
            };
            load8(va, 0);
            wait8(va);
            load8(vb, 8);
            drain8(va, 0);
            wait8(vb);
            load8(va, 16);
            drain8(vb, 8);
            wait8(va);
            load8(vb, 24);
            drain8(va, 16);
            wait8(vb);
            drain8(vb, 24);
            fence_before();
            mbar_arrive(acc_empty + 8 * b);
            if (full) {
                fence_async_smem();
                // The store issued at the previous full tile reads the other
                // buffer, which the next full tile writes: its read must be
                // over before the barrier that lets the writers go on.
                if (tid == 0) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
                named_sync_epilogue();
                if (tid == 0) tma_store_2d(&tmap, c0, t0, cbuf);
                ++nfull;
            }
            walk_next(a, w);
        }
        if (tid == 0) asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
    }

    fence_before();
    __syncthreads();
    if (tid == 0 && *abort && a.err) atomicOr(a.err, QSA_DEVERR_TIMEOUT);
    if (warp == MMA_WARP) {
        fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

}  // namespace

cudaError_t launch_score(const ScoreLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    const int ntok_pad = (a.ntok + TN - 1) / TN * TN;
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
    const int grid = (int)(total < sms ? total : sms);
    e = cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_ALLOC);
    if (e != cudaSuccess) return e;
    // Tensor map of the score rows for the TMA stores of fully causal tiles.
    // It needs 16-byte aligned rows; otherwise every tile takes the masked
    // element-wise path.
    CUtensorMap map;
    std::memset(&map, 0, sizeof map);
    int use_tma = 0;
    if (a.ld % 4 == 0 && (reinterpret_cast<uintptr_t>(a.scores) & 15) == 0) {
        if (auto encode = tensor_map_encoder()) {
            const cuuint64_t dims[2] = {(cuuint64_t)a.ld, (cuuint64_t)a.ntok};
            const cuuint64_t strides[1] = {(cuuint64_t)a.ld * sizeof(float)};
            const cuuint32_t box[2] = {(cuuint32_t)TM, (cuuint32_t)TN};
            const cuuint32_t estr[2] = {1, 1};
            use_tma = encode(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, a.scores, dims, strides, box, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
        }
    }
    score_kernel<<<grid, THREADS, SMEM_ALLOC, s>>>(a, map, use_tma);
    return cudaGetLastError();
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

constexpr size_t kNoAllocElems = (size_t)QSA_SCORE_NOALLOC_MAX_TOKENS * 2 * D;  // fp16 hi/lo rows
static __device__ __align__(256) uint16_t g_noalloc_qsum[kNoAllocElems];

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
    b.qsum = static_cast<uint16_t *>(scratch);
    return launch_score(b, s);
}

}  // namespace qsa
