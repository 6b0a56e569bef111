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
// Kernel layout: one persistent 128-thread CTA per SM owns a contiguous range
// of (token tile, cell tile) pairs.  Operands are written to shared memory by
// the CTA's threads in the 128-byte-swizzled K-major layout and read by the
// tensor core through shared-memory descriptors; accumulators are double
// buffered in tensor memory (2 x 4 groups x 64 columns = 512 columns) so the
// epilogue of tile i overlaps the MMAs of tile i+1.  Every mbarrier wait is
// bounded; on expiry the kernel records QSA_DEVERR_TIMEOUT, stops, frees its
// tensor memory and returns.
#include <cuda_fp16.h>

#include <mutex>

#include "qsa.h"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int D = 128;
constexpr int NG = 4;        // 32-dim scale groups
constexpr int TM = 128;      // cells per tile (MMA M)
constexpr int TN = 64;       // tokens per tile (MMA N)
constexpr int THREADS = 128;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t A_BYTES = TM * D * 2;        // fp16, two 64-wide K blocks
constexpr uint32_t A_KBLOCK = TM * 128;         // bytes of one 64-wide K block
constexpr uint32_t B_BYTES = TN * D * 2;
constexpr uint32_t B_KBLOCK = TN * 128;
constexpr uint32_t SMEM_USED = 2 * A_BYTES + 2 * B_BYTES + 64;
// Ask for more than half of an SM's shared memory so exactly one CTA (and one
// 512-column tensor-memory allocation) lives on each SM.
constexpr uint32_t SMEM_ALLOC = 120 * 1024;
constexpr long long WAIT_LIMIT = 1ll << 24;     // mbarrier polls before giving up

static_assert(SMEM_USED + 1024 <= SMEM_ALLOC, "shared memory layout");

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

// 4 int8 codes (xor 0x80 applied) -> two packed fp16 pairs holding the exact
// integers: 0x64xx is 1024 + xx, minus 1152 gives the signed code.
__device__ __forceinline__ void codes_to_h2(uint32_t wx, uint32_t &lo, uint32_t &hi) {
    const uint32_t m = 0x64646464u;
    uint32_t a = prmt(wx, m, 0x4140), b = prmt(wx, m, 0x4342);
    __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
    __half2 ha = __hsub2(*reinterpret_cast<__half2 *>(&a), bias);
    __half2 hb = __hsub2(*reinterpret_cast<__half2 *>(&b), bias);
    lo = *reinterpret_cast<uint32_t *>(&ha);
    hi = *reinterpret_cast<uint32_t *>(&hb);
}

// --- tcgen05 / mbarrier wrappers --------------------------------------------

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait; returns false if the phase did not complete in time.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
    for (long long i = 0; i < WAIT_LIMIT; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset); the leading byte offset is unused in
// this mode; bits 46..48 hold the fixed value 0b001.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024u >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B fp16
// (bits 7-9, 10-12 = 0), both K-major (bits 15, 16 = 0), N >> 3 at bit 17,
// M >> 4 at bit 24.
constexpr uint32_t IDESC = (1u << 4) | ((uint32_t)(TN >> 3) << 17) | ((uint32_t)(TM >> 4) << 24);

__device__ __forceinline__ void mma_f16(uint32_t dtmem, uint64_t adesc, uint64_t bdesc, uint32_t acc) {
    asm volatile(
        "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
        " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(dtmem),
        "l"(adesc), "l"(bdesc), "r"(IDESC), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n"
        : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
          "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
        : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// --- kernels ----------------------------------------------------------------

// qbar = sum over heads, split into fp16 hi/lo rows; rows >= ntok are zero.
template <bool F16>
__global__ void __launch_bounds__(D) qsum_kernel(ScoreLaunch a) {
    const int t = blockIdx.x, d = threadIdx.x;
    float s = 0.0f;
    if (t < a.ntok) {
        if (F16) {
            const __half *q = reinterpret_cast<const __half *>(a.q) + (size_t)t * a.n_q_heads * D + d;
            for (int h = 0; h < a.n_q_heads; ++h) s += __half2float(q[(size_t)h * D]);
        } else {
            const float *q = reinterpret_cast<const float *>(a.q) + (size_t)t * a.n_q_heads * D + d;
            for (int h = 0; h < a.n_q_heads; ++h) s += __ldg(q + (size_t)h * D);
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

__global__ void __launch_bounds__(THREADS, 1) score_kernel(ScoreLaunch a) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    const uint32_t sA0 = base, sB0 = base + 2 * A_BYTES;
    const uint32_t bar0 = sB0 + 2 * B_BYTES;  // two 8-byte mbarriers
    uint8_t *gen = smem_raw + (base - raw);   // generic pointer to `base`
    volatile uint32_t *tslot = reinterpret_cast<volatile uint32_t *>(gen + 2 * A_BYTES + 2 * B_BYTES + 16);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32((const void *)tslot)),
                     "r"(TMEM_COLS));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // Contiguous share of the linear (token tile, cell tile) sequence.
    const int ntt = (a.ntok + TN - 1) / TN;
    long long total = 0;
    for (int tt = 0; tt < ntt; ++tt) total += cell_tiles(a, tt);
    const long long begin = total * blockIdx.x / gridDim.x;
    const long long end = total * (blockIdx.x + 1) / gridDim.x;
    TileWalk cur{0, 0};
    {
        long long k = begin;
        while (cur.tt < ntt && k >= cell_tiles(a, cur.tt)) {
            k -= cell_tiles(a, cur.tt);
            ++cur.tt;
        }
        cur.ct = (int)k;
    }

    // Prefetch registers for the next A tile: 8 x 16 bytes of int8 codes.
    uint4 pre[8];
    auto load_a = [&](const TileWalk &w) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int q = it * THREADS + tid, m = q >> 3, dc = q & 7;
            const int c = w.ct * TM + m;
            pre[it] = c < a.cache_cells ? __ldg(reinterpret_cast<const uint4 *>(a.kq + (size_t)c * D) + dc)
                                        : make_uint4(0x0u, 0x0u, 0x0u, 0x0u);
        }
    };
    auto store_a = [&](uint32_t sA) {
#pragma unroll
        for (int it = 0; it < 8; ++it) {
            const int q = it * THREADS + tid, m = q >> 3, dc = q & 7;
            uint32_t h[8];
            codes_to_h2(pre[it].x ^ 0x80808080u, h[0], h[1]);
            codes_to_h2(pre[it].y ^ 0x80808080u, h[2], h[3]);
            codes_to_h2(pre[it].z ^ 0x80808080u, h[4], h[5]);
            codes_to_h2(pre[it].w ^ 0x80808080u, h[6], h[7]);
            const int kb = dc >> 2, cc = 2 * (dc & 3);
            const uint32_t row = sA + kb * A_KBLOCK + (m >> 3) * 1024 + (m & 7) * 128;
            const uint32_t p0 = row + (((cc) ^ (m & 7)) << 4), p1 = row + (((cc + 1) ^ (m & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p0), "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]));
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p1), "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]));
        }
    };
    auto load_b = [&](int tt) {
        // qbar hi (part 0) and lo (part 1) rows of this token tile.
#pragma unroll 4
        for (int it = 0; it < 16; ++it) {
            const int q = it * THREADS + tid, part = q >> 10, n = (q & 1023) >> 4, ci = q & 15;
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(a.qsum + ((size_t)(tt * TN + n) * 2 + part) * D) + ci);
            const int kb = ci >> 3, cc = ci & 7;
            const uint32_t p = sB0 + part * B_BYTES + kb * B_KBLOCK + (n >> 3) * 1024 + (n & 7) * 128 + ((cc ^ (n & 7)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};" ::"r"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w));
        }
    };

    bool timeout = false;
    auto epilogue = [&](const TileWalk &w, int k) {
        const int b = k & 1;
        if (!mbar_wait(bar0 + 8 * b, (uint32_t)((k >> 1) & 1))) {
            timeout = true;
            return;
        }
        tc_fence_after();
        const int cell = w.ct * TM + warp * 32 + lane;
        float ks[NG] = {0.f, 0.f, 0.f, 0.f};
        if (cell < a.cache_cells) {
            const uint2 kv = __ldg(reinterpret_cast<const uint2 *>(a.ksc + (size_t)cell * NG));
            ks[0] = __half2float(__ushort_as_half((unsigned short)(kv.x & 0xFFFF)));
            ks[1] = __half2float(__ushort_as_half((unsigned short)(kv.x >> 16)));
            ks[2] = __half2float(__ushort_as_half((unsigned short)(kv.y & 0xFFFF)));
            ks[3] = __half2float(__ushort_as_half((unsigned short)(kv.y >> 16)));
        }
        const uint32_t tbase = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(b * NG * TN);
#pragma unroll 1
        for (int j0 = 0; j0 < TN; j0 += 16) {
            const int t0 = w.tt * TN + j0;
            if (t0 >= a.ntok) break;  // warp-uniform
            uint32_t v[NG][16];
#pragma unroll
            for (int g = 0; g < NG; ++g) tmem_ld16(tbase + g * TN + j0, v[g]);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int t = t0 + j;
                if (t < a.ntok && cell <= a.pos0 + t) {
                    float s = ks[0] * __uint_as_float(v[0][j]);
                    s = fmaf(ks[1], __uint_as_float(v[1][j]), s);
                    s = fmaf(ks[2], __uint_as_float(v[2][j]), s);
                    s = fmaf(ks[3], __uint_as_float(v[3][j]), s);
                    a.scores[(size_t)t * a.ld + cell] = s;
                }
            }
        }
        tc_fence_before();
    };

    TileWalk prev{-1, -1};
    int cur_tt = -1;
    bool pending = false;
    const long long n = end - begin;
    if (n > 0) load_a(cur);
    for (long long k = 0; k < n; ++k) {
        if (__syncthreads_or(timeout ? 1 : 0)) {
            timeout = true;
            break;
        }
        const int b = (int)(k & 1);
        if (cur.tt != cur_tt) {
            if (pending) {  // the MMAs still reading the old B must finish first
                epilogue(prev, (int)(k - 1));
                pending = false;
                if (__syncthreads_or(timeout ? 1 : 0)) {
                    timeout = true;
                    break;
                }
            }
            load_b(cur.tt);
            cur_tt = cur.tt;
        }
        store_a(sA0 + b * A_BYTES);
        TileWalk next = cur;
        if (++next.ct >= cell_tiles(a, next.tt)) {
            next.ct = 0;
            ++next.tt;
        }
        if (k + 1 < n) load_a(next);
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        if (tid == 0) {
            tc_fence_after();
            const uint32_t sA = sA0 + b * A_BYTES;
#pragma unroll
            for (int g = 0; g < NG; ++g) {
                const uint32_t dt = tmem + (uint32_t)(b * NG * TN + g * TN);
#pragma unroll
                for (int s = 0; s < 2; ++s) {
                    const int ksx = 2 * g + s, kb = ksx >> 2;
                    const uint32_t koff = (ksx & 3) * 32;
                    const uint64_t ad = sw128_desc(sA + kb * A_KBLOCK + koff);
#pragma unroll
                    for (int part = 0; part < 2; ++part) {
                        const uint64_t bd = sw128_desc(sB0 + part * B_BYTES + kb * B_KBLOCK + koff);
                        mma_f16(dt, ad, bd, (s | part) ? 1u : 0u);
                    }
                }
            }
            mma_commit(bar0 + 8 * b);
        }
        if (pending) epilogue(prev, (int)(k - 1));
        prev = cur;
        pending = true;
        cur = next;
    }
    if (pending && !timeout) epilogue(prev, (int)(n - 1));
    if (timeout && a.err && lane == 0) atomicOr(a.err, QSA_DEVERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS));
    }
}

}  // namespace

cudaError_t launch_score(const ScoreLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    const int ntok_pad = (a.ntok + TN - 1) / TN * TN;
    if (a.q_f16)
        qsum_kernel<true><<<ntok_pad, D, 0, s>>>(a);
    else
        qsum_kernel<false><<<ntok_pad, D, 0, s>>>(a);
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
    score_kernel<<<grid, THREADS, SMEM_ALLOC, s>>>(a);
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
