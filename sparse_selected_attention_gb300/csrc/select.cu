// qsa_select: per-token selection of the cells attention reads (scores -> ids).
//
// The audit pages name this step's buffers ("Round 36 Track C: qsa_prep
// Single-Barrier norm_rope ...", section "Summary & Decision": scores, ids,
// pooled) and its decode window ("round 5 track b: cached residual norms and
// fused mtp attention", section "mtp attention": 64 sink + 256 previous local
// + 1 current cell) but never define the selection rule.  The reading built
// here: the forced cells of that window, plus the highest-scoring other causal
// cells (ties to the lower id), up to min(p + 1, budget) cells, ascending,
// padded with -1.
//
// The forced cells are two runs, the sink [0, fs) and the tail [max(fe, fs), p],
// around the free range [fs, fe), so the output is: the sink ids, the selected
// free ids ascending, the tail ids, then -1.  Only the free range is ranked.
//
// Ranking by (score descending, id ascending) is ranking by one unique 47-bit
// composite key, (order_key(score) << 15) | (32767 - id), so the selected free
// cells are exactly those whose composite is >= the need-th largest, K*.
// NaN scores rank below every number (ties among them to the lower id).  K*
// is found by a most-significant-digit radix select: the 12-bit top digit
// (bit 35), then 11-bit digits (bits 24, 13, 2) and the last two bits.  One
// 256-thread CTA per token row with 42 KB of shared memory, four per SM:
//   1. the free cells are streamed once from HBM as aligned float4 quads.  The
//      block's largest top digit in the first batch of loads places a window
//      of 256 top-digit values (223 below it, 32 above); each cell's top digit,
//      clamped into the window, goes into a 256-bin histogram and, as one
//      byte, into a digit cache in shared memory.  The bin where the count
//      from the top reaches `need` fixes the first digit, unless it is a
//      clamped end bin (the window missed: step 1b);
//   2. from the digit cache alone, each thread builds 32-cell words of the
//      selected bitmap (cells above the crossing bin) and appends the cells
//      in it (candidates, a few hundred for smooth scores) to a list; their
//      scores are then reloaded (from L2) as full keys;
//   3. the remaining digits are resolved on that list, at most 32 survivors
//      are ranked by brute force, and the candidates >= K* join the bitmap;
//   4. a block scan of the bitmap words places the selected free ids.
// 1b. When the window missed or more than CAP cells share the top digit
// (plateaus, outliers), digits are resolved by extra passes over the row, and
// step 2 then compares full composite keys.
//
// Bit positions are cell ids shifted by the row's misalignment `mis` (its
// address modulo 16, in floats), so that quad q holds shifted cells 4q..4q+3,
// bitmap word w holds quads 8w..8w+7, and every float4 load is aligned.  A
// quad that straddles the free range's ends lies inside one 16-byte block
// that also holds a valid cell, and its outside cells are masked.
#include <stdint.h>

#include "check.cuh"
#include "qsa.h"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int THREADS = 256;
constexpr int NWARP = THREADS / 32;
constexpr int WBINS = 256;                           // windowed top-digit bins
constexpr int BELOW = 223;                           // window: [dmax - 223, dmax + 32]
constexpr int CAP = 2048;                            // candidate list capacity
constexpr int NFIN = 32;                             // survivors ranked by brute force
constexpr int MAXQ = (kSelectMaxCells + 3 + 3) / 4;  // quads covering n + mis shifted cells
constexpr int NWORD = (MAXQ + 7) / 8;                // bitmap words (8 quads each)
constexpr int WPT = 4;                               // output scan: words per thread (the last thread 5)
constexpr int SWEEP = 5;                             // sweep: words per thread at stride THREADS
constexpr int UNROLL = 8;
constexpr int NLEVEL = 5;
constexpr int RELOAD = CAP / THREADS;                // candidate reloads per thread
static_assert(kSelectMaxCells <= 32768, "ids fit in 15 bits of the composite key");
static_assert(NWORD <= WPT * THREADS + 1, "the output scan gives four words per thread, five to the last");
static_assert(NWORD <= SWEEP * THREADS, "the sweep gives at most five words to a thread");

__device__ __forceinline__ int level_shift(int level) {
    return level == 0 ? 35 : level == 1 ? 24 : level == 2 ? 13 : level == 3 ? 2 : 0;
}
__device__ __forceinline__ int level_bins(int level) { return level == 0 ? 4096 : level == 4 ? 4 : 2048; }

struct Smem {
    // The digit cache while the row streams in; afterwards the histogram
    // (first 16 KB) and the candidate keys (next 16 KB).
    alignas(16) uint32_t dig[8 * NWORD];  // quad q's four windowed top digits, one byte each
    uint16_t cidx[CAP];                   // candidate cells
    int whist[WBINS];
    unsigned long long fin[NFIN];
    unsigned long long kstar;
    unsigned bits[NWORD + 7];
    int wtot[NWARP];
    int cross[3];  // bin, count still needed inside it, cells in it
    int ncand, nfin;
};
static_assert(sizeof(int) * 4096 + sizeof(unsigned long long) * CAP <= sizeof(uint32_t) * 8 * NWORD,
              "the histogram and the candidate keys fit in the digit cache");
constexpr size_t SMEM_BYTES = sizeof(Smem);

__device__ __forceinline__ int *hist_of(Smem &sm) { return reinterpret_cast<int *>(sm.dig); }
__device__ __forceinline__ unsigned long long *cand_of(Smem &sm) {
    return reinterpret_cast<unsigned long long *>(sm.dig + 4096);
}

// Order-preserving key: -0 and +0 are one value (adding +0 turns -0 into +0),
// and every NaN takes key 0, below -inf, so NaN scores rank last.
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = __float_as_uint(f + 0.0f);
    const uint32_t k = b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u);
    return f != f ? 0u : k;
}

__device__ __forceinline__ uint32_t top_digit(float f) { return order_key(f) >> 20; }

// The float whose order key is k (k is not a NaN's key).
__device__ __forceinline__ float key_float(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// The window bin of f: f (a NaN taken as lo) is clamped into [lo, hi], the
// numbers whose top digits are base .. base + 255, so its top digit less base
// is the bin.
__device__ __forceinline__ uint32_t window_bin(float f, float lo, float hi, int base) {
    const uint32_t b = __float_as_uint(fminf(fmaxf(f + 0.0f, lo), hi));
    return ((b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u)) >> 20) - (uint32_t)base;
}

__device__ __forceinline__ unsigned long long composite(float x, int c) {
    return ((unsigned long long)order_key(x) << 15) | (unsigned)(32767 - c);
}

__device__ __forceinline__ int warp_incl_scan(int v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    return v;
}

// Bit 7 of byte e of the result is set iff byte e of x is >= t, where T
// holds t (<= 255) in every byte: the low seven bits compare through one
// subtraction that cannot borrow across bytes ((x | 0x80) - (t & 0x7f) >= 1),
// and the top bits settle the rest.
__device__ __forceinline__ uint32_t bytes_ge(uint32_t x, uint32_t T) {
    const uint32_t d = (x | 0x80808080u) - (T & 0x7f7f7f7fu);
    return ((x & ~T) | (~(x ^ T) & d)) & 0x80808080u;
}

// Bit 7 of byte e of the result is set iff byte e of x equals w, where W
// holds w in every byte (an exact zero-byte test of x ^ W).
__device__ __forceinline__ uint32_t bytes_eq(uint32_t x, uint32_t W) {
    const uint32_t y = x ^ W;
    return ~(((y & 0x7f7f7f7fu) + 0x7f7f7f7fu) | y) & 0x80808080u;
}

// Bit 7 of each byte, as bits 0..3.
__device__ __forceinline__ uint32_t byte_flags(uint32_t f) { return ((f >> 7) * 0x01020408u) >> 24; }

// Bits of bitmap word w that fall in the shifted-cell range [lo, hi).
__device__ __forceinline__ unsigned range_bits(int w, int lo, int hi) {
    const int a = min(max(lo - 32 * w, 0), 32), b = min(max(hi - 32 * w, 0), 32);
    if (b <= a) return 0u;
    const unsigned upto_b = b == 32 ? 0xffffffffu : ((1u << b) - 1u);
    const unsigned below_a = a == 32 ? 0xffffffffu : ((1u << a) - 1u);
    return upto_b & ~below_a;
}

// Ranks of the set bits of bitmap words [wlo, whi) in cell order.  Thread tid
// owns words wlo + 4 tid .. wlo + 4 tid + 3 (the last thread a fifth one);
// returns the rank of its first set bit and the total over the block.
__device__ __forceinline__ int scan_words(Smem &sm, const unsigned *bm, int wlo, int whi, unsigned (&wv)[WPT + 1],
                                          int &total) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wb = wlo + WPT * tid, we = min(tid == THREADS - 1 ? wb + WPT + 1 : wb + WPT, whi);
    int mine = 0;
#pragma unroll
    for (int i = 0; i < WPT + 1; ++i) {
        wv[i] = wb + i < we ? bm[wb + i] : 0u;
        mine += __popc(wv[i]);
    }
    int incl = warp_incl_scan(mine, lane);
    if (lane == 31) sm.wtot[warp] = incl;
    __syncthreads();
    total = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
        const int v = sm.wtot[w];
        incl += w < warp ? v : 0;
        total += v;
    }
    return incl - mine;
}

__device__ __forceinline__ void clear_hist(int *h, int nb) {
    int4 *h4 = reinterpret_cast<int4 *>(h);
    for (int i = threadIdx.x; i < nb / 4; i += THREADS) h4[i] = make_int4(0, 0, 0, 0);
}

// Scans the nb-bin histogram h from the top bin down and publishes (bin, need
// left inside it, its count) for the bin where the running count reaches
// `need`.  Thread tid owns the nb / THREADS bins (one, for nb < THREADS)
// below bin nb - per * tid.
__device__ __forceinline__ void find_crossing(Smem &sm, const int *h, int nb, int need) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int per = nb >= THREADS ? nb / THREADS : 1;
    const int top = nb - per * tid;
    int s = 0;
    if (top > 0)
        for (int i = 1; i <= per; ++i) s += h[top - i];
    int incl = warp_incl_scan(s, lane);
    if (lane == 31) sm.wtot[warp] = incl;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NWARP; ++w) incl += w < warp ? sm.wtot[w] : 0;
    const int excl = incl - s;
    if (top > 0 && excl < need && incl >= need) {
        int run = excl;
        for (int i = 1; i <= per; ++i) {
            const int c = h[top - i];
            if (run + c >= need) {
                sm.cross[0] = top - i;
                sm.cross[1] = need - run;
                sm.cross[2] = c;
                break;
            }
            run += c;
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(THREADS, 4) select_kernel(SelectLaunch a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    wait_for_previous_grid();  // launched as a programmatic dependent: the scores may come from qsa_score
    allow_dependent_launch();
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int t = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int32_t *out = a.ids + (size_t)t * a.width;
    [[maybe_unused]] const size_t ids_n = (size_t)a.ntok * a.width, row0 = (size_t)t * a.width;
    const int p = a.pos0 + t, n = p + 1;

    if (n <= a.budget) {  // every causal cell is selected
        for (int c = tid; c < a.width; c += THREADS)
            if (QSA_IN(row0 + c, ids_n)) out[c] = c < n ? c : -1;
        return;
    }
    // Sink [0, fs), free [fs, fe), tail [tail_lo, p].
    const int fs = min(a.sink, n);
    const int fe = min(max(a.sink, p - a.local), p);
    const int tail_lo = max(fe, fs);
    const int nfree = max(fe - fs, 0);
    const int need = min(n, a.budget) - (n - nfree);  // free cells to take; <= 0: forced only
    const int nsel = max(need, 0);
    const int total = fs + nsel + (n - tail_lo);

    // Forced runs and padding go straight out.
    for (int i = tid; i < fs; i += THREADS)
        if (QSA_IN(row0 + i, ids_n)) out[i] = i;
    for (int i = tid; i < n - tail_lo; i += THREADS)
        if (QSA_IN(row0 + fs + nsel + i, ids_n)) out[fs + nsel + i] = tail_lo + i;
    for (int i = total + tid; i < a.width; i += THREADS)
        if (QSA_IN(row0 + i, ids_n)) out[i] = -1;
    if (need <= 0) return;

    const float *row = a.scores + (size_t)t * a.ld;
    const int mis = (int)((reinterpret_cast<uintptr_t>(row) >> 2) & 3u);
    const float4 *rowq = reinterpret_cast<const float4 *>(row - mis);
    const int sfs = fs + mis, sfe = fe + mis;  // shifted free range
    const int q0 = sfs >> 2, q1 = (sfe + 3) >> 2;
    const int w0 = sfs >> 5, w1 = (sfe + 31) >> 5;  // bitmap words of the free range
    [[maybe_unused]] const long long cells_n = (long long)a.ntok * a.ld, row_at = (long long)t * a.ld - mis;

    for (int w = w0 + tid; w < w1; w += THREADS) sm.bits[w] = 0u;
    for (int i = tid; i < WBINS; i += THREADS) sm.whist[i] = 0;
    if (tid == 0) {
        sm.ncand = 0;
        sm.nfin = 0;
        sm.cross[0] = 0;
        sm.cross[1] = 1;
        sm.cross[2] = 1;
        sm.kstar = ~0ull;
    }

    // 1. Windowed top-digit histogram and digit cache, one pass over the free
    //    quads.  The first batch's largest top digit places the window (the
    //    barrier there also publishes the clears above).
    int base = 0;
    for (int qb = q0; qb < q1; qb += THREADS * UNROLL) {
        float4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int q = qb + u * THREADS + tid;
            v[u] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (q < q1 && QSA_IN(row_at + max(4 * q, sfs), cells_n) && QSA_IN(row_at + min(4 * q + 3, sfe - 1), cells_n))
                v[u] = __ldg(rowq + q);
        }
        if (qb == q0) {
            uint32_t dm = 0u;
#pragma unroll
            for (int u = 0; u < UNROLL; ++u) {
                const int s0 = 4 * (qb + u * THREADS + tid);
                const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (s0 + e >= sfs && s0 + e < sfe) dm = max(dm, top_digit(x[e]));
            }
            dm = __reduce_max_sync(0xffffffffu, dm);
            if (lane == 0) sm.wtot[warp] = (int)dm;
            __syncthreads();
            int m = 0;
#pragma unroll
            for (int w = 0; w < NWARP; ++w) m = max(m, sm.wtot[w]);
            base = min(max(m - BELOW, 0), 4096 - WBINS);
        }
        // lo is at least -FLT_MAX and hi at most +inf (keys below 0x00800000
        // are -inf and negative NaNs, above 0xff800000 positive NaNs), so
        // both are numbers and every bin lies in [0, 255]; a window that
        // starts below -FLT_MAX counts as missed.
        // hi is never -0 either (key 0x7fffffff): whichever zero fminf
        // returned for (+0, -0), +0 would fall one bin past the window, so
        // the smallest negative subnormal, the same top digit, stands in.
        const float lo = key_float(max((uint32_t)base << 20, 0x00800000u));
        const uint32_t hik = min(((uint32_t)(base + WBINS) << 20) - 1u, 0xff800000u);
        const float hi = key_float(hik == 0x7fffffffu ? 0x7ffffffeu : hik);
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int q = qb + u * THREADS + tid;
            if (q < q1) {
                const uint32_t d0 = window_bin(v[u].x, lo, hi, base), d1 = window_bin(v[u].y, lo, hi, base);
                const uint32_t d2 = window_bin(v[u].z, lo, hi, base), d3 = window_bin(v[u].w, lo, hi, base);
                const int s0 = 4 * q;
                if (s0 >= sfs && s0 + 4 <= sfe) {
                    atomicAdd(&sm.whist[d0], 1);
                    atomicAdd(&sm.whist[d1], 1);
                    atomicAdd(&sm.whist[d2], 1);
                    atomicAdd(&sm.whist[d3], 1);
                } else {
                    if (s0 >= sfs && s0 < sfe) atomicAdd(&sm.whist[d0], 1);
                    if (s0 + 1 >= sfs && s0 + 1 < sfe) atomicAdd(&sm.whist[d1], 1);
                    if (s0 + 2 >= sfs && s0 + 2 < sfe) atomicAdd(&sm.whist[d2], 1);
                    if (s0 + 3 >= sfs && s0 + 3 < sfe) atomicAdd(&sm.whist[d3], 1);
                }
                sm.dig[q] = d0 | (d1 << 8) | (d2 << 16) | (d3 << 24);
            }
        }
    }
    __syncthreads();
    find_crossing(sm, sm.whist, WBINS, need);
    const int wbin = sm.cross[0];
    // A clamped end bin holds several top digits: the window missed.
    const bool miss = (wbin == WBINS - 1 && base + WBINS < 4096) || (wbin == 0 && base > 0) || base < 8;
    unsigned long long prefix = 0ull, mask = 0ull;
    int rem = need, cnt = 0x7fffffff, level = 0;
    if (!miss) {
        prefix = (unsigned long long)(base + wbin) << 35;
        mask = 0xfffull << 35;
        rem = sm.cross[1];
        cnt = sm.cross[2];
        level = 1;
    }

    // 1b. More digits over the row while the prefix group overflows the list
    //     (from the top digit when the window missed).
    int *hist = hist_of(sm);
    unsigned long long *cand = cand_of(sm);
    while (cnt > CAP && level < NLEVEL) {
        const int sh = level_shift(level), nb = level_bins(level);
        clear_hist(hist, nb);
        __syncthreads();
        for (int c = fs + tid; c < fe; c += THREADS) {
            if (!QSA_IN(c, a.ld)) continue;
            const unsigned long long k = composite(__ldg(row + c), c);
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> sh) & (unsigned)(nb - 1)], 1);
        }
        __syncthreads();
        find_crossing(sm, hist, nb, rem);
        prefix |= (unsigned long long)sm.cross[0] << sh;
        mask |= (unsigned long long)(nb - 1) << sh;
        rem = sm.cross[1];
        cnt = sm.cross[2];
        ++level;
    }

    // 2. Free cells above the prefix set their bits; cells equal to it are
    //    candidates (with one such cell left, it is K* and simply selected).
    const bool collect = cnt > 1;
    const bool fast = !miss && level == 1;  // only the top digit is fixed: work from the digit cache
    bool have_hist = false;                 // the histogram for `level` over the list is built
    if (fast) {
        // Selected: window bin >= thr; candidates: window bin == wbin.  Words
        // are dealt at stride THREADS; lanes 4..7 of each quarter warp read a
        // word's halves in the other order, so a warp's 16-byte loads fall in
        // distinct banks.
        const uint32_t thr = (uint32_t)wbin + (collect ? 1u : 0u);  // <= 256; 256 selects none
        const uint32_t T = (thr & 255u) * 0x01010101u, W = (uint32_t)wbin * 0x01010101u;
        const bool none = thr > 255u;
        const int swap = (lane >> 2) & 1;
#pragma unroll
        for (int i = 0; i < SWEEP; ++i) {
            const int w = w0 + tid + THREADS * i;
            uint32_t sel = 0u, eq = 0u;
            if (w < w1) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    const int h = hh ^ swap;
                    const uint4 v = reinterpret_cast<const uint4 *>(sm.dig + 8 * w)[h];
                    if (!none) {
                        const uint32_t g = byte_flags(bytes_ge(v.x, T)) | (byte_flags(bytes_ge(v.y, T)) << 4) |
                                           (byte_flags(bytes_ge(v.z, T)) << 8) | (byte_flags(bytes_ge(v.w, T)) << 12);
                        sel |= g << (16 * h);
                    }
                    if (collect) {  // the crossing bin: disjoint from the selected bins above it
                        const uint32_t e = byte_flags(bytes_eq(v.x, W)) | (byte_flags(bytes_eq(v.y, W)) << 4) |
                                           (byte_flags(bytes_eq(v.z, W)) << 8) | (byte_flags(bytes_eq(v.w, W)) << 12);
                        eq |= e << (16 * h);
                    }
                }
                const unsigned vm = range_bits(w, sfs, sfe);
                sel &= vm;
                eq &= vm;
                sm.bits[w] = sel;
            }
            if (collect) {
                // Append the word's candidates: one shared atomic per warp.
                const int nc = __popc(eq);
                const int incl = warp_incl_scan(nc, lane);
                int slot = 0;
                if (lane == 31 && incl > 0) slot = atomicAdd(&sm.ncand, incl);
                slot = __shfl_sync(0xffffffffu, slot, 31) + incl - nc;
                for (uint32_t m = eq; m; m &= m - 1u, ++slot)
                    if (slot < CAP) sm.cidx[slot] = (uint16_t)(32 * w + __ffs(m) - 1 - mis);
            }
        }
        __syncthreads();  // the digit cache is dead: the histogram and the keys take its place
        if (collect) {
            const int nc = min(sm.ncand, CAP);
            have_hist = cnt > NFIN;
            if (have_hist) {
                clear_hist(hist, level_bins(1));
                __syncthreads();
            }
            // Every reload of the thread in flight at once (serial reloads
            // would each pay a loaded L2 round trip).
            float x[RELOAD];
#pragma unroll
            for (int j = 0; j < RELOAD; ++j) {
                const int i = tid + THREADS * j;
                const int c = i < nc ? (int)sm.cidx[i] : 0;
                x[j] = (i < nc && QSA_IN(c, a.ld)) ? __ldg(row + c) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < RELOAD; ++j) {
                const int i = tid + THREADS * j;
                if (i < nc) {
                    const unsigned long long k = composite(x[j], sm.cidx[i]);
                    cand[i] = k;
                    if (have_hist) atomicAdd(&hist[(k >> 24) & 2047u], 1);
                }
            }
            if (tid == 0) sm.ncand = nc;
        }
    } else {
        for (int c = fs + tid; c < fe; c += THREADS) {
            if (!QSA_IN(c, a.ld)) continue;
            const unsigned long long k = composite(__ldg(row + c), c);
            const unsigned long long km = k & mask;
            const int s = c + mis;
            if (collect ? km > prefix : km >= prefix) atomicOr(&sm.bits[s >> 5], 1u << (s & 31));
            if (collect && km == prefix) {
                const int slot = atomicAdd(&sm.ncand, 1);
                if (slot < CAP) cand[slot] = k;
            }
        }
    }
    __syncthreads();

    // 3. Remaining digits on the candidate list; brute force at <= NFIN.
    if (collect) {
        const int ncand = min(sm.ncand, CAP);
        while (cnt > NFIN && level < NLEVEL) {
            const int sh = level_shift(level), nb = level_bins(level);
            if (!have_hist) {
                clear_hist(hist, nb);
                __syncthreads();
                for (int i = tid; i < ncand; i += THREADS) {
                    const unsigned long long k = cand[i];
                    if ((k & mask) == prefix) atomicAdd(&hist[(k >> sh) & (unsigned)(nb - 1)], 1);
                }
                __syncthreads();
            }
            have_hist = false;
            find_crossing(sm, hist, nb, rem);
            prefix |= (unsigned long long)sm.cross[0] << sh;
            mask |= (unsigned long long)(nb - 1) << sh;
            rem = sm.cross[1];
            cnt = sm.cross[2];
            ++level;
        }
        for (int i = tid; i < ncand; i += THREADS) {
            const unsigned long long k = cand[i];
            if ((k & mask) == prefix) {
                const int slot = atomicAdd(&sm.nfin, 1);
                if (slot < NFIN) sm.fin[slot] = k;
            }
        }
        __syncthreads();
        const int nf = min(sm.nfin, NFIN);
        if (tid < nf) {
            const unsigned long long k = sm.fin[tid];
            int rank = 0;
            for (int m = 0; m < nf; ++m) rank += sm.fin[m] > k;
            if (rank == rem - 1) sm.kstar = k;
        }
        __syncthreads();
        const unsigned long long kstar = sm.kstar;
        for (int i = tid; i < ncand; i += THREADS) {
            const unsigned long long k = cand[i];
            if (k >= kstar) {
                const int s = 32767 - (int)(k & 32767u) + mis;
                atomicOr(&sm.bits[s >> 5], 1u << (s & 31));
            }
        }
        __syncthreads();
    }

    // 4. Selected free ids, ascending, after the sink.
    unsigned wv[WPT + 1];
    int nbits;
    int pos = scan_words(sm, sm.bits, w0, w1, wv, nbits);
    const int wb = w0 + WPT * tid;
#pragma unroll
    for (int i = 0; i < WPT + 1; ++i)
        for (unsigned m = wv[i]; m && pos < nsel; m &= m - 1u, ++pos)
            if (QSA_IN(row0 + fs + pos, ids_n)) out[fs + pos] = 32 * (wb + i) + __ffs(m) - 1 - mis;
}

}  // namespace

cudaError_t launch_select(const SelectLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return launch_dependent(select_kernel, dim3(a.ntok), dim3(THREADS), SMEM_BYTES, s, a);
}

}  // namespace qsa

QSA_DEFINE_CHECK_READER(take_check_word_select)
