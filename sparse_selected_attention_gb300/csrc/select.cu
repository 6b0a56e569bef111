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
// cells are exactly those whose composite is >= the need-th largest, K*.  K*
// is found by a most-significant-digit radix select with 12-bit digits
// (shifts 35, 23, 11, 0).  One 512-thread CTA per token row, two per SM:
//   1. the free cells are streamed once from HBM as aligned float4 quads; each
//      cell's top digit goes into a 4096-bin histogram and into a 16-bit digit
//      cache in shared memory; the bin where the count from the top reaches
//      `need` fixes the first digit;
//   2. from the digit cache alone, each thread builds its two 32-cell words
//      of two bitmaps: free cells whose top digit beats the crossing bin
//      (selected) and free cells in it (candidates, a few hundred for smooth
//      scores); a block scan of the candidate counts ranks them in cell order
//      and their scores are reloaded (from L2) into the list, one per thread;
//   3. the remaining digits are resolved on that list, at most 32 survivors
//      are ranked by brute force, and each owner adds its candidates >= K*
//      to its selected words;
//   4. a block scan of the selected words places the selected free ids.
// When more than CAP cells share the top digit (plateaus, outliers), further
// digits are first resolved by extra passes over the row, and step 2 then
// compares full composite keys.
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

constexpr int THREADS = 512;
constexpr int NWARP = THREADS / 32;
constexpr int NBIN = 4096;            // 12-bit digits
constexpr int BPT = NBIN / THREADS;   // bins per thread in the threshold scan
constexpr int CAP = 2048;             // candidate list capacity
constexpr int NFIN = 32;              // survivors ranked by brute force
constexpr int MAXQ = (kSelectMaxCells + 3 + 3) / 4;  // quads covering n + mis shifted cells
constexpr int NWORD = (MAXQ + 7) / 8;                // bitmap words (8 quads each)
constexpr int UNROLL = 8;
constexpr int NLEVEL = 4;
static_assert(kSelectMaxCells <= 32768, "ids fit in 15 bits of the composite key");
static_assert(NWORD <= 2 * THREADS + 1, "the output scan gives two words per thread, three to the last");
static_assert(BPT == 8 && NBIN % 4 == 0, "two int4 loads per thread in the threshold scan");

__device__ __forceinline__ int level_shift(int level) {
    return level == 0 ? 35 : level == 1 ? 23 : level == 2 ? 11 : 0;
}

struct Smem {
    int hist[NBIN];
    unsigned long long cand[CAP];
    unsigned long long fin[NFIN];
    unsigned long long kstar;
    unsigned bits[NWORD + 7];
    int wtot[NWARP];
    int cross[3];  // digit, count still needed inside it, cells in it
    int ncand, nfin;
    alignas(16) uint2 dig[8 * NWORD];  // top digits of quad q's four cells, 16 bits each
};
constexpr size_t SMEM_BYTES = sizeof(Smem);

// Order-preserving key; -0 and +0 are one value (they tie, lower id first).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = f == 0.0f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

// order_key(f) >> 20 in integer operations.
__device__ __forceinline__ uint32_t top_digit(float f) {
    uint32_t b = __float_as_uint(f);
    b = b == 0x80000000u ? 0u : b;
    return (b ^ ((uint32_t)((int32_t)b >> 31) | 0x80000000u)) >> 20;
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

// Bit e of the result is set iff the e-th of the four 12-bit digits packed in
// (x, y) is >= thr, where c = 0x80008000 - (thr | thr << 16): each 16-bit lane
// plus (0x8000 - thr) has bit 15 set exactly then, with no carry or borrow
// between lanes.
__device__ __forceinline__ uint32_t digits_ge(uint32_t x, uint32_t y, uint32_t c) {
    const uint32_t gx = x + c, gy = y + c;
    return ((gx >> 15) & 1u) | ((gx >> 30) & 2u) | ((gy >> 13) & 4u) | ((gy >> 28) & 8u);
}

// Bits of bitmap word w that fall in the shifted-cell range [lo, hi).
__device__ __forceinline__ unsigned range_bits(int w, int lo, int hi) {
    const int a = min(max(lo - 32 * w, 0), 32), b = min(max(hi - 32 * w, 0), 32);
    if (b <= a) return 0u;
    const unsigned upto_b = b == 32 ? 0xffffffffu : ((1u << b) - 1u);
    const unsigned below_a = a == 32 ? 0xffffffffu : ((1u << a) - 1u);
    return upto_b & ~below_a;
}

// Ranks of the set bits of bitmap words [wlo, whi) in cell order.  Thread tid
// owns words wlo + 2 tid and wlo + 2 tid + 1 (the last thread a third one);
// returns the rank of its first set bit and the total over the block.
__device__ __forceinline__ int scan_words(Smem &sm, const unsigned *bm, int wlo, int whi, unsigned (&wv)[3],
                                          int &total) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wb = wlo + 2 * tid, we = min(tid == THREADS - 1 ? wb + 3 : wb + 2, whi);
    int mine = 0;
#pragma unroll
    for (int i = 0; i < 3; ++i) {
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

__device__ __forceinline__ void clear_hist(Smem &sm) {
    int4 *h = reinterpret_cast<int4 *>(sm.hist);
    for (int i = threadIdx.x; i < NBIN / 4; i += THREADS) h[i] = make_int4(0, 0, 0, 0);
}

// Scans hist from the top bin down and publishes (digit, need left inside it,
// its count) for the digit where the running count reaches `need`.  Thread
// tid owns bins NBIN-8(tid+1) .. NBIN-1-8tid, read as two int4.
__device__ __forceinline__ void find_crossing(Smem &sm, int need) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int4 *h = reinterpret_cast<const int4 *>(sm.hist + NBIN - BPT * (tid + 1));
    const int4 lo = h[0], hi = h[1];
    const int cnt[BPT] = {hi.w, hi.z, hi.y, hi.x, lo.w, lo.z, lo.y, lo.x};  // descending bins
    int s = 0;
#pragma unroll
    for (int i = 0; i < BPT; ++i) s += cnt[i];
    int incl = warp_incl_scan(s, lane);
    if (lane == 31) sm.wtot[warp] = incl;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < NWARP; ++w) incl += w < warp ? sm.wtot[w] : 0;
    const int excl = incl - s;
    if (excl < need && incl >= need) {
        int run = excl;
#pragma unroll
        for (int i = 0; i < BPT; ++i) {
            if (run + cnt[i] >= need) {
                sm.cross[0] = NBIN - 1 - BPT * tid - i;
                sm.cross[1] = need - run;
                sm.cross[2] = cnt[i];
                break;
            }
            run += cnt[i];
        }
    }
    __syncthreads();
}

__global__ void __launch_bounds__(THREADS, 2) select_kernel(SelectLaunch a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    wait_for_previous_grid();  // launched as a programmatic dependent: the scores may come from qsa_score
    allow_dependent_launch();
    Smem &sm = *reinterpret_cast<Smem *>(smem_raw);
    const int t = blockIdx.x, tid = threadIdx.x;
    const int warp = tid >> 5, lane = tid & 31;
    int32_t *out = a.ids + (size_t)t * a.width;
    const int p = a.pos0 + t, n = p + 1;

    if (n <= a.budget) {  // every causal cell is selected
        for (int c = tid; c < a.width; c += THREADS)
            if (QSA_IN((size_t)t * a.width + c, (size_t)a.ntok * a.width)) out[c] = c < n ? c : -1;
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
    for (int i = tid; i < fs; i += THREADS) out[i] = i;
    for (int i = tid; i < n - tail_lo; i += THREADS) out[fs + nsel + i] = tail_lo + i;
    for (int i = total + tid; i < a.width; i += THREADS) out[i] = -1;
    if (need <= 0) return;

    const float *row = a.scores + (size_t)t * a.ld;
    const int mis = (int)((reinterpret_cast<uintptr_t>(row) >> 2) & 3u);
    const float4 *rowq = reinterpret_cast<const float4 *>(row - mis);
    const int sfs = fs + mis, sfe = fe + mis;  // shifted free range
    const int q0 = sfs >> 2, q1 = (sfe + 3) >> 2;
    const int w0 = sfs >> 5, w1 = (sfe + 31) >> 5;  // bitmap words of the free range

    for (int w = w0 + tid; w < w1; w += THREADS) sm.bits[w] = 0u;
    clear_hist(sm);
    if (tid == 0) {
        sm.ncand = 0;
        sm.nfin = 0;
        sm.cross[0] = 0;
        sm.cross[1] = 1;
        sm.cross[2] = 1;
        sm.kstar = ~0ull;
    }
    __syncthreads();

    // 1. Top-digit histogram and digit cache, one pass over the free quads.
    for (int qb = q0 + tid; qb < q1; qb += THREADS * UNROLL) {
        float4 v[UNROLL];
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int q = qb + u * THREADS;
            if (q < q1 && QSA_IN((long long)t * a.ld - mis + 4 * q, (long long)a.ntok * a.ld) &&
                QSA_IN((long long)t * a.ld - mis + 4 * q + 3, (long long)a.ntok * a.ld))
                v[u] = __ldg(rowq + q);
        }
#pragma unroll
        for (int u = 0; u < UNROLL; ++u) {
            const int q = qb + u * THREADS;
            if (q < q1) {
                const uint32_t d0 = top_digit(v[u].x), d1 = top_digit(v[u].y);
                const uint32_t d2 = top_digit(v[u].z), d3 = top_digit(v[u].w);
                const int s0 = 4 * q;
                if (s0 >= sfs && s0 + 4 <= sfe) {
                    atomicAdd(&sm.hist[d0], 1);
                    atomicAdd(&sm.hist[d1], 1);
                    atomicAdd(&sm.hist[d2], 1);
                    atomicAdd(&sm.hist[d3], 1);
                } else {
                    if (s0 >= sfs && s0 < sfe) atomicAdd(&sm.hist[d0], 1);
                    if (s0 + 1 >= sfs && s0 + 1 < sfe) atomicAdd(&sm.hist[d1], 1);
                    if (s0 + 2 >= sfs && s0 + 2 < sfe) atomicAdd(&sm.hist[d2], 1);
                    if (s0 + 3 >= sfs && s0 + 3 < sfe) atomicAdd(&sm.hist[d3], 1);
                }
                sm.dig[q] = make_uint2(d0 | (d1 << 16), d2 | (d3 << 16));
            }
        }
    }
    __syncthreads();
    find_crossing(sm, need);
    unsigned long long prefix = (unsigned long long)sm.cross[0] << 35;
    unsigned long long mask = (unsigned long long)(NBIN - 1) << 35;
    int rem = sm.cross[1], cnt = sm.cross[2], level = 1;

    // More digits over the row while the prefix group overflows the list.
    while (cnt > CAP && level < NLEVEL) {
        const int sh = level_shift(level);
        clear_hist(sm);
        __syncthreads();
        for (int c = fs + tid; c < fe; c += THREADS) {
            if (!QSA_IN(c, a.ld)) continue;
            const unsigned long long k = composite(__ldg(row + c), c);
            if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> sh) & (NBIN - 1)], 1);
        }
        __syncthreads();
        find_crossing(sm, rem);
        prefix |= (unsigned long long)sm.cross[0] << sh;
        mask |= (unsigned long long)(NBIN - 1) << sh;
        rem = sm.cross[1];
        cnt = sm.cross[2];
        ++level;
    }

    // 2. Free cells above the prefix set their bits; cells equal to it are
    //    candidates (with one such cell left, it is K* and simply selected).
    const bool collect = cnt > 1;
    const bool fast = level == 1;  // only the top digit is fixed: work from the digit cache
    bool have_hist = false;        // the histogram for `level` over the list is built
    // Thread tid owns bitmap words wb .. wb + nown - 1 (two, the last thread
    // three) of the free range.
    const int wb = w0 + 2 * tid;
    const int nown = max(0, min(tid == THREADS - 1 ? 3 : 2, w1 - wb));
    uint32_t selw[3] = {0u, 0u, 0u}, eqw[3] = {0u, 0u, 0u};
    int epos = 0;  // rank of the thread's first candidate in the list
    if (fast) {
        const uint32_t bs = sm.cross[0];
        const uint32_t thr = bs + (collect ? 1u : 0u);  // selected: top digit >= thr
        const uint32_t c_sel = 0x80008000u - (thr | (thr << 16));
        const uint32_t c_ge = 0x80008000u - (bs | (bs << 16));
        clear_hist(sm);  // free since find_crossing; refilled by the reload below
        // A word's 8 quads are 64 contiguous bytes of the cache; the two words
        // are read as eight 16-byte pieces in a lane-rotated order so that a
        // warp's loads spread over all banks.
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int r = (j + lane) & 7, wi = r >> 2, k = r & 3;
            if (wi < nown) {
                const uint4 v = reinterpret_cast<const uint4 *>(sm.dig + 8 * (wb + wi))[k];
                const uint32_t g0 = digits_ge(v.x, v.y, c_sel), g1 = digits_ge(v.z, v.w, c_sel);
                const uint32_t sb = (g0 | (g1 << 4)) << (8 * k);
                uint32_t eb = 0u;
                if (collect) {
                    const uint32_t e0 = digits_ge(v.x, v.y, c_ge) & ~g0, e1 = digits_ge(v.z, v.w, c_ge) & ~g1;
                    eb = (e0 | (e1 << 4)) << (8 * k);
                }
                if (wi == 0) {
                    selw[0] |= sb;
                    eqw[0] |= eb;
                } else {
                    selw[1] |= sb;
                    eqw[1] |= eb;
                }
            }
        }
        if (nown == 3) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint4 v = reinterpret_cast<const uint4 *>(sm.dig + 8 * (wb + 2))[k];
                const uint32_t g0 = digits_ge(v.x, v.y, c_sel), g1 = digits_ge(v.z, v.w, c_sel);
                selw[2] |= (g0 | (g1 << 4)) << (8 * k);
                if (collect) {
                    const uint32_t e0 = digits_ge(v.x, v.y, c_ge) & ~g0, e1 = digits_ge(v.z, v.w, c_ge) & ~g1;
                    eqw[2] |= (e0 | (e1 << 4)) << (8 * k);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < 3; ++i) {
            const uint32_t vm = i < nown ? range_bits(wb + i, sfs, sfe) : 0u;
            selw[i] &= vm;
            eqw[i] &= vm;
        }
        if (collect) {
            // Candidate ranks in cell order: a block scan of the owners' counts.
            const int mine = __popc(eqw[0]) + __popc(eqw[1]) + __popc(eqw[2]);
            int incl = warp_incl_scan(mine, lane);
            if (lane == 31) sm.wtot[warp] = incl;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < NWARP; ++w) incl += w < warp ? sm.wtot[w] : 0;
            epos = incl - mine;
            // Candidate ids at their ranks, into the dead digit cache; then
            // their full keys with one load per thread, all in flight at once
            // (serial reloads by owners would each pay a loaded L2 round
            // trip), building the next digit's histogram on the way.
            int *cidx = reinterpret_cast<int *>(sm.dig);
            int pos = epos;
#pragma unroll
            for (int i = 0; i < 3; ++i)
                for (uint32_t m = eqw[i]; m; m &= m - 1u, ++pos)
                    if (pos < CAP) cidx[pos] = 32 * (wb + i) + __ffs(m) - 1 - mis;
            __syncthreads();
            const int nc = min(cnt, CAP);
            if (tid == 0) sm.ncand = nc;
            have_hist = cnt > NFIN;
            for (int i = tid; i < nc; i += THREADS) {
                const int c = cidx[i];
                const unsigned long long k = QSA_IN(c, a.ld) ? composite(__ldg(row + c), c) : 0ull;
                sm.cand[i] = k;
                if (have_hist) atomicAdd(&sm.hist[(k >> 23) & (NBIN - 1)], 1);
            }
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
                if (slot < CAP) sm.cand[slot] = k;
            }
        }
    }
    __syncthreads();

    // 3. Remaining digits on the candidate list; brute force at <= NFIN.
    if (collect) {
        const int ncand = min(sm.ncand, CAP);
        while (cnt > NFIN && level < NLEVEL) {
            const int sh = level_shift(level);
            if (!have_hist) {
                clear_hist(sm);
                __syncthreads();
                for (int i = tid; i < ncand; i += THREADS) {
                    const unsigned long long k = sm.cand[i];
                    if ((k & mask) == prefix) atomicAdd(&sm.hist[(k >> sh) & (NBIN - 1)], 1);
                }
                __syncthreads();
            }
            have_hist = false;
            find_crossing(sm, rem);
            prefix |= (unsigned long long)sm.cross[0] << sh;
            mask |= (unsigned long long)(NBIN - 1) << sh;
            rem = sm.cross[1];
            cnt = sm.cross[2];
            ++level;
        }
        for (int i = tid; i < ncand; i += THREADS) {
            const unsigned long long k = sm.cand[i];
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
        if (fast) {
            // Each owner decides its own candidates, found at its ranks.
            int pos = epos;
#pragma unroll
            for (int i = 0; i < 3; ++i)
                for (uint32_t m = eqw[i]; m; m &= m - 1u, ++pos)
                    if (pos < CAP && sm.cand[pos] >= kstar) selw[i] |= 1u << (__ffs(m) - 1);
        } else {
            for (int i = tid; i < ncand; i += THREADS) {
                const unsigned long long k = sm.cand[i];
                if (k >= kstar) {
                    const int s = 32767 - (int)(k & 32767u) + mis;
                    atomicOr(&sm.bits[s >> 5], 1u << (s & 31));
                }
            }
            __syncthreads();
        }
    }
    if (fast) {
#pragma unroll
        for (int i = 0; i < 3; ++i)
            if (i < nown) sm.bits[wb + i] = selw[i];
    }

    // 4. Selected free ids, ascending, after the sink.
    unsigned wv[3];
    int nbits;
    int pos = scan_words(sm, sm.bits, w0, w1, wv, nbits);
#pragma unroll
    for (int i = 0; i < 3; ++i)
        for (unsigned m = wv[i]; m && pos < nsel; m &= m - 1u, ++pos)
            if (QSA_IN(fs + pos, a.width)) out[fs + pos] = 32 * (wb + i) + __ffs(m) - 1 - mis;
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

