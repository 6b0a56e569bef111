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
// One 512-thread CTA per token.  Each thread keeps 64 of the row's scores in
// registers as order-preserving 32-bit keys (cell tid + 512 j).  A 4-pass
// radix select (8 bits per pass, shared-memory histograms) finds the key of
// the k-th best free cell; a final pass over the cells in id order marks the
// selected ones (forced, above the threshold, or tied at it with a low enough
// tie rank) and compacts them with block-wide ballot scans, so the output is
// ascending by construction.
#include "qsa.h"
#include "qsa_internal.h"

namespace qsa {
namespace {

constexpr int THREADS = 512;
constexpr int PER = 64;
constexpr int NWARP = THREADS / 32;
static_assert(THREADS * PER == kSelectMaxCells, "row capacity");

// Order-preserving key; -0 and +0 are one value (they tie, lower id first).
__device__ __forceinline__ uint32_t order_key(float f) {
    const uint32_t b = f == 0.0f ? 0u : __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

struct Row {
    int p, n, sink_end, lo;
    __device__ __forceinline__ bool forced(int c) const {
        return c < sink_end || (c >= lo && c < p) || c == p;
    }
};

// Exclusive block-wide rank of `flag` in thread order, plus the block total.
__device__ __forceinline__ int block_rank(bool flag, int *wtot, int &total) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    if (lane == 0) wtot[warp] = __popc(bal);
    __syncthreads();
    int base = 0, tot = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) {
        const int v = wtot[w];
        base += w < warp ? v : 0;
        tot += v;
    }
    __syncthreads();
    total = tot;
    return base + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(THREADS, 1) select_kernel(SelectLaunch a) {
    __shared__ int hist[256];
    __shared__ int wtot[NWARP];
    __shared__ int bcast[4];
    const int t = blockIdx.x, tid = threadIdx.x;
    int32_t *out = a.ids + (size_t)t * a.width;
    Row R;
    R.p = a.pos0 + t;
    R.n = R.p + 1;
    R.sink_end = min(a.sink, R.n);
    R.lo = max(a.sink, R.p - a.local);
    const int kbud = min(R.n, a.budget);

    if (R.n <= a.budget) {  // every causal cell is selected
        for (int c = tid; c < a.width; c += THREADS) out[c] = c < R.n ? c : -1;
        return;
    }

    // Keys of the free (not forced) causal cells; forced cells counted.
    const float *row = a.scores + (size_t)t * a.ld;
    uint32_t key[PER];
    uint64_t valid = 0;
    int nforced = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int c = tid + THREADS * j;
        key[j] = 0u;
        if (c < R.n) {
            if (R.forced(c)) {
                ++nforced;
            } else {
                key[j] = order_key(__ldg(row + c));
                valid |= 1ull << j;
            }
        }
    }
    for (int o = 16; o > 0; o >>= 1) nforced += __shfl_xor_sync(0xffffffffu, nforced, o);
    if ((tid & 31) == 0) wtot[tid >> 5] = nforced;
    __syncthreads();
    int nf = 0;
#pragma unroll
    for (int w = 0; w < NWARP; ++w) nf += wtot[w];
    __syncthreads();
    int need = kbud - nf;  // free cells to take (<= 0: forced cells only)

    // Radix select of the need-th largest free key.
    uint32_t prefix = 0u, mask = 0u;
    int ties_total = 0;
    if (need > 0) {
        for (int shift = 24; shift >= 0; shift -= 8) {
            for (int i = tid; i < 256; i += THREADS) hist[i] = 0;
            __syncthreads();
#pragma unroll
            for (int j = 0; j < PER; ++j)
                if (((valid >> j) & 1ull) && (key[j] & mask) == prefix) atomicAdd(&hist[(key[j] >> shift) & 255], 1);
            __syncthreads();
            if (tid < 32) {
                // Lane l owns digits 255-8l .. 248-8l (descending); find the digit
                // where the count from the top reaches `need`.
                int cnt[8], s = 0;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    cnt[i] = hist[255 - 8 * tid - i];
                    s += cnt[i];
                }
                int incl = s;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, o);
                    if (tid >= o) incl += v;
                }
                const int excl = incl - s;
                const bool here = excl < need && incl >= need;
                if (here) {
                    int run = excl;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (run + cnt[i] >= need) {
                            bcast[0] = 255 - 8 * tid - i;
                            bcast[1] = need - run;  // still needed within this digit
                            bcast[2] = cnt[i];      // keys with this digit (and the prefix)
                            break;
                        }
                        run += cnt[i];
                    }
                }
            }
            __syncthreads();
            prefix |= (uint32_t)bcast[0] << shift;
            mask |= 0xFFu << shift;
            need = bcast[1];
            ties_total = bcast[2];
            __syncthreads();
        }
    }
    // Now: free keys > prefix are taken, and `need` of the `ties_total` keys
    // equal to prefix, lowest ids first.
    const bool split_ties = need > 0 && need < ties_total;

    int out_base = 0, tie_base = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        if (THREADS * j >= R.n) continue;  // uniform across the block
        const int c = tid + THREADS * j;
        const bool v = (valid >> j) & 1ull;
        const bool forced = c < R.n && R.forced(c);
        const bool gt = need > 0 && v && key[j] > prefix;
        bool tie = need > 0 && v && key[j] == prefix;
        if (split_ties) {
            int tot;
            const int rank = block_rank(tie, wtot, tot);
            tie = tie && (tie_base + rank < need);
            tie_base += tot;
        }
        const bool sel = forced || gt || tie;
        int tot;
        const int pos = block_rank(sel, wtot, tot);
        if (sel) out[out_base + pos] = c;
        out_base += tot;
    }
    for (int c = out_base + tid; c < a.width; c += THREADS) out[c] = -1;
}

}  // namespace

cudaError_t launch_select(const SelectLaunch &a, cudaStream_t s) {
    if (a.ntok == 0) return cudaSuccess;
    select_kernel<<<a.ntok, THREADS, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
