// qsa_fill_ids_decode / qsa_fill_ids_even: the per-token selected-id lists of
// the two workload families, written on the device.
//
// "round 5 track b: cached residual norms and fused mtp attention", section
// "mtp attention": the decode window is 64 sink cells, the 256 previous local
// cells and the token's own cell.  "round 11 track b: qsa attention and
// score", sections "boundaries and provenance" and "implementation and
// evaluator": explicit prompt lists are evenly spaced unique causal cells;
// the unused slots are poisoned with -1.
//
// One thread per id slot; every slot's value is a closed form of (token, slot),
// all in integer arithmetic, so the lists are exact.
#include <stdint.h>

#include "check.cuh"
#include "qsa_internal.h"

namespace qsa {
namespace {

__global__ void fill_decode_kernel(FillIdsLaunch a) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)a.ntok * a.width) return;
    const int t = (int)(i / a.width), j = (int)(i % a.width);
    const int p = a.pos0 + t;
    // [0, n1) sink, then [lo, p) local, then p itself.
    const int n1 = min(a.sink, p);
    const int lo = max(a.sink, p - a.local);
    const int n2 = max(0, p - lo);
    int v = -1;
    if (j < n1)
        v = j;
    else if (j < n1 + n2)
        v = lo + (j - n1);
    else if (j == n1 + n2)
        v = p;
    if (QSA_IN(i, (long long)a.ntok * a.width)) a.ids[i] = v;
}

__global__ void fill_even_kernel(FillIdsLaunch a) {
    const long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (long long)a.ntok * a.width) return;
    const int t = (int)(i / a.width), j = (int)(i % a.width);
    const long long n = (long long)a.pos0 + t + 1;  // causal cells 0 .. p
    const long long k = n < a.select ? n : a.select;
    int v = -1;
    if (j < k) v = (k == n) ? j : (int)(((long long)j * (n - 1)) / (k - 1));
    if (QSA_IN(i, (long long)a.ntok * a.width)) a.ids[i] = v;
}

}  // namespace

cudaError_t launch_fill_ids(const FillIdsLaunch &a, bool even, cudaStream_t s) {
    const long long n = (long long)a.ntok * a.width;
    if (n == 0) return cudaSuccess;
    const int threads = 256;
    const unsigned blocks = (unsigned)((n + threads - 1) / threads);
    if (even)
        fill_even_kernel<<<blocks, threads, 0, s>>>(a);
    else
        fill_decode_kernel<<<blocks, threads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa

QSA_DEFINE_CHECK_READER(take_check_word_ids)

