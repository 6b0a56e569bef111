// Device-side index checks of the QSA_CHECK build.
//
// Built with QSA_CHECK=1 (libqsa_check.so), the kernels test the index of
// their global-memory accesses against the size of the buffer, as the call's
// arguments define it (cells, tokens, widths, row pitches).  An index outside
// sets bit 0 of this translation unit's check word and the access is skipped;
// nothing traps.  qsa_check_word() reads and clears the words of every unit.
// In the release build QSA_IN(i, n) is the constant true and the checks
// compile away.
#pragma once

#include <cuda_runtime.h>

#ifndef QSA_CHECK
#define QSA_CHECK 0
#endif

namespace qsa {
namespace {

#if QSA_CHECK
__device__ unsigned int g_check_word;

__device__ __forceinline__ bool check_index(long long i, long long n) {
    if (i >= 0 && i < n) return true;
    atomicOr(&g_check_word, 1u);
    return false;
}

// This unit's word, then cleared (host; synchronises with the device).
inline cudaError_t take_unit_check_word(unsigned int *out) {
    unsigned int v = 0u, z = 0u;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_check_word, sizeof v);
    if (e == cudaSuccess) e = cudaMemcpyToSymbol(g_check_word, &z, sizeof z);
    *out = v;
    return e;
}
#define QSA_IN(i, n) ::qsa::check_index((long long)(i), (long long)(n))
#else
#define QSA_IN(i, n) true
#endif

}  // namespace
}  // namespace qsa

// Each checked .cu file defines its reader with this, under its own name.
#if QSA_CHECK
#define QSA_DEFINE_CHECK_READER(name) \
    namespace qsa {                   \
    cudaError_t name(unsigned int *out) { return take_unit_check_word(out); } \
    }
#else
#define QSA_DEFINE_CHECK_READER(name)
#endif
