// Internal launch interface between the C ABI (api.cpp) and the kernels.
// Host-only declarations; every pointer here has already been validated.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace qsa {

struct PrepLaunch {
    int ntok, pos0, n_q_heads, rope_dims;
    float eps, rope_theta;
    float inv_freq[64];  // fp32(rope_theta^(-2i/rope_dims)), i < rope_dims/2, filled by the launcher
    const float *q_in, *k_in, *v_in, *norm_w;
    uint16_t *q_out;
    float *q_out_f32;
    int8_t *kq, *vq;
    uint16_t *ksc, *vsc;
    int rope_k;  // rotate the key rows (same pairs and angles as the queries) before quantising
    uint16_t *qbar;  // NULL or [ntok_pad, 2, 128] fp16: the score's scaled head sum (hi row, lo row)
    int *qexp;       // [ntok_pad]: each token's power-of-two exponent of that scaling (with qbar)
    int ntok_pad;    // ntok rounded up to 64 (rows of qbar)
    int cache_cells; // rows of kq, vq, ksc, vsc
};

struct ScoreLaunch {
    int ntok, pos0, n_q_heads, cache_cells;
    const void *q;
    int q_f16;
    const int8_t *kq;
    const uint16_t *ksc;
    float *scores;
    int64_t ld;
    uint16_t *qsum;  // workspace: [ntok_pad, 2, 128] fp16 (hi row, lo row) of the scaled head sum,
    int *qexp;       // then [ntok_pad] int32 exponents: head sum = (hi + lo) * 2^-qexp
    unsigned int *err;
    int qsum_ready;  // the workspace already holds the head sum (written by prep)
    int max_ctas;    // 0: one persistent CTA per SM; n > 0: at most n
};

struct AttnLaunch {
    int ntok, n_q_heads, cache_cells, width;
    const uint16_t *q;
    const int8_t *kq, *vq;
    const uint16_t *ksc, *vsc;
    const int32_t *ids;
    float softmax_scale;
    uint16_t *out;
    float *part;
    unsigned int *err;
    int n_kv_heads, head_dim;  // head_dim 128 (group 32) or 256 (group 64): four scale groups per row
    const float *gate;         // NULL or [ntok, n_q_heads, head_dim] output-gate logits
};

struct SelectLaunch {
    int ntok, pos0, width, budget, sink, local;
    const float *scores;
    int64_t ld;
    int32_t *ids;
};

struct FillIdsLaunch {
    int ntok, pos0, width;
    int sink, local;  // decode window
    int select;       // even lists: cells per token (at most)
    int32_t *ids;     // [ntok, width]
};

// Launches `kernel` as a programmatic dependent of the previous kernel in the
// stream: its CTAs may be scheduled while that kernel finishes, and each one
// waits (griddepcontrol.wait, at its start) for that grid's completion and
// memory before it reads anything.  With no such predecessor it runs as a
// plain launch.
template <class... Args, class... Params>
cudaError_t launch_dependent(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                             Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

#ifdef __CUDACC__
// The two halves of a programmatic dependency (sm_90 and later).
__device__ __forceinline__ void wait_for_previous_grid() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;"); }
#endif

// Longest score row (cells) the selection kernel holds on chip.
constexpr int kSelectMaxCells = 32768;

// Token rows of the score workspace are padded to this multiple.
constexpr int kScoreTokTile = 64;
// Workspace bytes per (padded) token: the fp16 hi and lo rows of 128 dims,
// then one int32 exponent.
constexpr int kScoreRowBytes = 2 * 128 * 2;
constexpr int kScoreWsBytesPerTok = kScoreRowBytes + 4;

#ifdef __CUDACC__
// The head sum's per-token power of two.  m is the largest |qbar[t, d]| of
// the token.  The fp16 hi/lo pair represents values in [2^-4, 2^14) to about
// 2^-22 of the row's maximum, so such rows keep exponent 0 (no scaling, the
// common case); other finite non-zero rows are scaled by 2^e so that m 2^e
// lies in [2^13, 2^14), with e limited to [-120, 120] so that 2^-e stays a
// normal float.  A zero, infinite or all-NaN row keeps 0.
__device__ __forceinline__ int head_sum_exponent(float m) {
    if (!(m > 0.0f) || m > 3.4028234663852886e38f) return 0;
    if (m >= 0.0625f && m < 16384.0f) return 0;
    int adj = 0;
    if (m < 1e-30f) {  // bring subnormal maxima into the normal range first (exact)
        m *= 18446744073709551616.0f;  // 2^64
        adj = 64;
    }
    const int lg = (int)((__float_as_uint(m) >> 23) & 0xFFu) - 127 - adj;  // floor(log2 m)
    const int e = 13 - lg;
    return e < -120 ? -120 : (e > 120 ? 120 : e);
}
__device__ __forceinline__ float exp2i(int e) { return __uint_as_float((uint32_t)(127 + e) << 23); }  // |e| <= 126
#endif

cudaError_t launch_prep(const PrepLaunch &a, cudaStream_t s);
cudaError_t launch_score(const ScoreLaunch &a, cudaStream_t s);
// Same launch with the library's static scratch array as the workspace;
// a.qsum is ignored.  At most QSA_SCORE_NOALLOC_MAX_TOKENS tokens.
cudaError_t launch_score_noalloc(const ScoreLaunch &a, cudaStream_t s);
cudaError_t launch_attn(const AttnLaunch &a, cudaStream_t s);
cudaError_t launch_select(const SelectLaunch &a, cudaStream_t s);
// Decode windows (even = false) or evenly spaced causal lists (even = true).
cudaError_t launch_fill_ids(const FillIdsLaunch &a, bool even, cudaStream_t s);

#if QSA_CHECK
// The QSA_CHECK build's per-file check words (check.cuh), read and cleared.
cudaError_t take_check_word_attn(unsigned int *out);
cudaError_t take_check_word_score(unsigned int *out);
cudaError_t take_check_word_prep(unsigned int *out);
cudaError_t take_check_word_select(unsigned int *out);
cudaError_t take_check_word_ids(unsigned int *out);
#endif

}  // namespace qsa
