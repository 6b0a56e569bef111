/*
 * qsa.h -- C ABI of the QSA attention hot path for NVIDIA GB300 (sm_103a).
 *
 * The path has three steps, named after the kernels of the audit pages on
 * sparse selected attention:
 *   qsa_prep   query RMS-norm + RoPE, K/V int8 quantisation into the cache;
 *   qsa_score  head-reduced fp32 scores of every causal cache cell;
 *   qsa_attn   chunked attention over a per-token list of selected cell ids.
 *
 * Conventions shared by every entry point:
 *  - All buffer pointers in the argument structs are DEVICE pointers owned by
 *    the caller.  The library allocates nothing and keeps no state between
 *    calls; it only reads the structs during the call.
 *  - Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL means the legacy default stream).  A QSA_OK return means the
 *    arguments were accepted and the kernels were enqueued.
 *  - Argument errors are detected on the host before anything is enqueued and
 *    are returned synchronously (QSA_ERR_INVALID_ARG, QSA_ERR_UNSUPPORTED).
 *    Argument validation makes no CUDA call.
 *  - Conditions only the device can see (an id outside [-1, cache_cells), a
 *    bounded wait that gave up) set bits (QSA_DEVERR_*) in the caller's
 *    optional device word `err` with atomicOr; read it after synchronising.
 *  - Outputs are never pre-cleared: cells a call does not define (scores
 *    beyond the causal boundary) keep whatever the caller put there.
 *  - fp16 values are passed as uint16_t bit patterns (IEEE binary16).
 *  - No C++ exception crosses this boundary.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define QSA_ABI_VERSION 3

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1,  /* null or misaligned pointer, bad size, bad dtype */
    QSA_ERR_UNSUPPORTED = 2,  /* a shape outside the built kernels (heads, head_dim, group) */
    QSA_ERR_CUDA = 3          /* a CUDA runtime call or launch failed; see qsa_last_error() */
} qsa_status;

/* Bits of the device error word. */
#define QSA_DEVERR_BAD_ID 1u   /* an id < -1 or >= cache_cells was seen and treated as padding */
#define QSA_DEVERR_TIMEOUT 2u  /* a bounded wait gave up; that launch's outputs are incomplete */

typedef enum { QSA_F32 = 0, QSA_F16 = 1 } qsa_dtype;

/*
 * qsa_prep -- "Round 36 Track C: qsa_prep Single-Barrier norm_rope & w == 128
 * tg_sum + qsa_score_mm Loop Unrolling", section "Summary & Decision": the
 * prep kernel normalises the query rows (RMS reduction, scale rs, weight g),
 * rotates the dims below QROT against partner tid ^ 32, and writes int8 K/V
 * codes kq, vq with their scales ksc, vsc ("round 11 track b: qsa attention
 * and score", "implementation and evaluator": four scale groups per row).
 *
 * For token t (position p = pos0 + t) and query head h, with x = q_in[t,h,:]:
 *   rs = 1/sqrt(mean(x^2) + eps);  y = (rs*x)*norm_w
 *   for i < rope_dims/2, a = p * fp32(rope_theta^(-2i/rope_dims)):
 *     y'[i] = y[i] cos a - y[i+rope_dims/2] sin a
 *     y'[i+rope_dims/2] = y[i+rope_dims/2] cos a + y[i] sin a
 *   q_out[t,h,:] = fp16_rne(y');  q_out_f32[t,h,:] = y' (if non-NULL)
 * K and V rows t are quantised into cache row pos0 + t, per group of `group`
 * dims: s = fp16_rne(fp32(amax/127)); code = s == 0 ? 0 :
 * clamp(rint_half_even(fp32(x / s)), -127, 127).  Bit-exact by definition.
 * With rope_k = 1 the key row is first rotated with the same pairs and
 * angles (no norm), in float32 steps: c = fp32(cos a), s = fp32(sin a) from
 * double-precision cos / sin, k'[i] = fp32(fp32(k[i] c) - fp32(k[i+h] s)),
 * k'[i+h] = fp32(fp32(k[i+h] c) + fp32(k[i] s)); the pages rotate only the
 * query rows, so this is an option (off = 0).
 * qbar_out: NULL, or a qsa_score workspace for these ntok tokens (at least
 * qsa_score_workspace_bytes(ntok, head_dim) bytes, 256-byte aligned) that
 * receives the score's head sum of the rotated queries: per token, fp32
 * qbar[d] = sum_h q_out_f32[t,h,d] in head order, scaled by the token's power
 * of two 2^e (see qsa_score) and stored as the fp16 pair hi = fp16(qbar 2^e),
 * lo = fp16(qbar 2^e - hi), with e after the rows; padding rows zero.  A
 * following qsa_score with workspace_holds_qbar = 1 then needs neither q nor
 * its own head-sum pass.
 *
 * Layouts (row-major, contiguous): q_in [ntok, n_q_heads, head_dim] fp32;
 * k_in, v_in [ntok, n_kv_heads, head_dim] fp32; norm_w [head_dim] fp32;
 * q_out [ntok, n_q_heads, head_dim] fp16; q_out_f32 same shape fp32 or NULL;
 * kq, vq [cache_cells, head_dim] int8; ksc, vsc [cache_cells, head_dim/group]
 * fp16.  Requires pos0 + ntok <= cache_cells.  Supported: n_kv_heads == 1,
 * head_dim == 128, group == 32, 1 <= n_q_heads <= 30, rope_dims a multiple
 * of 8 in [0, head_dim].  Float pointers and kq/vq must be 16-byte aligned.
 */
typedef struct {
    int ntok, pos0, n_q_heads, n_kv_heads, head_dim, group, rope_dims, cache_cells;
    float eps, rope_theta;
    const float *q_in, *k_in, *v_in, *norm_w;
    uint16_t *q_out;
    float *q_out_f32;
    int8_t *kq, *vq;
    uint16_t *ksc, *vsc;
    int rope_k; /* added in ABI version 2: 1 = rotate the key rows before quantising, 0 = not */
    void *qbar_out; /* added in ABI version 2: NULL or a qsa_score workspace, see above */
} qsa_prep_args;

/*
 * qsa_score -- "Round 36 Track C ..." section "Summary & Decision" (the
 * qsa_score_mm 64x64x128 tile matmul of queries against the int8 key cache)
 * and "round 11 track b: qsa attention and score", sections "implementation
 * and evaluator" and "score: valid negative result" (head-reduced output,
 * scalar dead-key tail, untouched beyond-causal cells).
 *
 *   scores[t*ld + c] = sum_h sum_g ksc[c,g] * sum_{d in g} q[t,h,d] * kq[c,d]
 * for 0 <= c <= pos0 + t; every other element of `scores` is left untouched.
 *
 * q: [ntok, n_q_heads, head_dim] in q_dtype (QSA_F32 or QSA_F16).
 * kq [cache_cells, head_dim] int8, ksc [cache_cells, head_dim/group] fp16.
 * scores: fp32, row stride ld (elements), ld >= pos0 + ntok.
 * workspace: device scratch of at least qsa_score_workspace_bytes(ntok,
 * head_dim) bytes, 256-byte aligned; the call overwrites it.  Two calls that
 * share a workspace must not run concurrently.  It holds the head sum the
 * score is computed from: with workspace_holds_qbar = 1 the caller has
 * already filled it through qsa_prep's qbar_out for the same tokens, q is
 * ignored (it may be NULL) and the head-sum pass is skipped; the scores are
 * bit-identical to those computed from the fp32 q_out_f32 of that prep.
 * max_ctas: 0 runs one persistent CTA per SM (each CTA takes all of an SM's
 * tensor memory); n > 0 runs at most n.  A caller that overlaps the score with
 * other kernels on another stream caps it so that those kernels keep the
 * remaining SMs; the scores do not depend on the cap.  Negative is rejected.
 * Range: the head sum qbar[t,:] = sum_h q[t,h,:] travels as an fp16 pair
 * hi + lo under a per-token power of two 2^e_t: e_t = 0 while the row's
 * largest |qbar| lies in [2^-4, 2^14), otherwise the row is scaled into
 * [2^13, 2^14) (|e_t| <= 120), and the scores are multiplied back by 2^-e_t.
 * Each element then carries about 22 significant bits relative to its row's
 * largest, for any finite row whose largest element is between about 2^-107
 * and the fp32 maximum; the scores meet 1e-4 * sum|terms| across that range.
 * Elements more than about 2^37 below their row's largest keep less (the fp16
 * lo part underflows), and a row with an inf or NaN gives non-finite scores,
 * as the definition does.
 * Requires pos0 + ntok <= cache_cells.  Supported: head_dim == 128,
 * group == 32, 1 <= n_q_heads <= 64.  q, kq 16-byte aligned; ksc 8-byte.
 */
typedef struct {
    int ntok, pos0, n_q_heads, head_dim, group, cache_cells;
    const void *q;
    int q_dtype;
    const int8_t *kq;
    const uint16_t *ksc;
    float *scores;
    int64_t ld;
    void *workspace;
    size_t workspace_bytes;
    unsigned int *err;
    int workspace_holds_qbar; /* added in ABI version 2: 0 or 1, see above */
    int max_ctas;             /* added in ABI version 3: 0 = one CTA per SM, n > 0 = at most n, see above */
} qsa_score_args;

/* Bytes of workspace qsa_score needs for `ntok` tokens (0 on bad input). */
size_t qsa_score_workspace_bytes(int ntok, int head_dim);

/*
 * qsa_attn -- "round 11 track b: qsa attention and score", section
 * "implementation and evaluator" (per-token selected ids, -1 padding, 64-cell
 * chunks, incomplete chunks) and "round 5 track b: cached residual norms and
 * fused mtp attention", sections "mtp attention" and "preflight / ownership"
 * (per-chunk maxima and denominators, max-first chunk merge, one value load
 * per dimension per cell shared by all query heads).
 *
 * For token t and head h, chunk c covers id slots 64c .. 64c+63; a slot is
 * valid when 0 <= id < cache_cells (ids < -1 or >= cache_cells are treated
 * as padding and set QSA_DEVERR_BAD_ID).  Head h reads KV head
 * kv = h / (n_q_heads / n_kv_heads) (the pages' mtp grid: two KV heads per
 * token, 12 query heads on each).
 *   s_j = softmax_scale * sum_g ksc[id,kv,g] * sum_{d in g} q[t,h,d] * kq[id,kv,d]
 *   m_c = max s_j, l_c = sum exp(s_j - m_c), o_c = sum exp(s_j - m_c) v_j
 *   with v_j[d] = vsc[id, kv, d/group] * vq[id, kv, d];
 *   O = sum_c exp(m_c - M) o_c / sum_c exp(m_c - M) l_c, M = max m_c;
 *   out = fp16(O), or with a gate (same section: "sigmoid gate", fp32 gates)
 *   out[t,h,d] = fp16(O[t,h,d] / (1 + exp(-gate[t,h,d]))).
 * A token with no valid slot outputs +0.
 *
 * q [ntok, n_q_heads, head_dim] fp16; kq, vq [cache_cells, n_kv_heads,
 * head_dim] int8; ksc, vsc [cache_cells, n_kv_heads, head_dim/group] fp16;
 * ids [ntok, width] int32, width a multiple of 64; out [ntok, n_q_heads,
 * head_dim] fp16; gate NULL or [ntok, n_q_heads, head_dim] fp32.
 * part: NULL, or [ntok, width/64, n_q_heads, head_dim + 2] fp32 receiving each
 * chunk's ungated (o_c[0..head_dim), m_c, l_c); an empty chunk gives
 * (0, -inf, 0).  A non-NULL part selects the split path (per-chunk kernel,
 * then a merge kernel that reads part back); NULL selects the fused
 * single-kernel path.  All pointers are device pointers owned by the caller.
 * Supported: (head_dim 128, group 32) -- the workload's shape -- or
 * (head_dim 256, group 64) -- the pages' own; n_q_heads a multiple of
 * n_kv_heads with 1..16 query heads per KV head; otherwise
 * QSA_ERR_UNSUPPORTED.  q, kq, vq, out, part 16-byte aligned; ksc, vsc
 * 8-byte; ids, gate 4-byte.
 */
typedef struct {
    int ntok, n_q_heads, n_kv_heads, head_dim, group, cache_cells, width;
    const uint16_t *q;
    const int8_t *kq, *vq;
    const uint16_t *ksc, *vsc;
    const int32_t *ids;
    float softmax_scale;
    uint16_t *out;
    float *part;
    unsigned int *err;
    const float *gate; /* added in ABI version 2 */
} qsa_attn_args;

/*
 * qsa_score_noalloc -- the pages have no counterpart to this entry point; it
 * exists for callers that cannot allocate device memory at the time they
 * score: for instance a plugin whose host engine owns all device memory and
 * forbids allocation inside its execute callback, or a serving loop that must
 * not call cudaMalloc because that call can synchronise the device and has no
 * latency bound.  It computes exactly what qsa_score computes, but instead of
 * the caller's workspace it uses a scratch array built into the library
 * (QSA_SCORE_NOALLOC_MAX_TOKENS * 516 bytes, about 4 MiB of device memory,
 * held on every GPU that loads the library until the process exits).  The
 * `workspace`, `workspace_bytes` and `workspace_holds_qbar` fields are ignored:
 * the head sum is always computed from q; `max_ctas` applies as in qsa_score.
 *
 *  - ntok above QSA_SCORE_NOALLOC_MAX_TOKENS is rejected with
 *    QSA_ERR_INVALID_ARG; nothing is enqueued.
 *  - It never allocates: no cudaMalloc, cudaFree or allocating library call.
 *  - The first call on each device looks up the scratch array's device
 *    address (cudaGetSymbolAddress) with that device current; make that
 *    first call before any stream capture.  The address is kept for the
 *    life of the process: it does not survive cudaDeviceReset(), after
 *    which this entry point must not be called on that device again.
 *  - All calls share the one array and it keeps the last call's contents.
 *    Every call rewrites what it reads, so nothing needs clearing, but two
 *    calls whose kernels overlap on the GPU (different streams without an
 *    ordering dependency, or different host threads) race on it and give
 *    wrong scores: order them on one stream or with events.
 */
#define QSA_SCORE_NOALLOC_MAX_TOKENS 8192
qsa_status qsa_score_noalloc(const qsa_score_args *args, void *stream);

/*
 * qsa_select -- the scores -> ids step between qsa_score and qsa_attn.  The
 * pages name its buffers ("Round 36 Track C ...", section "Summary &
 * Decision": scores, ids, pooled) and the decode window ("round 5 track b:
 * cached residual norms and fused mtp attention", section "mtp attention":
 * 64 sink + 256 previous local + 1 current cell) but not the rule; this is
 * the plainest reading.  For token t (p = pos0 + t):
 *   forced = {0 .. min(sink, p+1)-1} U {max(sink, p-local) .. p-1} U {p};
 *   the other causal cells c <= p are ranked by scores[t*ld + c] (float32,
 *   descending; equal scores, -0 and +0 included, rank the lower id first;
 *   a NaN ranks below every number, -inf included, NaNs among themselves by
 *   id) and the best min(p+1, budget) - |forced| of them are added (none
 *   when the forced cells alone reach the budget: they are all kept);
 *   ids[t, :] = the chosen cells ascending, then -1 up to width.
 * Deterministic and bit-exact for a given score array.
 * scores [ntok, ld] fp32: the ranked cells are read in aligned 16-byte
 * blocks, so up to three neighbouring cells on either side (within those
 * blocks) may be read too and are ignored; ids [ntok, width] int32, every
 * element written.  Both device pointers, owned by the caller, 4-byte
 * aligned.
 * Requires 1 <= budget <= width, width % 64 == 0, sink, local >= 0,
 * sink + local + 1 <= width and pos0 + ntok <= ld, else
 * QSA_ERR_INVALID_ARG; pos0 + ntok <= QSA_SELECT_MAX_CELLS (a row's top
 * digits are cached on chip), else QSA_ERR_UNSUPPORTED.  Nothing is
 * enqueued on an error.  Uses about 42 KB of shared memory per block and
 * no global scratch.
 */
#define QSA_SELECT_MAX_CELLS 32768
typedef struct {
    int ntok, pos0, width, budget, sink, local;
    const float *scores;
    int64_t ld;
    int32_t *ids;
} qsa_select_args;

qsa_status qsa_select(const qsa_select_args *args, void *stream);

/*
 * qsa_fill_ids_decode, qsa_fill_ids_even -- the per-token selected-id lists of
 * the two workload families, written on the device (ids [ntok, width] int32,
 * a device pointer owned by the caller, 4-byte aligned; every element is
 * written).  For token t at position p = pos0 + t:
 *  decode ("round 5 track b: cached residual norms and fused mtp attention",
 *  section "mtp attention": 64 sink + 256 previous local + the current
 *  cell): the cells 0 .. min(sink, p)-1, then max(sink, p-local) .. p-1,
 *  then p, ascending, then -1.  Requires sink + local + 1 <= width.
 *  even ("round 11 track b: qsa attention and score", sections "boundaries
 *  and provenance" and "implementation and evaluator": evenly spaced unique
 *  causal cells, unused slots poisoned with -1): with n = p + 1 and
 *  k = min(n, select), slot j < k holds j when k == n and
 *  floor(j (n-1) / (k-1)) otherwise (so 0 and p are always present), then
 *  -1.  Requires 2 <= select <= width.
 * Both are integer closed forms, exact.  Arguments are checked before
 * anything is enqueued (QSA_ERR_INVALID_ARG).
 */
qsa_status qsa_fill_ids_decode(int ntok, int pos0, int width, int sink, int local, int32_t *ids, void *stream);
qsa_status qsa_fill_ids_even(int ntok, int pos0, int width, int select, int32_t *ids, void *stream);

qsa_status qsa_prep(const qsa_prep_args *args, void *stream);
qsa_status qsa_score(const qsa_score_args *args, void *stream);
qsa_status qsa_attn(const qsa_attn_args *args, void *stream);

/*
 * qsa_check_word -- the pages have no counterpart to this call; it serves the
 * device bounds-check build of the library.  Built with QSA_CHECK=1
 * (libqsa_check.so), every kernel tests the index of its global-memory
 * accesses against the size of its buffer as the call's arguments define
 * it; an index outside sets bit 0 of a device word and that access is
 * skipped (nothing traps).  This call ORs the words of every kernel file
 * into *out (a host pointer) and clears them; it synchronises with the
 * device.  The release build returns QSA_ERR_UNSUPPORTED and writes 0.
 */
qsa_status qsa_check_word(unsigned int *out);

/* Static description of a status code. */
const char *qsa_status_str(qsa_status s);
/* Message of the last QSA_ERR_* returned on this host thread ("" if none). */
const char *qsa_last_error(void);
/* QSA_ABI_VERSION of the built library. */
int qsa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
