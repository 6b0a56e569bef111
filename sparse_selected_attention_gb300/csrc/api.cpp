// C ABI of the QSA hot path: host-side argument validation and dispatch.
//
// Validation makes no CUDA call, so every argument error is reported before
// anything touches the device (and can be exercised on a machine without a
// GPU).  Only accepted arguments reach the launchers in the .cu files.
#include <cmath>
#include <cstdio>
#include <cstring>

#include "qsa.h"
#include "qsa_internal.h"

namespace {

thread_local char g_last_error[256] = "";

qsa_status fail(qsa_status s, const char *what) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s", what);
    return s;
}

qsa_status cuda_fail(cudaError_t e, const char *where) {
    std::snprintf(g_last_error, sizeof g_last_error, "%s: %s", where, cudaGetErrorString(e));
    return QSA_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

constexpr int kHeadDim = 128;
constexpr int kGroup = 32;
constexpr long long kMaxPos = 1ll << 29;  // positions stay exact in the rotation angle product

}  // namespace

extern "C" {

int qsa_abi_version(void) { return QSA_ABI_VERSION; }

const char *qsa_last_error(void) { return g_last_error; }

const char *qsa_status_str(qsa_status s) {
    switch (s) {
        case QSA_OK: return "ok";
        case QSA_ERR_INVALID_ARG: return "invalid argument";
        case QSA_ERR_UNSUPPORTED: return "unsupported shape";
        case QSA_ERR_CUDA: return "CUDA error";
    }
    return "unknown status";
}

size_t qsa_score_workspace_bytes(int ntok, int head_dim) {
    if (ntok < 0 || head_dim != kHeadDim) return 0;
    const size_t pad = ((size_t)ntok + qsa::kScoreTokTile - 1) / qsa::kScoreTokTile * qsa::kScoreTokTile;
    return pad * qsa::kScoreWsBytesPerTok;
}

qsa_status qsa_prep(const qsa_prep_args *a, void *stream) {
    g_last_error[0] = 0;
    if (!a) return fail(QSA_ERR_INVALID_ARG, "qsa_prep: args is NULL");
    if (a->ntok < 0 || a->pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_prep: negative ntok or pos0");
    if (a->head_dim != kHeadDim || a->group != kGroup || a->n_kv_heads != 1 || a->n_q_heads < 1 ||
        a->n_q_heads > 30)
        return fail(QSA_ERR_UNSUPPORTED, "qsa_prep: supported shapes are head_dim 128, group 32, 1 KV head, 1..30 query heads");
    if (a->rope_dims < 0 || a->rope_dims > a->head_dim || a->rope_dims % 8 != 0)
        return fail(QSA_ERR_UNSUPPORTED, "qsa_prep: rope_dims must be a multiple of 8 in [0, head_dim]");
    if ((long long)a->pos0 + a->ntok > a->cache_cells)
        return fail(QSA_ERR_INVALID_ARG, "qsa_prep: pos0 + ntok exceeds cache_cells");
    if ((long long)a->pos0 + a->ntok > kMaxPos) return fail(QSA_ERR_INVALID_ARG, "qsa_prep: positions beyond 2^29");
    if (!(a->eps >= 0.0f) || !std::isfinite(a->eps) || !(a->rope_theta > 0.0f) || !std::isfinite(a->rope_theta))
        return fail(QSA_ERR_INVALID_ARG, "qsa_prep: eps must be finite >= 0 and rope_theta finite > 0");
    if (a->rope_k != 0 && a->rope_k != 1) return fail(QSA_ERR_INVALID_ARG, "qsa_prep: rope_k must be 0 or 1");
    if (a->qbar_out && !aligned(a->qbar_out, 256)) return fail(QSA_ERR_INVALID_ARG, "qsa_prep: misaligned qbar_out");
    if (a->ntok == 0) return QSA_OK;
    if (!a->q_in || !a->k_in || !a->v_in || !a->norm_w || !a->q_out || !a->kq || !a->vq || !a->ksc || !a->vsc)
        return fail(QSA_ERR_INVALID_ARG, "qsa_prep: NULL buffer");
    if (!aligned(a->q_in, 16) || !aligned(a->k_in, 16) || !aligned(a->v_in, 16) || !aligned(a->norm_w, 16) ||
        !aligned(a->q_out, 16) || (a->q_out_f32 && !aligned(a->q_out_f32, 16)) || !aligned(a->kq, 16) ||
        !aligned(a->vq, 16) || !aligned(a->ksc, 8) || !aligned(a->vsc, 8))
        return fail(QSA_ERR_INVALID_ARG, "qsa_prep: misaligned buffer");
    qsa::PrepLaunch L{};
    L.ntok = a->ntok;
    L.pos0 = a->pos0;
    L.n_q_heads = a->n_q_heads;
    L.rope_dims = a->rope_dims;
    L.eps = a->eps;
    L.rope_theta = a->rope_theta;
    L.rope_k = a->rope_k;
    L.cache_cells = a->cache_cells;
    L.qbar = static_cast<uint16_t *>(a->qbar_out);
    L.ntok_pad = (a->ntok + 63) / 64 * 64;
    L.qexp = a->qbar_out ? reinterpret_cast<int *>(static_cast<uint8_t *>(a->qbar_out) +
                                                   (size_t)L.ntok_pad * qsa::kScoreRowBytes)
                         : nullptr;
    L.q_in = a->q_in;
    L.k_in = a->k_in;
    L.v_in = a->v_in;
    L.norm_w = a->norm_w;
    L.q_out = a->q_out;
    L.q_out_f32 = a->q_out_f32;
    L.kq = a->kq;
    L.vq = a->vq;
    L.ksc = a->ksc;
    L.vsc = a->vsc;
    cudaError_t e = qsa::launch_prep(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_prep");
}

qsa_status qsa_score(const qsa_score_args *a, void *stream) {
    g_last_error[0] = 0;
    if (!a) return fail(QSA_ERR_INVALID_ARG, "qsa_score: args is NULL");
    if (a->ntok < 0 || a->pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_score: negative ntok or pos0");
    if (a->head_dim != kHeadDim || a->group != kGroup || a->n_q_heads < 1 || a->n_q_heads > 64)
        return fail(QSA_ERR_UNSUPPORTED, "qsa_score: supported shapes are head_dim 128, group 32, 1..64 query heads");
    if (a->q_dtype != QSA_F32 && a->q_dtype != QSA_F16) return fail(QSA_ERR_INVALID_ARG, "qsa_score: bad q_dtype");
    if ((long long)a->pos0 + a->ntok > a->cache_cells)
        return fail(QSA_ERR_INVALID_ARG, "qsa_score: pos0 + ntok exceeds cache_cells");
    if (a->ld < (long long)a->pos0 + a->ntok) return fail(QSA_ERR_INVALID_ARG, "qsa_score: ld < pos0 + ntok");
    if (a->workspace_holds_qbar != 0 && a->workspace_holds_qbar != 1)
        return fail(QSA_ERR_INVALID_ARG, "qsa_score: workspace_holds_qbar must be 0 or 1");
    if (a->max_ctas < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_score: negative max_ctas");
    if (a->ntok == 0) return QSA_OK;
    const bool need_q = !a->workspace_holds_qbar;
    if ((need_q && !a->q) || !a->kq || !a->ksc || !a->scores || !a->workspace)
        return fail(QSA_ERR_INVALID_ARG, "qsa_score: NULL buffer");
    if (a->workspace_bytes < qsa_score_workspace_bytes(a->ntok, a->head_dim))
        return fail(QSA_ERR_INVALID_ARG, "qsa_score: workspace smaller than qsa_score_workspace_bytes()");
    if ((need_q && !aligned(a->q, 16)) || !aligned(a->kq, 16) || !aligned(a->ksc, 8) || !aligned(a->scores, 4) ||
        !aligned(a->workspace, 256))
        return fail(QSA_ERR_INVALID_ARG, "qsa_score: misaligned buffer");
    const size_t pad = (size_t)(a->ntok + qsa::kScoreTokTile - 1) / qsa::kScoreTokTile * qsa::kScoreTokTile;
    qsa::ScoreLaunch L{a->ntok,   a->pos0, a->n_q_heads, a->cache_cells, a->q, a->q_dtype == QSA_F16 ? 1 : 0,
                       a->kq,     a->ksc,  a->scores,    a->ld,          static_cast<uint16_t *>(a->workspace),
                       reinterpret_cast<int *>(static_cast<uint8_t *>(a->workspace) + pad * qsa::kScoreRowBytes),
                       a->err,    a->workspace_holds_qbar, a->max_ctas};
    cudaError_t e = qsa::launch_score(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_score");
}

qsa_status qsa_attn(const qsa_attn_args *a, void *stream) {
    g_last_error[0] = 0;
    if (!a) return fail(QSA_ERR_INVALID_ARG, "qsa_attn: args is NULL");
    if (a->ntok < 0 || a->cache_cells < 1) return fail(QSA_ERR_INVALID_ARG, "qsa_attn: negative ntok or empty cache");
    const bool shape128 = a->head_dim == 128 && a->group == 32, shape256 = a->head_dim == 256 && a->group == 64;
    if (!(shape128 || shape256) || a->n_kv_heads < 1 || a->n_q_heads < 1 || a->n_q_heads % a->n_kv_heads != 0 ||
        a->n_q_heads / a->n_kv_heads > 16 || a->n_kv_heads > 65535)
        return fail(QSA_ERR_UNSUPPORTED,
                    "qsa_attn: supported shapes are (head_dim 128, group 32) or (head_dim 256, group 64), "
                    "n_q_heads a multiple of n_kv_heads with at most 16 query heads per KV head");
    if (a->width <= 0 || a->width % 64 != 0)
        return fail(QSA_ERR_INVALID_ARG, "qsa_attn: width must be a positive multiple of 64");
    if (!std::isfinite(a->softmax_scale)) return fail(QSA_ERR_INVALID_ARG, "qsa_attn: softmax_scale not finite");
    if (a->ntok == 0) return QSA_OK;
    if (!a->q || !a->kq || !a->vq || !a->ksc || !a->vsc || !a->ids || !a->out)
        return fail(QSA_ERR_INVALID_ARG, "qsa_attn: NULL buffer");
    if (!aligned(a->q, 16) || !aligned(a->kq, 16) || !aligned(a->vq, 16) || !aligned(a->ksc, 8) ||
        !aligned(a->vsc, 8) || !aligned(a->ids, 4) || !aligned(a->out, 16) || (a->part && !aligned(a->part, 16)) ||
        (a->gate && !aligned(a->gate, 4)))
        return fail(QSA_ERR_INVALID_ARG, "qsa_attn: misaligned buffer");
    qsa::AttnLaunch L{a->ntok,   a->n_q_heads, a->cache_cells, a->width, a->q,          a->kq,
                      a->vq,     a->ksc,       a->vsc,         a->ids,   a->softmax_scale, a->out,
                      a->part,   a->err,       a->n_kv_heads,  a->head_dim, a->gate};
    cudaError_t e = qsa::launch_attn(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_attn");
}

qsa_status qsa_select(const qsa_select_args *a, void *stream) {
    g_last_error[0] = 0;
    if (!a) return fail(QSA_ERR_INVALID_ARG, "qsa_select: args is NULL");
    if (a->ntok < 0 || a->pos0 < 0 || a->sink < 0 || a->local < 0 || a->budget < 1)
        return fail(QSA_ERR_INVALID_ARG, "qsa_select: negative ntok/pos0/sink/local or budget < 1");
    if (a->width <= 0 || a->width % 64 != 0 || a->budget > a->width)
        return fail(QSA_ERR_INVALID_ARG, "qsa_select: width must be a positive multiple of 64 and >= budget");
    if (a->ld < (long long)a->pos0 + a->ntok) return fail(QSA_ERR_INVALID_ARG, "qsa_select: ld < pos0 + ntok");
    if ((long long)a->pos0 + a->ntok > QSA_SELECT_MAX_CELLS)
        return fail(QSA_ERR_UNSUPPORTED, "qsa_select: rows longer than QSA_SELECT_MAX_CELLS cells");
    if ((long long)a->sink + a->local + 1 > a->width)
        return fail(QSA_ERR_INVALID_ARG, "qsa_select: the forced window (sink + local + 1) exceeds width");
    if (a->ntok == 0) return QSA_OK;
    if (!a->scores || !a->ids) return fail(QSA_ERR_INVALID_ARG, "qsa_select: NULL buffer");
    if (!aligned(a->scores, 4) || !aligned(a->ids, 4)) return fail(QSA_ERR_INVALID_ARG, "qsa_select: misaligned buffer");
    qsa::SelectLaunch L{a->ntok, a->pos0, a->width, a->budget, a->sink, a->local, a->scores, a->ld, a->ids};
    cudaError_t e = qsa::launch_select(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_select");
}

qsa_status qsa_fill_ids_decode(int ntok, int pos0, int width, int sink, int local, int32_t *ids, void *stream) {
    g_last_error[0] = 0;
    if (ntok < 0 || pos0 < 0 || sink < 0 || local < 0)
        return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_decode: negative ntok, pos0, sink or local");
    if (width <= 0 || (long long)sink + local + 1 > width)
        return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_decode: width must hold sink + local + 1 ids");
    if ((long long)pos0 + ntok > 0x7fffffffll) return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_decode: positions beyond int32");
    if (ntok == 0) return QSA_OK;
    if (!ids || !aligned(ids, 4)) return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_decode: NULL or misaligned ids");
    qsa::FillIdsLaunch L{ntok, pos0, width, sink, local, 0, ids};
    cudaError_t e = qsa::launch_fill_ids(L, false, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_fill_ids_decode");
}

qsa_status qsa_fill_ids_even(int ntok, int pos0, int width, int select, int32_t *ids, void *stream) {
    g_last_error[0] = 0;
    if (ntok < 0 || pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_even: negative ntok or pos0");
    if (select < 2 || width <= 0 || select > width)
        return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_even: need 2 <= select <= width");
    if ((long long)pos0 + ntok > 0x7fffffffll) return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_even: positions beyond int32");
    if (ntok == 0) return QSA_OK;
    if (!ids || !aligned(ids, 4)) return fail(QSA_ERR_INVALID_ARG, "qsa_fill_ids_even: NULL or misaligned ids");
    qsa::FillIdsLaunch L{ntok, pos0, width, 0, 0, select, ids};
    cudaError_t e = qsa::launch_fill_ids(L, true, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_fill_ids_even");
}

qsa_status qsa_check_word(unsigned int *out) {
    g_last_error[0] = 0;
    if (!out) return fail(QSA_ERR_INVALID_ARG, "qsa_check_word: out is NULL");
#if QSA_CHECK
    unsigned int w = 0u;
    cudaError_t (*const readers[])(unsigned int *) = {qsa::take_check_word_attn, qsa::take_check_word_score,
                                                      qsa::take_check_word_prep, qsa::take_check_word_select,
                                                      qsa::take_check_word_ids};
    for (auto rd : readers) {
        unsigned int v = 0u;
        const cudaError_t e = rd(&v);
        if (e != cudaSuccess) return cuda_fail(e, "qsa_check_word");
        w |= v;
    }
    *out = w;
    return QSA_OK;
#else
    *out = 0u;
    return fail(QSA_ERR_UNSUPPORTED, "qsa_check_word: this library was built without device index checks (QSA_CHECK)");
#endif
}

// Allocation-free scoring: same checks as qsa_score minus the workspace, plus
// the built-in scratch limit.
qsa_status qsa_score_noalloc(const qsa_score_args *a, void *stream) {
    g_last_error[0] = 0;
    if (!a) return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: args is NULL");
    if (a->ntok < 0 || a->pos0 < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: negative ntok or pos0");
    if (a->ntok > QSA_SCORE_NOALLOC_MAX_TOKENS)
        return fail(QSA_ERR_INVALID_ARG,
                    "qsa_score_noalloc: ntok exceeds the built-in scratch limit (QSA_SCORE_NOALLOC_MAX_TOKENS = 8192); "
                    "use qsa_score with a workspace");
    if (a->head_dim != kHeadDim || a->group != kGroup || a->n_q_heads < 1 || a->n_q_heads > 64)
        return fail(QSA_ERR_UNSUPPORTED,
                    "qsa_score_noalloc: supported shapes are head_dim 128, group 32, 1..64 query heads");
    if (a->q_dtype != QSA_F32 && a->q_dtype != QSA_F16)
        return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: bad q_dtype");
    if ((long long)a->pos0 + a->ntok > a->cache_cells)
        return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: pos0 + ntok exceeds cache_cells");
    if (a->ld < (long long)a->pos0 + a->ntok) return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: ld < pos0 + ntok");
    if (a->max_ctas < 0) return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: negative max_ctas");
    if (a->ntok == 0) return QSA_OK;
    if (!a->q || !a->kq || !a->ksc || !a->scores) return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: NULL buffer");
    if (!aligned(a->q, 16) || !aligned(a->kq, 16) || !aligned(a->ksc, 8) || !aligned(a->scores, 4))
        return fail(QSA_ERR_INVALID_ARG, "qsa_score_noalloc: misaligned buffer");
    qsa::ScoreLaunch L{a->ntok, a->pos0, a->n_q_heads, a->cache_cells, a->q, a->q_dtype == QSA_F16 ? 1 : 0,
                       a->kq,   a->ksc,  a->scores,    a->ld,          nullptr, nullptr, a->err,
                       0,       a->max_ctas};
    cudaError_t e = qsa::launch_score_noalloc(L, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? QSA_OK : cuda_fail(e, "qsa_score_noalloc");
}

}  // extern "C"
