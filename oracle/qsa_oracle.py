"""CPU oracle for the QSA attention hot path (test infrastructure only).

Only the test suite, the smoke check in ``__graft_entry__`` and the CPU-baseline
leg of ``bench.py`` import this module.  The product path never calls it and
shares no code with it: the CUDA kernels live in
``sparse_selected_attention_gb300/csrc`` and this file is plain numpy.

Arithmetic is float64 except where the method fixes a narrower type: the K/V
quantiser is an encoding, so its float32 division, fp16 scale rounding and
round-half-to-even are its definition and are reproduced exactly here.

Sources.  The pages describe Metal kernels by name, buffer list and preserved
invariants rather than by formulas:

* "Round 36 Track C: qsa_prep Single-Barrier norm_rope & w == 128 tg_sum +
  qsa_score_mm Loop Unrolling" (argon_r36_qsa), section "Summary & Decision":
  qsa_prep writes the query row, the int8 K/V codes and their scales; norm_rope
  is an RMS reduction, a scale ``rs``, a weight ``g`` and a rotation of the
  dims below QROT with partner ``tid ^ 32``; qsa_score_mm is a 64x64x128
  tile matmul.
* "round 11 track b: qsa attention and score" (sol_r11_qsa), sections
  "boundaries and provenance", "implementation and evaluator" and "score:
  valid negative result": random signed int8 caches with positive fp16 scales,
  four scale groups per row, padding ids of -1, incomplete 64-cell chunks,
  a head-reduced score tile, beyond-causal score cells left untouched.
* "round 5 track b: cached residual norms and fused mtp attention"
  (sol_r5_mtp_qsa), section "mtp attention" and "preflight / ownership":
  per-64-cell chunk arithmetic, per-chunk maxima and denominators, a
  max-first chunk merge, and value accumulation shared by all 12 heads.

Readings taken where the pages are silent are restated next to each function.

Pins (tests/test_oracle_pins.py):
  quantize_rows   -- hand-derived codes and scales, invariants (round trip
                     within half a step, group maximum maps to +-127, zero
                     groups, code range), a brute-force per-element loop.
  prep_queries    -- closed form for constant rows, identity rotation at
                     position 0, pair-norm preservation, rotation composition,
                     one-hot closed form (cos/sin of the position).
  score           -- closed form for one-hot queries, zero-scale cells,
                     head linearity, and the special case equal to a dense
                     library matmul on dequantised keys.
  attention       -- width-1 closed form, equal-score mean, dense causal
                     softmax attention (torch scaled_dot_product_attention in
                     float64) for contiguous ids, chunked = unchunked softmax,
                     padding / permutation / duplication invariants.
  select_ids      -- hand-built tiny rows (ranking by score, ties to the
                     lower id, forced cells, causality), invariants on random
                     rows (count, forced cells present, every selected free
                     cell outranks every unselected one), and the special case
                     of short contexts where every causal cell is selected.
No function is left without a pin.
"""
from __future__ import annotations

import numpy as np

LOG2E = 1.4426950408889634


# ---------------------------------------------------------------------------
# qsa_prep: query RMS-norm + RoPE  (argon_r36_qsa, "Summary & Decision")
# ---------------------------------------------------------------------------

def rope_inv_freq(rope_dims: int, theta: float) -> np.ndarray:
    """Rotation frequencies of the pairs (i, i + rope_dims/2), i < rope_dims/2.

    Reading: the pages give the pairing (partner tid ^ 32 for tid < QROT=64)
    but not the frequency table; the plainest reading is the usual RoPE table
    theta ** (-2 i / rope_dims), stored as float32.
    """
    half = rope_dims // 2
    i = np.arange(half, dtype=np.float64)
    return (float(theta) ** (-2.0 * i / rope_dims)).astype(np.float32)


def prep_queries(q_in: np.ndarray, norm_w: np.ndarray, pos0: int, eps: float = 1e-6,
                 rope_theta: float = 10000.0, rope_dims: int = 64):
    """RMS-norm each (token, head) row, weight it, then rotate dims < rope_dims.

    rs = 1 / sqrt(mean(x^2) + eps); y = (rs * x) * g   (the pages' order)
    for i < rope_dims/2, a = (pos0 + t) * inv_freq_i:
        y'_i        = y_i cos a - y_{i+h} sin a
        y'_{i+h}    = y_{i+h} cos a + y_i sin a          (h = rope_dims/2)
    dims >= rope_dims pass through.

    Returns (y' in float64, fp16 round-to-nearest of y', float32 of y').
    """
    x = q_in.astype(np.float64)
    T, H, D = x.shape
    g = norm_w.astype(np.float64)
    rs = 1.0 / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + float(eps))
    y = (rs * x) * g
    out = y.copy()
    half = rope_dims // 2
    if half > 0:
        pos = (pos0 + np.arange(T, dtype=np.float64))[:, None, None]
        a = pos * rope_inv_freq(rope_dims, rope_theta).astype(np.float64)[None, None, :]
        c, s = np.cos(a), np.sin(a)
        lo, hi = y[..., :half], y[..., half:rope_dims]
        out[..., :half] = lo * c - hi * s
        out[..., half:rope_dims] = hi * c + lo * s
    return out, out.astype(np.float16), out.astype(np.float32)


# ---------------------------------------------------------------------------
# qsa_prep: K/V int8 quantiser  (argon_r36_qsa "Summary & Decision" buffer
# list kq, vq, ksc, vsc; sol_r11_qsa "implementation and evaluator": four
# scale groups per row)
# ---------------------------------------------------------------------------

def quantize_rows(x: np.ndarray, group: int = 32):
    """Symmetric int8 codes with one fp16 scale per `group` consecutive dims.

    Reading (the pages fix int8 codes in [-127, 127] and fp16 scales only):
      amax = max |x| over the group            (float32, exact)
      s    = fp16_rne(float32(amax / 127))     (float32 IEEE division)
      code = 0                                 if s == 0
           = clamp(rint_half_even(float32(x / s)), -127, 127) otherwise
    The division uses the stored (fp16) scale, so decoding code * s is the
    value the cache represents.  Returns (codes int8 [..., D],
    scales float16 [..., D // group]).
    """
    x = np.asarray(x, dtype=np.float32)
    shp = x.shape
    D = shp[-1]
    xg = x.reshape(-1, D // group, group)
    amax = np.max(np.abs(xg), axis=-1)
    with np.errstate(over="ignore"):
        s32 = (amax / np.float32(127.0)).astype(np.float32)
        s16 = s32.astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.rint(xg / np.where(sf == 0, np.float32(1.0), sf))
    codes = np.where(sf == 0, np.float32(0.0), np.clip(r, -127.0, 127.0)).astype(np.int8)
    return codes.reshape(shp), s16.reshape(shp[:-1] + (D // group,))


def rotate_keys_f32(k_in: np.ndarray, pos0: int, rope_theta: float = 10000.0, rope_dims: int = 64):
    """Optional RoPE on the new key rows before they are quantised.

    Reading (the pages rotate the query rows in norm_rope and say nothing of
    the keys; rotating keys with the same pairs and angles is the usual RoPE
    and is offered as an option): for i < h = rope_dims/2 and a = (pos0 + t)
    * inv_freq_i (exact in float64),
        c = fp32(cos a), s = fp32(sin a)            (from float64 cos / sin)
        k'_i     = fp32(fp32(k_i * c) - fp32(k_{i+h} * s))
        k'_{i+h} = fp32(fp32(k_{i+h} * c) + fp32(k_i * s))
    every step rounded to float32 in that order.  The rotated values decide
    the int8 codes, so the arithmetic that makes them is part of the
    definition: the GPU takes the same float32 steps.  No norm on keys.
    """
    k = np.array(k_in, dtype=np.float32, copy=True)
    T = k.shape[0]
    half = rope_dims // 2
    if half == 0:
        return k
    pos = (pos0 + np.arange(T, dtype=np.float64))[:, None, None]
    a = pos * rope_inv_freq(rope_dims, rope_theta).astype(np.float64)[None, None, :]
    c, sn = np.cos(a).astype(np.float32), np.sin(a).astype(np.float32)
    lo, hi = k[..., :half].copy(), k[..., half:rope_dims].copy()
    k[..., :half] = (lo * c).astype(np.float32) - (hi * sn).astype(np.float32)
    k[..., half:rope_dims] = (hi * c).astype(np.float32) + (lo * sn).astype(np.float32)
    return k


def prep(q_in, k_in, v_in, norm_w, pos0, kq, vq, ksc, vsc, eps=1e-6,
         rope_theta=10000.0, rope_dims=64, group=32, rope_k=False):
    """The whole prep step: queries normalised and rotated, K/V rows
    quantised into cache rows pos0 .. pos0+T-1 (one KV head); with rope_k
    the key rows are rotated first (rotate_keys_f32).  The cache arrays are
    updated in place; returns prep_queries' triple."""
    T = q_in.shape[0]
    q64, q16, q32 = prep_queries(q_in, norm_w, pos0, eps, rope_theta, rope_dims)
    if rope_k:
        k_in = rotate_keys_f32(k_in, pos0, rope_theta, rope_dims)
    kc, ks = quantize_rows(k_in.reshape(T, -1), group)
    vc, vs = quantize_rows(v_in.reshape(T, -1), group)
    kq[pos0:pos0 + T] = kc
    ksc[pos0:pos0 + T] = ks
    vq[pos0:pos0 + T] = vc
    vsc[pos0:pos0 + T] = vs
    return q64, q16, q32


# ---------------------------------------------------------------------------
# qsa_score_mm  (argon_r36_qsa "Summary & Decision"; sol_r11_qsa "score:
# valid negative result" and "implementation and evaluator")
# ---------------------------------------------------------------------------

def score(q: np.ndarray, kq: np.ndarray, ksc: np.ndarray, pos0: int, rows=None, group: int = 32):
    """Head-reduced score of every causal cell.

    S[t, c] = sum_h sum_g ksc[c, g] * sum_{d in g} q[t, h, d] * kq[c, d]
    for c <= pos0 + t; cells beyond that are not defined (NaN here; the GPU
    must leave them untouched).  Reading: no softmax scale, weights or
    nonlinearity are mentioned, and the rejected variants' head reduction was
    bitwise equal to the baseline, so the output is the plain sum over heads.

    `rows` selects token indices (default all); returns float64 [len(rows), C].
    """
    q = np.asarray(q)
    T, H, D = q.shape
    rows = np.arange(T) if rows is None else np.asarray(rows)
    C = kq.shape[0]
    qf = q[rows].astype(np.float64)
    kf = kq.astype(np.float64)
    sf = ksc.astype(np.float64)
    S = np.zeros((len(rows), C), dtype=np.float64)
    for h in range(H):
        for g in range(D // group):
            sl = slice(g * group, (g + 1) * group)
            S += sf[None, :, g] * (qf[:, h, sl] @ kf[:, sl].T)
    causal = np.arange(C)[None, :] <= (pos0 + rows)[:, None]
    S[~causal] = np.nan
    return S


def score_abs_bound(q, kq, ksc, pos0, rows=None, group: int = 32):
    """A[t, c] = sum_h sum_g ksc[c,g] sum_{d in g} |q[t,h,d] * kq[c,d]|, the
    magnitude that bounds the rounding error of any evaluation order of S."""
    return score(np.abs(np.asarray(q, dtype=np.float64)), np.abs(kq.astype(np.float64)),
                 np.abs(ksc.astype(np.float64)), pos0, rows, group)


# ---------------------------------------------------------------------------
# qsa_attn_mm / qsa_flash / qsa_mtp_attn_merge  (sol_r11_qsa "implementation
# and evaluator"; sol_r5_mtp_qsa "mtp attention" and "preflight / ownership";
# sol_r32_qsa "contract")
# ---------------------------------------------------------------------------

CHUNK = 64


def attention(q: np.ndarray, kq, vq, ksc, vsc, ids: np.ndarray, softmax_scale: float,
              rows=None, group: int = 32, want_part: bool = False, gate=None):
    """Chunked attention over each token's selected cells, max-first merge.

    For token t and head h, chunk c holds id slots 64c .. 64c+63; J_c is the
    set of slots with a valid id (0 <= id < cells; -1 and out-of-range ids
    are padding and contribute nothing).  Head h reads KV head
    kv = h // (H / Hkv) ("round 5 track b: cached residual norms and fused mtp
    attention", section "mtp attention": a grid of 2 KV heads per token, 24
    heads of partials, 12 query heads per KV row).  kq, vq are [cells, D] for
    one KV head or [cells, Hkv, D]; ksc, vsc [cells, D/group] or
    [cells, Hkv, D/group].
      s_j  = scale * sum_g ksc[id,kv,g] * sum_{d in g} q[t,h,d] * kq[id,kv,d]
      m_c  = max_{j in J_c} s_j ;  p_j = exp(s_j - m_c) ;  l_c = sum p_j
      o_c[d] = sum_j p_j * vsc[id, kv, d // group] * vq[id, kv, d]
    Empty chunks are skipped.  Merge (max-first):
      M = max_c m_c ; L = sum_c exp(m_c - M) l_c ;  O = sum_c exp(m_c - M) o_c / L
    Output gate (same section: "sigmoid gate", fp32 gates beside the fp32
    queries), optional, one value per (t, h, d):
      out = fp16_rne( O * 1 / (1 + exp(-gate[t,h,d])) )   (ungated: fp16_rne(O))
    A token with no valid id outputs +0.

    Returns (out float64 [R,H,D] before fp16 rounding, out fp16,
    part float64 [R, W/64, H, D+2] = (o_c, m_c, l_c) or None, bad_id flag).
    The partials are the ungated chunk values.
    """
    q = np.asarray(q)
    T, H, D = q.shape
    kq, vq, ksc, vsc = (np.asarray(x) for x in (kq, vq, ksc, vsc))
    if kq.ndim == 2:                                       # one KV head
        kq, vq, ksc, vsc = kq[:, None], vq[:, None], ksc[:, None], vsc[:, None]
    Hkv = kq.shape[1]
    assert H % Hkv == 0, "query heads must split evenly over the KV heads"
    per = H // Hkv
    rows = np.arange(T) if rows is None else np.asarray(rows)
    C = kq.shape[0]
    W = ids.shape[1]
    nch = (W + CHUNK - 1) // CHUNK
    ng = D // group
    out = np.zeros((len(rows), H, D), dtype=np.float64)
    part = np.zeros((len(rows), nch, H, D + 2), dtype=np.float64) if want_part else None
    bad = bool(np.any((ids < -1) | (ids >= C)))
    kscale = ksc.astype(np.float64)
    vscale = vsc.astype(np.float64)
    for r, t in enumerate(rows):
        row = np.full(nch * CHUNK, -1, dtype=np.int64)
        row[:W] = ids[t]
        row = row.reshape(nch, CHUNK)
        valid = (row >= 0) & (row < C)
        safe = np.where(valid, row, 0)
        nonempty = valid.any(axis=1)                       # [nch]
        for kv in range(Hkv):
            hs = slice(kv * per, (kv + 1) * per)
            qt = q[t, hs].astype(np.float64)               # [per, D]
            k = kq[safe, kv].astype(np.float64)            # [nch, 64, D]
            v = vq[safe, kv].astype(np.float64)
            s = np.zeros((nch, CHUNK, per), dtype=np.float64)
            for g in range(ng):
                sl = slice(g * group, (g + 1) * group)
                s += kscale[safe, kv][..., g:g + 1] * (k[..., sl] @ qt[:, sl].T)
            s *= softmax_scale
            s = np.where(valid[..., None], s, -np.inf)
            m = np.where(nonempty[:, None], s.max(axis=1), -np.inf)     # [nch, per]
            p = np.where(valid[..., None], np.exp(s - np.where(nonempty[:, None], m, 0.0)[:, None, :]), 0.0)
            l = p.sum(axis=1)                              # [nch, per]
            vdq = v * np.repeat(vscale[safe, kv], group, axis=-1)       # [nch, 64, D]
            o = np.einsum("cjh,cjd->chd", p, vdq)          # [nch, per, D]
            if want_part:
                part[r, :, hs, :D] = o
                part[r, :, hs, D] = m
                part[r, :, hs, D + 1] = l
            if not nonempty.any():
                continue
            M = m[nonempty].max(axis=0)                    # [per]
            w = np.exp(m[nonempty] - M[None, :])           # [nne, per]
            L = (w * l[nonempty]).sum(axis=0)
            O = (w[..., None] * o[nonempty]).sum(axis=0)
            out[r, hs] = O / L[:, None]
        if gate is not None:
            with np.errstate(over="ignore"):                # exp(+huge) = inf gives the closed gate 0
                out[r] *= 1.0 / (1.0 + np.exp(-np.asarray(gate[t], dtype=np.float64)))
    return out, out.astype(np.float16), part, bad


# ---------------------------------------------------------------------------
# Selection: scores -> ids  (argon_r36_qsa "Summary & Decision" buffer list:
# scores, ids, pooled; sol_r5_mtp_qsa "mtp attention": the decode window of
# 64 sink + 256 previous local + 1 current cell)
# ---------------------------------------------------------------------------

def select_ids(scores: np.ndarray, pos0: int, width: int = 2048, budget: int = 2048,
               sink: int = 64, local: int = 256):
    """Per token t (position p = pos0 + t), the ids its attention reads.

    Reading (the pages name the scores -> ids step and its buffers but never
    define it): the forced cells of the decode window -- sink cells
    0 .. min(sink, p)-1, the previous `local` cells and the token's own cell
    p -- plus the highest-scoring other causal cells c <= p, ties going to the
    lower id, until min(p + 1, budget) cells are chosen; ascending, then -1 up
    to `width`.  `scores` is [T, >= pos0 + T] (row t holds cells 0..p); the
    decision is taken in the scores' own precision (float32).
    """
    T = scores.shape[0]
    out = np.full((T, width), -1, dtype=np.int32)
    for t in range(T):
        p = pos0 + t
        n = p + 1
        k = min(n, budget)
        forced = np.zeros(n, dtype=bool)
        forced[: min(sink, n)] = True
        forced[max(sink, p - local): p] = True
        forced[p] = True
        nf = int(forced.sum())
        chosen = forced.copy()
        if k > nf:
            free = np.nonzero(~forced)[0]
            s = scores[t, free].astype(np.float32)
            order = np.lexsort((free, -s.astype(np.float64)))   # score descending, then id ascending
            chosen[free[order[: k - nf]]] = True
        ids = np.nonzero(chosen)[0]
        out[t, : len(ids)] = ids
    return out
