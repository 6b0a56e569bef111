"""Pins of the CPU oracle against facts that do not come from the oracle itself:
hand-derived values, closed forms, invariants and library routines.

The pages print no worked values, so every pin here is one of: arithmetic done by
hand from the quantiser's definition, a closed form of the normalisation /
rotation / attention formulas, an invariant the method guarantees (rotation
composition, chunked == unchunked softmax, padding and permutation
invariance), or a special case that reduces to a library routine (numpy matmul
for dequantised scores, torch's scaled_dot_product_attention for dense causal
attention).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention, prep_queries, quantize_rows, score, score_abs_bound
from sparse_selected_attention_gb300 import workloads as wl

# ----------------------------------------------------------------------------
# quantiser
# ----------------------------------------------------------------------------


def _group(vals, n=32):
    g = np.zeros(n, dtype=np.float32)
    g[: len(vals)] = vals
    return g


def test_quantize_unit_scale_rounds_half_to_even():
    # amax = 127 -> 127/127 = 1.0 exactly -> fp16 1.0; codes are rint(x) with
    # ties to even, then the clamp.
    x = _group([127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -127.0, 126.5, -0.5, 0.49999997])
    codes, scales = quantize_rows(x[None, :])
    assert scales.dtype == np.float16 and float(scales[0, 0]) == 1.0
    assert codes[0, :11].tolist() == [127, 2, 4, -2, -4, 0, 2, -127, 126, 0, 0]
    assert not codes[0, 11:].any()


def test_quantize_scale_is_fp16_of_fp32_quotient_and_divides_by_stored_scale():
    # amax = 1: 1/127 = 0.0078740157..., between 2^-7 and 2^-6; the fp16
    # significand is round(1.0078740 * 1024) = 1032 -> scale = 1032 * 2^-17
    # = 0.00787353515625 (bits 0x2008).
    s = 1032 * 2.0 ** -17
    x = _group([1.0,
                516 * 2.0 ** -17,     # x / s = 0.5 exactly -> 0 (tie to even)
                1548 * 2.0 ** -17,    # x / s = 1.5 exactly -> 2
                -0.25,                # -31.7505... -> -32
                0.79132])             # / stored scale = 100.5038 -> 101
                                      # (/ unrounded 1/127 would be 100.4976 -> 100)
    codes, scales = quantize_rows(x[None, :])
    assert int(scales.view(np.uint16)[0, 0]) == 0x2008
    assert float(scales[0, 0]) == s
    assert codes[0, :5].tolist() == [127, 0, 2, -32, 101]


def test_quantize_zero_group_and_subnormal_scale():
    x = np.zeros((1, 128), dtype=np.float32)
    # group 1: amax = 127 * 2^-20 -> scale 2^-20 (an fp16 subnormal, exact).
    x[0, 32] = 127 * 2.0 ** -20
    x[0, 33] = 3.5 * 2.0 ** -20      # -> 4
    x[0, 34] = -2.5 * 2.0 ** -20     # -> -2
    # group 2: a negative maximum maps to -127.
    x[0, 64] = -3.0
    x[0, 65] = 1.5                   # 1.5 / fp16(3/127) -> 63.5... -> 64 (see below)
    codes, scales = quantize_rows(x)
    assert float(scales[0, 0]) == 0.0 and not codes[0, :32].any()
    assert float(scales[0, 1]) == 2.0 ** -20
    assert codes[0, 32:35].tolist() == [127, 4, -2]
    assert codes[0, 64] == -127
    # 3/127 = 0.0236220..., fp16 significand round(1.511811 * 1024) = 1548
    # -> 1548 * 2^-16 = 0.02362060546875; 1.5 / that = 63.5039 -> 64.
    assert float(scales[0, 2]) == 1548 * 2.0 ** -16
    assert codes[0, 65] == 64
    assert float(scales[0, 3]) == 0.0


def test_quantize_invariants_random():
    x = (wl.normal(11, 1, (257, 128)) * wl.uniform(11, 2, (257, 1), 1e-3, 30.0)).astype(np.float32)
    codes, scales = quantize_rows(x)
    assert codes.dtype == np.int8 and codes.min() >= -127 and codes.max() <= 127
    sf = np.repeat(scales.astype(np.float64), 32, axis=1)
    err = np.abs(x.astype(np.float64) - codes.astype(np.float64) * sf)
    # Round trip within half a step (plus the float32 quotient's rounding,
    # at most 127 * 2^-24 of a step).
    assert np.all(err <= sf * (0.5 + 1e-5))
    # Every group's largest magnitude maps to +-127: the fp16 scale is within
    # 2^-11 relative of amax/127, so amax/scale is within 0.07 of 127.
    xg = np.abs(x.reshape(257, 4, 32))
    cg = np.abs(codes.reshape(257, 4, 32).astype(np.int32))
    at_max = np.take_along_axis(cg, xg.argmax(-1)[..., None], -1)[..., 0]
    assert np.all(at_max == 127)


# ----------------------------------------------------------------------------
# query RMS-norm + rotation
# ----------------------------------------------------------------------------


def test_prep_constant_row_closed_form():
    c, eps = 0.37, 1e-6
    x = np.full((1, 1, 128), c, dtype=np.float32)
    g = wl.uniform(3, 1, (128,), 0.5, 1.5).astype(np.float32)
    y, _, _ = prep_queries(x, g, pos0=0, eps=eps)
    cf = float(np.float32(c))
    want = g.astype(np.float64) * cf / math.sqrt(cf * cf + eps)
    np.testing.assert_allclose(y[0, 0], want, rtol=1e-14)


@pytest.mark.parametrize("p", [1, 2, 3, 1000, 31983])
def test_prep_one_hot_rotates_by_position(p):
    # x = e_0 (or e_1, e_100), g = 1, eps = 0 -> rs * x = sqrt(128) e_i.
    g = np.ones(128, dtype=np.float32)
    for i, f in ((0, 1.0), (1, float(np.float32(10000.0 ** (-2.0 / 64))))):
        x = np.zeros((1, 1, 128), dtype=np.float32)
        x[0, 0, i] = 1.0
        y, _, _ = prep_queries(x, g, pos0=p, eps=0.0)
        r = math.sqrt(128.0)
        want = np.zeros(128)
        want[i] = r * math.cos(p * f)
        want[i + 32] = r * math.sin(p * f)
        np.testing.assert_allclose(y[0, 0], want, atol=1e-12)
    x = np.zeros((1, 1, 128), dtype=np.float32)
    x[0, 0, 100] = 1.0
    y, _, _ = prep_queries(x, g, pos0=p, eps=0.0)
    want = np.zeros(128)
    want[100] = math.sqrt(128.0)
    np.testing.assert_allclose(y[0, 0], want, atol=1e-12)


def test_prep_rotation_preserves_pair_norms_and_composes():
    inp = wl.prep_inputs(3, seed=9)
    ones = np.ones(128, dtype=np.float32)
    y0, _, _ = prep_queries(inp.q_in, inp.norm_w, pos0=0)
    y1, _, _ = prep_queries(inp.q_in, inp.norm_w, pos0=12345)
    n0 = y0[..., :32] ** 2 + y0[..., 32:64] ** 2
    n1 = y1[..., :32] ** 2 + y1[..., 32:64] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-12)
    np.testing.assert_array_equal(y1[..., 64:], y0[..., 64:])
    # With g = 1 and eps = 0 the normalised row has unit RMS, so normalising
    # again is the identity and rotations by p1 then p2 equal one by p1 + p2.
    a, _, _ = prep_queries(inp.q_in, ones, pos0=700, eps=0.0)
    b, _, _ = prep_queries(a.astype(np.float32), ones, pos0=2100, eps=0.0)
    c, _, _ = prep_queries(inp.q_in, ones, pos0=2800, eps=0.0)
    # Token t is at position pos0 + t in each call, so compare token 0 only.
    np.testing.assert_allclose(b[0], c[0], atol=2e-6)


# ----------------------------------------------------------------------------
# score
# ----------------------------------------------------------------------------


def test_score_one_hot_query_closed_form():
    cache = wl.make_cache(300, seed=4)
    q = np.zeros((2, 12, 128), dtype=np.float32)
    q[0, 7, 77] = 1.0           # group 2
    q[1, 0, 5] = -2.0           # group 0
    S = score(q, cache.kq, cache.ksc, pos0=250)
    c = np.arange(251)
    np.testing.assert_array_equal(S[0, :251], cache.ksc[c, 2].astype(np.float64) * cache.kq[c, 77])
    np.testing.assert_array_equal(S[1, :252], -2.0 * cache.ksc[:252, 0].astype(np.float64) * cache.kq[:252, 5])
    assert np.all(np.isnan(S[0, 251:])) and np.all(np.isnan(S[1, 252:]))


def test_score_equals_dense_matmul_on_dequantised_keys_and_is_head_linear():
    cache = wl.make_cache(400, seed=6)
    cache.ksc[17] = 0                               # a dead key row
    q = wl.queries_f32(40, seed=6)
    S = score(q, cache.kq, cache.ksc, pos0=360)
    kdq = cache.kq.astype(np.float64) * np.repeat(cache.ksc.astype(np.float64), 32, axis=1)
    dense = q.astype(np.float64).sum(axis=1) @ kdq.T
    causal = np.arange(400)[None, :] <= (360 + np.arange(40))[:, None]
    np.testing.assert_allclose(S[causal], dense[causal], rtol=1e-12, atol=1e-12)
    assert np.all(S[:, 17] == 0.0)
    # All heads equal -> 12x the one-head score.
    q1 = np.repeat(q[:, :1], 12, axis=1)
    S12 = score(q1, cache.kq, cache.ksc, pos0=360)
    S1 = score(q[:, :1], cache.kq, cache.ksc, pos0=360)
    np.testing.assert_allclose(S12[causal], 12.0 * S1[causal], rtol=1e-12, atol=1e-12)
    A = score_abs_bound(q, cache.kq, cache.ksc, pos0=360)
    assert np.all(np.abs(S[causal]) <= A[causal] * (1 + 1e-12))


# ----------------------------------------------------------------------------
# attention
# ----------------------------------------------------------------------------

SCALE = 1.0 / math.sqrt(128.0)


def _dequant(cache):
    k = cache.kq.astype(np.float64) * np.repeat(cache.ksc.astype(np.float64), 32, axis=1)
    v = cache.vq.astype(np.float64) * np.repeat(cache.vsc.astype(np.float64), 32, axis=1)
    return k, v


def _softmax_attn(q, k, v, cells, weights=None):
    """Textbook single softmax over the listed cells (float64)."""
    s = SCALE * (q.astype(np.float64) @ k[cells].T)            # [H, n]
    s = s - s.max(axis=1, keepdims=True)
    e = np.exp(s) * (1.0 if weights is None else weights[None, :])
    return (e @ v[cells]) / e.sum(axis=1, keepdims=True)


def test_attention_width_one_is_the_dequantised_value_row():
    cache = wl.make_cache(50, seed=2)
    q = wl.queries_f16(3, seed=2)
    ids = np.full((3, 64), -1, dtype=np.int32)
    ids[0, 0], ids[1, 63], ids[2, 17] = 5, 49, 0
    out64, out16, _, bad = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    _, v = _dequant(cache)
    for t, c in enumerate([5, 49, 0]):
        np.testing.assert_array_equal(out64[t], np.broadcast_to(v[c], (12, 128)))
        np.testing.assert_array_equal(out16[t], np.broadcast_to(v[c], (12, 128)).astype(np.float16))
    assert not bad


def test_attention_equal_scores_give_the_plain_mean():
    cache = wl.make_cache(700, seed=8)
    q = np.zeros((2, 12, 128), dtype=np.float16)
    q[1] = np.float16(-0.0)
    ids = wl.even_ids(2, 698, width=704, select=650)
    out64, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    _, v = _dequant(cache)
    for t in range(2):
        cells = ids[t][ids[t] >= 0]
        np.testing.assert_allclose(out64[t], np.broadcast_to(v[cells].mean(axis=0), (12, 128)), rtol=1e-12, atol=1e-15)


def test_attention_contiguous_ids_equal_dense_causal_sdpa():
    T, pos0 = 70, 100
    cache = wl.make_cache(pos0 + T, seed=12)
    q = wl.queries_f16(T, seed=12)
    ids = wl.even_ids(T, pos0, width=192, select=4096)   # all cells 0..p
    out64, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    k, v = _dequant(cache)
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]       # [1, H, T, D]
    K = torch.from_numpy(k)[None, None].expand(1, 12, -1, -1)
    V = torch.from_numpy(v)[None, None].expand(1, 12, -1, -1)
    mask = torch.arange(pos0 + T)[None, :] <= (pos0 + torch.arange(T))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=SCALE)
    np.testing.assert_allclose(out64, ref[0].permute(1, 0, 2).numpy(), rtol=1e-11, atol=1e-14)


def test_attention_chunked_merge_equals_single_softmax_for_arbitrary_ids():
    cache = wl.make_cache(5000, seed=13)
    q = wl.queries_f16(6, seed=13)
    k, v = _dequant(cache)
    rng = np.random.default_rng(13)
    ids = np.full((6, 448), -1, dtype=np.int32)
    for t in range(6):
        n = int(rng.integers(1, 448))
        ids[t, :n] = rng.choice(5000, size=n, replace=False)
    out64, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    for t in range(6):
        cells = ids[t][ids[t] >= 0]
        np.testing.assert_allclose(out64[t], _softmax_attn(q[t], k, v, cells), rtol=1e-11, atol=1e-14)


def test_attention_padding_permutation_and_duplication():
    cache = wl.make_cache(3000, seed=14)
    q = wl.queries_f16(1, seed=14)
    k, v = _dequant(cache)
    base = np.full((1, 320), -1, dtype=np.int32)
    cells = np.arange(2, 3000, 11)[:250].astype(np.int32)
    base[0, :250] = cells
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, base, SCALE)
    # -1 slots inserted anywhere (whole chunks too) leave the result unchanged.
    padded = np.full((1, 640), -1, dtype=np.int32)
    pos = np.sort(np.random.default_rng(1).choice(np.arange(64, 640), size=250, replace=False))
    padded[0, pos] = cells
    out, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, padded, SCALE)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
    # A permutation of the list changes nothing.
    perm = base.copy()
    perm[0, :250] = np.random.default_rng(2).permutation(cells)
    out, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, perm, SCALE)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-15)
    # A duplicated id counts twice: softmax with weight 2 on that cell.
    dup = base.copy()
    dup[0, 250] = cells[40]
    out, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, dup, SCALE)
    w = np.ones(250)
    w[40] = 2.0
    np.testing.assert_allclose(out[0], _softmax_attn(q[0], k, v, cells, w), rtol=1e-11, atol=1e-14)


def test_attention_part_and_empty_and_bad_ids():
    cache = wl.make_cache(200, seed=15)
    q = wl.queries_f16(3, seed=15)
    ids = np.full((3, 128), -1, dtype=np.int32)
    ids[0, :64] = np.arange(64)            # one full chunk, second chunk empty
    ids[2, 70] = 500                        # out of range -> padding + flag
    ids[2, 71] = -7                         # below -1 -> padding + flag
    ids[2, 72] = 3
    out64, out16, part, bad = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE, want_part=True)
    assert bad
    assert np.all(out16[1] == 0) and not np.signbit(out16[1]).any()
    k, v = _dequant(cache)
    s = SCALE * (q[0].astype(np.float64) @ k[:64].T)
    np.testing.assert_allclose(part[0, 0, :, 128], s.max(axis=1), rtol=1e-13)
    np.testing.assert_allclose(part[0, 0, :, :128] / part[0, 0, :, 129:130], out64[0], rtol=1e-12)
    assert np.all(part[0, 1, :, 128] == -np.inf) and np.all(part[0, 1, :, 129] == 0)
    _, vv = _dequant(cache)
    np.testing.assert_array_equal(out64[2], np.broadcast_to(vv[3], (12, 128)))


# ----------------------------------------------------------------------------
# selection
# ----------------------------------------------------------------------------

from oracle import select_ids  # noqa: E402


def test_select_short_context_takes_every_causal_cell():
    sc = wl.uniform(3, 9, (5, 2100), -1, 1).astype(np.float32)
    ids = select_ids(sc, pos0=10, width=2048)
    for t in range(5):
        p = 10 + t
        assert np.array_equal(ids[t, : p + 1], np.arange(p + 1)) and np.all(ids[t, p + 1:] == -1)


def test_select_hand_built_row():
    # budget 6 with sink 2 and local 1: p = 9 forces {0, 1, 8, 9}; the two free
    # slots go to the best of cells 2..7 by score, ties to the lower id.
    sc = np.zeros((1, 10), dtype=np.float32)
    sc[0, 2:8] = [0.5, 3.0, 3.0, -1.0, 3.0, 2.0]     # cells 3, 4, 6 tie at 3.0
    sc[0, 8] = -100.0                                # forced cells ignore their score
    ids = select_ids(sc, pos0=9, width=8, budget=6, sink=2, local=1)
    assert ids[0].tolist() == [0, 1, 3, 4, 8, 9, -1, -1]


def test_select_invariants_random():
    T, pos0 = 9, 3000
    sc = wl.normal(4, 10, (T, pos0 + T)).astype(np.float32)
    sc[:, ::97] = 1.5                                # plenty of ties
    ids = select_ids(sc, pos0, width=2048)
    for t in range(T):
        p = pos0 + t
        row = ids[t][ids[t] >= 0]
        assert len(row) == 2048 and np.all(np.diff(row) > 0) and row[-1] == p and row.max() <= p
        forced = set(range(64)) | set(range(p - 256, p + 1))
        assert forced <= set(row.tolist())
        free_sel = np.array(sorted(set(row.tolist()) - forced))
        unsel = np.array(sorted(set(range(p + 1)) - set(row.tolist())))
        # every selected free cell outranks every unselected cell
        worst = min(free_sel, key=lambda c: (sc[t, c], -c))
        best_out = max(unsel, key=lambda c: (sc[t, c], -c))
        assert (sc[t, worst], -worst) > (sc[t, best_out], -best_out)


def test_select_signed_zeros_tie():
    # -0.0 and +0.0 are the same score: the lower id wins, whatever the sign.
    sc = np.full((1, 8), -1.0, dtype=np.float32)
    sc[0, 2], sc[0, 3], sc[0, 4] = 0.0, -0.0, 0.0
    ids = select_ids(sc, pos0=7, width=8, budget=4, sink=1, local=0)
    assert ids[0].tolist() == [0, 2, 3, 7, -1, -1, -1, -1]


def test_select_nan_ranks_last():
    # A NaN score is no score: every number, -inf included, outranks it, and
    # NaNs tie with each other (the lower id wins).  p = 9 with sink 1 and
    # local 0 forces {0, 9}; budget 7 leaves five free slots among cells 1..8.
    sc = np.zeros((1, 10), dtype=np.float32)
    sc[0, 1:9] = [np.nan, -np.inf, np.nan, 1.0, np.nan, np.inf, -np.nan, -2.0]
    with np.errstate(invalid="ignore"):
        ids = select_ids(sc, pos0=9, width=8, budget=7, sink=1, local=0)
    # free ranking: 6 (+inf), 4 (1.0), 8 (-2.0), 2 (-inf), then NaNs 1, 3, 5, 7
    assert ids[0].tolist() == [0, 1, 2, 4, 6, 8, 9, -1]


# ----------------------------------------------------------------------------
# attention: output gate and several KV heads
# ----------------------------------------------------------------------------

def test_attention_gate_zero_halves_the_output_exactly():
    cache = wl.make_cache(400, seed=31)
    q = wl.queries_f16(3, seed=31)
    ids = wl.even_ids(3, 390, width=256, select=256)
    plain, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    gated, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE,
                               gate=np.zeros((3, 12, 128), np.float32))
    assert np.array_equal(gated, plain * 0.5)


def test_attention_gate_applies_per_head_and_dim():
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4; the pattern varies along
    # both the head and the dim axis, so a transposed or per-head gate fails.
    cache = wl.make_cache(300, seed=32)
    q = wl.queries_f16(2, seed=32)
    ids = wl.even_ids(2, 290, width=128, select=128)
    h, d = np.meshgrid(np.arange(12), np.arange(128), indexing="ij")
    code = (h + 2 * d) % 3                                   # 0, 1, 2
    gate = np.where(code == 0, 0.0, np.where(code == 1, np.log(3.0), -np.log(3.0)))
    factor = np.where(code == 0, 0.5, np.where(code == 1, 0.75, 0.25))
    plain, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE)
    gated, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE,
                               gate=np.broadcast_to(gate, (2, 12, 128)))
    np.testing.assert_allclose(gated, plain * factor[None], rtol=1e-14, atol=0)


def test_attention_two_kv_heads_equal_grouped_sdpa():
    # The pages' shape: 2 KV heads, 12 query heads each, d = 256, per-64
    # scales.  Contiguous causal ids reduce it to dense causal attention with
    # grouped KV heads, which torch computes with enable_gqa.
    T, pos0 = 20, 60
    H, Hkv, D, grp = wl.PAGES_Q_HEADS, wl.PAGES_KV_HEADS, wl.PAGES_HEAD_DIM, wl.PAGES_GROUP
    cache = wl.make_cache(pos0 + T, seed=33, head_dim=D, group=grp, kv_heads=Hkv)
    q = wl.queries_f16(T, seed=33, heads=H, head_dim=D)
    ids = wl.even_ids(T, pos0, width=128, select=4096)
    out64, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, wl.PAGES_SCALE, group=grp)
    k = cache.kq.astype(np.float64) * np.repeat(cache.ksc.astype(np.float64), grp, axis=-1)   # [C, Hkv, D]
    v = cache.vq.astype(np.float64) * np.repeat(cache.vsc.astype(np.float64), grp, axis=-1)
    Q = torch.from_numpy(q.astype(np.float64)).permute(1, 0, 2)[None]      # [1, H, T, D]
    K = torch.from_numpy(k).permute(1, 0, 2)[None]                          # [1, Hkv, C, D]
    V = torch.from_numpy(v).permute(1, 0, 2)[None]
    mask = torch.arange(pos0 + T)[None, :] <= (pos0 + torch.arange(T))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=wl.PAGES_SCALE,
                                                           enable_gqa=True)
    np.testing.assert_allclose(out64, ref[0].permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-13)


def test_attention_kv_head_slices_are_independent():
    # Changing KV head 1's rows changes only query heads 12..23.
    T, pos0, D, grp = 3, 200, 256, 64
    cache = wl.make_cache(pos0 + T, seed=34, head_dim=D, group=grp, kv_heads=2)
    q = wl.queries_f16(T, seed=34, heads=24, head_dim=D)
    ids = wl.even_ids(T, pos0, width=128, select=128)
    a, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 0.0625, group=grp)
    vq2 = cache.vq.copy()
    vq2[:, 1] = -vq2[:, 1]
    b, _, _, _ = attention(q, cache.kq, vq2, cache.ksc, cache.vsc, ids, 0.0625, group=grp)
    assert np.array_equal(a[:, :12], b[:, :12])
    np.testing.assert_allclose(b[:, 12:], -a[:, 12:], rtol=1e-12, atol=1e-15)


# ----------------------------------------------------------------------------
# prep: optional key rotation
# ----------------------------------------------------------------------------

from oracle import prep as _prep, rotate_keys_f32  # noqa: E402


def _prep_cache(T, pos0, seed, rope_k):
    inp = wl.prep_inputs(T, seed=seed)
    c = wl.make_cache(pos0 + T, seed=seed)
    _prep(inp.q_in, inp.k_in, inp.v_in, inp.norm_w, pos0, c.kq, c.vq, c.ksc, c.vsc, rope_k=rope_k)
    return inp, c


def test_rope_k_at_position_zero_is_the_plain_quantiser():
    inp, a = _prep_cache(1, 0, 61, rope_k=True)
    _, b = _prep_cache(1, 0, 61, rope_k=False)
    assert np.array_equal(a.kq, b.kq) and np.array_equal(a.ksc.view(np.uint16), b.ksc.view(np.uint16))
    assert np.array_equal(a.vq, b.vq)


def test_rope_k_one_hot_row():
    # k = A e_i (i < 32) at position p rotates to A cos(p f_i) at dim i and
    # A sin(p f_i) at dim i + 32; each is alone in its 32-dim group, so both
    # quantise to +-127 with scale fp16(|A cos| / 127), fp16(|A sin| / 127).
    p, i, A = 977, 5, 3.0
    k = np.zeros((1, 1, 128), np.float32)
    k[0, 0, i] = A
    r = rotate_keys_f32(k, p)
    ang = p * float(np.float32(10000.0 ** (-2 * i / 64)))
    assert r[0, 0, i] == np.float32(A) * np.float32(np.cos(ang))
    assert r[0, 0, i + 32] == np.float32(A) * np.float32(np.sin(ang))
    assert np.count_nonzero(r) == 2
    codes, scales = wl_quant(r)
    assert codes[0, 0, i] == 127 * np.sign(np.cos(ang)) and codes[0, 0, i + 32] == 127 * np.sign(np.sin(ang))
    assert scales[0, 0, 0] == np.float16(np.float32(abs(A * np.cos(ang))) / np.float32(127))
    assert np.count_nonzero(codes) == 2


def wl_quant(x):
    from oracle import quantize_rows
    return quantize_rows(x)


def test_rope_k_rotation_preserves_pair_norms_and_composes():
    k = wl.prep_inputs(4, seed=62).k_in
    r = rotate_keys_f32(k, 1234).astype(np.float64)
    k64 = k.astype(np.float64)
    n0 = k64[..., :32] ** 2 + k64[..., 32:64] ** 2
    n1 = r[..., :32] ** 2 + r[..., 32:64] ** 2
    np.testing.assert_allclose(n1, n0, rtol=2e-6)
    assert np.array_equal(r[..., 64:], k64[..., 64:])
    # rotating by p1 then p2 is rotating by p1 + p2 (one token: its position is pos0)
    k1 = k[:1]
    two = rotate_keys_f32(rotate_keys_f32(k1, 300), 700).astype(np.float64)
    np.testing.assert_allclose(two, rotate_keys_f32(k1, 1000).astype(np.float64), atol=2e-5)
