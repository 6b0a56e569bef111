"""qsa_select on the GPU against the oracle's select_ids on the same fp32
scores (the selection is decided in the scores' precision, so ids must match
bit for bit), including heavy ties and short contexts; and the pipeline
score -> select -> attention, where the oracle runs the chain from the same
inputs on its own scores."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, score, score_abs_bound, select_ids
from sparse_selected_attention_gb300 import (qsa_attn, qsa_score, qsa_score_workspace_bytes, qsa_select)
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import assert_f16_close, assert_score_close, assert_valid_selection, dev

pytestmark = pytest.mark.gpu


def run(scores, pos0, width=2048, budget=2048, sink=64, local=256):
    T = scores.shape[0]
    ids = torch.full((T, width), -7, dtype=torch.int32, device="cuda")
    qsa_select(dev(scores), pos0, ids, budget=budget, sink=sink, local=local)
    torch.cuda.synchronize()
    return ids.cpu().numpy()


@pytest.mark.parametrize("T,pos0", [(64, 30000), (300, 2000), (8, 31970)])
def test_select_matches_oracle_random(cuda_device, T, pos0):
    sc = wl.normal(70, 1, (T, pos0 + T)).astype(np.float32)
    got = run(sc, pos0)
    assert np.array_equal(got, select_ids(sc, pos0))


def test_select_full_size_all_rows(cuda_device):
    T, pos0 = 1984, 30000
    sc = wl.normal(71, 1, (T, pos0 + T)).astype(np.float32)
    got = run(sc, pos0)
    bad = [t for t in range(T) if not np.array_equal(got[t], select_ids(sc[t:t + 1], pos0 + t)[0])]
    assert not bad, f"{len(bad)} rows differ, first {bad[:5]}"


def test_select_on_score_kernel_output_full_size(cuda_device):
    """The bench's selection workload: qsa_score's own fp32 scores of 1984
    tokens at pos0 30000 (fp32 queries N(0,1), the seed-5 key cache), then
    qsa_select over them in one call; every row against select_ids on the
    same scores."""
    T, pos0 = 1984, 30000
    C = pos0 + T
    cache = wl.make_cache(C, seed=5)
    sc = torch.empty((T, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    qsa_score(dev(wl.queries_f32(T, seed=5)), dev(cache.kq), dev(cache.ksc), pos0, sc, ws)
    ids = torch.full((T, 2048), -7, dtype=torch.int32, device="cuda")
    qsa_select(sc, pos0, ids)
    torch.cuda.synchronize()
    got, host = ids.cpu().numpy(), sc.cpu().numpy()
    bad = [t for t in range(T) if not np.array_equal(got[t], select_ids(host[t:t + 1], pos0 + t)[0])]
    assert not bad, f"{len(bad)} rows differ, first {bad[:5]}"


def test_select_sample_misses_the_threshold(cuda_device):
    """Rows where every score inside 32 evenly spread runs of 32 cells is far
    below all others: a selection that estimated its threshold from such a
    sample would miss it.  Ids must equal the oracle's."""
    T, pos0, sink, local = 6, 20000, 64, 256
    sc = wl.normal(78, 1, (T, pos0 + T)).astype(np.float32)
    for t in range(T):
        p = pos0 + t
        fs, fe = sink, p - local
        nfree = fe - fs
        for k in range(32):
            start = fs + k * (nfree - 32) // 31
            sc[t, start:start + 32] = -50.0 - k
    assert np.array_equal(run(sc, pos0), select_ids(sc, pos0))


def test_select_heavy_ties(cuda_device):
    T, pos0 = 40, 6000
    sc = np.round(wl.normal(72, 1, (T, pos0 + T)) * 2) / 2      # few distinct values
    sc = sc.astype(np.float32)
    sc[:, 100:3000] = 0.5                                          # a wide plateau
    sc[:, 3000:3200:2] = -0.0                                      # signed zeros tie with +0
    sc[:, 3001:3200:2] = 0.0
    assert np.array_equal(run(sc, pos0), select_ids(sc, pos0))


def test_select_short_rows_and_window_only(cuda_device):
    sc = wl.normal(73, 1, (50, 2100)).astype(np.float32)
    assert np.array_equal(run(sc, 100), select_ids(sc, 100))        # n <= budget: every cell
    sc2 = wl.normal(74, 1, (6, 4100)).astype(np.float32)
    got = run(sc2, 4094, width=384, budget=321)                       # forced window only
    assert np.array_equal(got, select_ids(sc2, 4094, width=384, budget=321))


def test_score_select_attention_pipeline(cuda_device):
    """score -> select -> attention with every stage on the GPU.  The oracle
    runs the same chain from the same inputs (float64 scores, selection on
    their fp32 rounding); rows whose ids match are compared on the output,
    rows that differ must be a valid selection within the score bound."""
    T, pos0 = 96, 9000
    C = pos0 + T
    cache = wl.make_cache(C, seed=75)
    q32 = wl.queries_f32(T, seed=75)
    q16 = q32.astype(np.float16)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    scores = torch.empty((T, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    qsa_score(dev(q32), kq, ksc, pos0, scores, ws)
    ids = torch.empty((T, 2048), dtype=torch.int32, device="cuda")
    qsa_select(scores, pos0, ids)
    out = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    qsa_attn(dev(q16), kq, vq, ksc, vsc, ids, out)
    torch.cuda.synchronize()
    q64 = q32.astype(np.float64)
    S = score(q64, cache.kq, cache.ksc, pos0)
    A = score_abs_bound(q64, cache.kq, cache.ksc, pos0)
    assert_score_close(scores.cpu().numpy(), S, A, "pipeline scores")
    ref_ids = select_ids(np.where(np.isnan(S), 0.0, S).astype(np.float32), pos0)
    got = ids.cpu().numpy()
    differ = assert_valid_selection(got, ref_ids, S, A, pos0, what="pipeline selection")
    assert len(differ) <= T // 8, f"{len(differ)} of {T} rows chose differently"
    same = np.setdiff1d(np.arange(T), differ)
    o64, _, _, _ = attention(q16, cache.kq, cache.vq, cache.ksc, cache.vsc, ref_ids, 1 / math.sqrt(128))
    assert_f16_close(out.cpu()[same], o64[same], "score -> select -> attention")


@pytest.mark.parametrize("kind", ["all_equal", "outlier", "inf_range", "tiny_range", "two_plateaus", "mid_plateau"])
def test_select_degenerate_rows(cuda_device, kind):
    """Rows whose scores crowd into few values: plateaus at and around the
    threshold, extreme outliers and spans a few ulps wide."""
    T, pos0 = 12, 5000
    sc = wl.normal(76, 1, (T, pos0 + T)).astype(np.float32)
    if kind == "all_equal":
        sc[:] = 1.25
    elif kind == "outlier":
        sc[:, 777] = 3e38
    elif kind == "inf_range":
        sc[:, 777] = 3e38                    # max - min overflows fp32
        sc[:, 1234] = -3e38
    elif kind == "tiny_range":
        sc = (1.0 + np.round(sc * 4) * np.float32(2 ** -23)).astype(np.float32)  # a handful of ulps apart
    elif kind == "mid_plateau":
        sc[:, 1000:1800] = np.float32(0.33)  # ~800 ties straddling the threshold
    else:
        sc[:, :] = -2.0
        sc[:, 200:2500] = 7.0                # more cells at 7.0 than the budget leaves free
    assert np.array_equal(run(sc, pos0), select_ids(sc, pos0))


@pytest.mark.parametrize("kind", ["small_head", "huge_head", "negative", "negative_tiny"])
def test_select_rows_far_from_their_first_cells(cuda_device, kind):
    """Rows whose leading cells say little about the threshold: the first
    9000 cells far smaller (or far larger) than the rest, and rows of
    negative scores only.  A selection that sizes its first histogram from
    the leading cells must still find the exact threshold."""
    T, pos0 = 6, 20000
    sc = wl.normal(78, 1, (T, pos0 + T)).astype(np.float32)
    if kind == "small_head":
        sc[:, :9000] *= np.float32(1e-6)
    elif kind == "huge_head":
        sc[:, :9000] *= np.float32(1e12)
    elif kind == "negative":
        sc = -np.abs(sc) - np.float32(1.0)
    else:
        # Negative scores near -1e-37 whose largest order key has top digit
        # 2015 (0x7df), so a 256-digit window reaching 32 digits above it ends
        # just below +0; 500 zeros of both signs after the leading cells rank
        # above every one of them.
        v = np.array([~np.uint32((2015 << 20) | 0xFFFFF)], dtype=np.uint32).view(np.float32)[0]
        sc = (v * (np.float32(1.0) + np.abs(sc))).astype(np.float32)
        sc[:, 100] = v
        sc[:, 12000:12500] = np.float32(0.0)
        sc[:, 12000:12500:2] = np.float32(-0.0)
    assert np.array_equal(run(sc, pos0), select_ids(sc, pos0))


def test_select_nan_and_infinite_scores(cuda_device):
    """NaN scores (either sign, any payload) rank below every number, -inf
    included, with ties among them going to the lower id; +inf ranks first."""
    T, pos0 = 8, 5000
    sc = wl.normal(79, 1, (T, pos0 + T)).astype(np.float32)
    bits = sc.view(np.uint32)
    bits[0, 100:4000] = 0x7FC00000                    # most of row 0 is NaN
    bits[1, 100:4000:2] = 0xFFC00001                  # negative NaN with a payload
    bits[1, 101:4000:2] = 0x7F800001                  # signalling NaN
    sc[2, 300:700] = np.float32(np.inf)
    sc[2, 700:4900] = np.float32(-np.inf)
    bits[2, 900:1200] = 0x7FC00000
    sc[3, :] = np.float32(-np.inf)
    bits[3, 2000:2100] = 0xFFFFFFFF
    bits[4, 64:4700:3] = 0x7FC00000                   # every third free cell NaN
    got = run(sc, pos0)
    with np.errstate(invalid="ignore"):  # the signalling NaNs, widened to float64
        ref = select_ids(sc, pos0)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("sink,local,budget", [(64, 256, 2048), (0, 5, 1000), (3, 0, 777)])
def test_select_misaligned_rows(cuda_device, sink, local, budget):
    """An odd row stride puts row starts at every offset modulo 16 bytes."""
    T, pos0 = 16, 7001
    sc = wl.normal(77, 1, (T, pos0 + T)).astype(np.float32)
    assert sc.shape[1] % 2 == 1
    got = run(sc, pos0, budget=budget, sink=sink, local=local)
    assert np.array_equal(got, select_ids(sc, pos0, budget=budget, sink=sink, local=local))
