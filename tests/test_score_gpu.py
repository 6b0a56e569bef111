"""qsa_score on the GPU against the CPU oracle, through the C ABI.

Small shapes are compared on every causal cell; the full-size sweep (T =
1984 at pos0 0 / 2048 / 8192 / 30000, plus the pages' 2050 and 2052) on 128
seeded token rows each, plus the rows at every 128-token tile boundary.
Every non-causal element of the output must still hold the caller's sentinel
bit pattern, over the whole buffer.
"""
import numpy as np
import pytest
import torch

from oracle import score, score_abs_bound
from sparse_selected_attention_gb300 import qsa_score, qsa_score_workspace_bytes
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import SENTINEL_BITS, assert_score_close, dev

pytestmark = pytest.mark.gpu


def run_gpu(q, cache, pos0, ld=None, dtype=np.float32, max_ctas=0):
    T = q.shape[0]
    C = cache.cells
    ld = ld or pos0 + T
    qd = dev(q.astype(dtype))
    kq, ksc = dev(cache.kq), dev(cache.ksc)
    scores = torch.full((T, ld), 0, dtype=torch.int32, device="cuda").fill_(SENTINEL_BITS).view(torch.float32)
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qsa_score(qd, kq, ksc, pos0, scores, ws, err=err, max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    # Untouched cells keep the sentinel: checked on the device over the whole buffer.
    causal = torch.arange(ld, device="cuda")[None, :] <= (pos0 + torch.arange(T, device="cuda"))[:, None]
    bits = scores.view(torch.int32)
    assert bool(torch.all(bits[~causal] == SENTINEL_BITS))
    assert not bool(torch.any(bits[causal] == SENTINEL_BITS))
    return scores


def _compare(q, cache, pos0, scores, rows, what, q_used=None):
    qq = q if q_used is None else q_used
    ref = score(qq, cache.kq, cache.ksc, pos0, rows=rows)
    A = score_abs_bound(qq, cache.kq, cache.ksc, pos0, rows=rows)
    g = scores[torch.as_tensor(rows, device="cuda")].cpu().numpy()[:, : ref.shape[1]]
    return assert_score_close(g, ref, A, what)


@pytest.mark.parametrize("T,pos0", [(1, 0), (5, 0), (70, 0), (200, 100), (130, 2050), (64, 2052), (129, 127)])
@pytest.mark.parametrize("dtype", [np.float32, np.float16])
@pytest.mark.parametrize("row_align", [4, 16], ids=["rows4B", "rows16B"])
def test_small_all_cells(cuda_device, T, pos0, dtype, row_align):
    # Two row pitches: ld = pos0 + T + 5 (rows only 4-byte aligned) and ld
    # rounded up to a multiple of 4 floats (16-byte aligned rows).
    cache = wl.make_cache(pos0 + T, seed=31)
    dead = 3 if cache.cells > 3 else None
    if dead is not None:
        cache.ksc[dead] = 0     # a dead key: scores exactly 0
    q = wl.queries_f32(T, seed=31)
    ld = pos0 + T + 5 if row_align == 4 else -(-(pos0 + T + 5) // 4) * 4
    scores = run_gpu(q, cache, pos0, ld=ld, dtype=dtype)
    q_used = q.astype(dtype)
    _compare(q, cache, pos0, scores, np.arange(T), f"T={T} pos0={pos0} {dtype.__name__}", q_used)
    if dead is not None:
        rows = [t for t in range(T) if dead <= pos0 + t]
        assert torch.all(scores[rows, dead] == 0)


@pytest.mark.parametrize("pos0", sorted(set(wl.SCORE_POS0) | {1984, 2050, 2052}))
def test_full_size_sampled_rows(cuda_device, pos0):
    # The sweep's positions ("Round 36 Track C", 2. qsa_score_mm Loop
    # Unrolling: pos0 0 / 2048 / 8192 / 30000) and the pages' others
    # ("round 11 track b", score: valid negative result: 1984, 2050, 2052).
    T = wl.SCORE_NTOK
    cache = wl.make_cache(pos0 + T, seed=5)
    q = wl.queries_f32(T, seed=5)
    scores = run_gpu(q, cache, pos0)
    rng = np.random.default_rng(pos0)
    edges = {e for k in range(0, T + 1, 128) for e in (k - 1, k) if 0 <= e < T}
    rows = np.array(sorted(set(rng.choice(T, 128, replace=False).tolist()) | edges))
    _compare(q, cache, pos0, scores, rows, f"T=1984 pos0={pos0}")


# The rest of the pages' score matrix ("round 11 track b: qsa attention and
# score", score: valid negative result: T = 96 / 512 / 1024 / 1984 at pos0 =
# 0 / 1984 / 2050 / 2052 / 30000); T = 1984 is above.  Every causal cell of
# every row.
@pytest.mark.parametrize("T", [96, 512, 1024])
@pytest.mark.parametrize("pos0", [0, 1984, 2050, 2052, 30000])
def test_pages_score_matrix(cuda_device, T, pos0):
    cache = wl.make_cache(pos0 + T, seed=5)
    q = wl.queries_f32(T, seed=5)
    scores = run_gpu(q, cache, pos0)
    _compare(q, cache, pos0, scores, np.arange(T), f"T={T} pos0={pos0}")


@pytest.mark.parametrize("cap", [1, 3, 7, 40])
def test_cta_cap_gives_identical_scores(cuda_device, cap):
    # Every tile is computed the same way whichever CTA runs it, so capping the
    # persistent grid changes only who computes what, never a bit of the output.
    T, pos0 = 300, 2100
    cache = wl.make_cache(pos0 + T, seed=33)
    q = wl.queries_f32(T, seed=33)
    base = run_gpu(q, cache, pos0)
    capped = run_gpu(q, cache, pos0, max_ctas=cap)
    assert torch.equal(base.view(torch.int32), capped.view(torch.int32))
    _compare(q, cache, pos0, capped, np.array([0, 1, 127, 128, 299]), f"max_ctas={cap}")


@pytest.mark.parametrize("ratio", [1e2, 1e4, 3e5])
def test_mixed_group_scales(cuda_device, ratio):
    # The kernel folds each cell's four group scales into its codes under one
    # power of two per cell, set by the largest scale; a much smaller group
    # then sits low in fp16's range.  Cells here mix groups whose scales differ
    # by `ratio` (the quantiser's own scales are a group's amax / 127), and
    # some cells have a zero group or only their smallest group non-zero.
    T, pos0 = 96, 1000
    cache = wl.make_cache(pos0 + T, seed=35)
    s = cache.ksc.view(np.float16).astype(np.float32)
    s[:, 1] = s[:, 0] / ratio
    s[::3, 2] = 0.0
    s[1::5, 0] = 0.0
    s[1::5, 2:] = 0.0            # only group 1 (the small one) left
    cache.ksc[...] = s.astype(np.float16).view(cache.ksc.dtype)
    q = wl.queries_f32(T, seed=35)
    scores = run_gpu(q, cache, pos0)
    _compare(q, cache, pos0, scores, np.arange(T), f"group scale ratio {ratio:g}")


@pytest.mark.parametrize("mag", [1e-30, 1e-6, 1e-4, 3e-3, 1.0, 1e3, 1e6, 1e30])
def test_query_magnitudes(cuda_device, mag):
    # The head sum travels as an fp16 hi/lo pair under a per-token power of
    # two, so the 1e-4 A bound holds for query rows of any finite magnitude:
    # rows far below fp16's normal range and far above its maximum alike.
    T, pos0 = 70, 300
    cache = wl.make_cache(pos0 + T, seed=37)
    q = (wl.queries_f32(T, seed=37).astype(np.float64) * mag).astype(np.float32)
    scores = run_gpu(q, cache, pos0)
    assert bool(torch.isfinite(scores[0, : pos0 + 1]).all())
    _compare(q, cache, pos0, scores, np.arange(T), f"query magnitude {mag:g}")


def test_query_magnitudes_mixed_in_one_tile(cuda_device):
    # Tokens of very different magnitudes side by side in every 128-token
    # tile (each token has its own power of two), plus all-zero rows and rows
    # at the edges of the unscaled range.
    T, pos0 = 300, 700
    cache = wl.make_cache(pos0 + T, seed=39)
    mags = np.array([1.0, 1e4, 1e-4, 1e-30, 1e30, 0.0, 2e-2, 5e3, 3e-3, 1e-12, 7e9])
    m = mags[np.arange(T) % len(mags)]
    q = (wl.queries_f32(T, seed=39).astype(np.float64) * m[:, None, None]).astype(np.float32)
    scores = run_gpu(q, cache, pos0)
    zero_rows = np.nonzero(m == 0)[0]
    assert bool(torch.all(scores[torch.as_tensor(zero_rows, device="cuda"), : pos0 + 1] == 0))
    _compare(q, cache, pos0, scores, np.arange(T), "mixed magnitudes")
