"""Shared pieces of the GPU parity tests: device copies and the tolerances.

Tolerances (the fp16 and fp32 bounds the method is specified with):
  fp16 attention / query outputs: |gpu - ref| <= 2e-3 + 1e-2 * |ref|, with ref the
  oracle's float64 value before fp16 rounding (max abs error 2e-3 and max
  relative error 1e-2, combined so the bound stays defined near zero);
  fp32 scores: |gpu - ref| <= 1e-4 * A, with A = sum |each product term| (the
  magnitude that bounds any evaluation order's rounding; cancelling sums make a
  plain |ref|-relative bound meaningless).
Integer, id, scale-bit and untouched-sentinel comparisons are bitwise.
"""
import numpy as np
import torch

F16_ATOL, F16_RTOL = 2e-3, 1e-2
SCORE_RTOL_A = 1e-4
SENTINEL_BITS = -1  # 0xFFFFFFFF, a NaN


def dev(x):
    return torch.from_numpy(np.ascontiguousarray(x)).cuda()


def cache_dev(cache):
    return dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)


def assert_f16_close(gpu, ref64, what=""):
    g = gpu.float().cpu().numpy().astype(np.float64) if isinstance(gpu, torch.Tensor) else gpu.astype(np.float64)
    err = np.abs(g - ref64)
    bound = F16_ATOL + F16_RTOL * np.abs(ref64)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {err.size} outside tolerance; worst at {i}: gpu={g[i]} "
                             f"ref={ref64[i]} err={err[i]:.3g}")
    return float(err.max()) if err.size else 0.0


def assert_score_close(gpu_rows, ref, A, what=""):
    causal = ~np.isnan(ref)
    g = gpu_rows.astype(np.float64)
    err = np.where(causal, np.abs(g - np.where(causal, ref, 0.0)), 0.0)
    bound = SCORE_RTOL_A * A
    bad = causal & ~(err <= bound)
    if bad.any():
        i = np.unravel_index(np.argmax(np.where(causal, err / np.maximum(bound, 1e-300), 0)), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {causal.sum()} outside 1e-4*A; worst at {i}: gpu={g[i]} "
                             f"ref={ref[i]} A={A[i]}")
    rel = np.where(causal, err / np.maximum(A, 1e-300), 0.0)
    return float(rel.max()) if rel.size else 0.0


def assert_valid_selection(got, ref_ids, S, A, pos0, budget=2048, sink=64, local=256, what=""):
    """Selection made by the GPU from its own scores, judged against the
    oracle's float64 scores S (bound 1e-4 * A).  Rows equal to the oracle's
    ids (selected from fp32(S)) pass outright.  A row that differs must still
    be a valid choice: ascending distinct causal ids, -1 after them, the right
    count, every forced decode-window cell present, and no unchosen free cell
    scoring above a chosen one by more than the two cells' score bounds
    (which is where fp32 rounding of the scores can swap near-ties)."""
    got = np.asarray(got)
    differ = []
    for t in range(got.shape[0]):
        if np.array_equal(got[t], ref_ids[t]):
            continue
        differ.append(t)
        p = pos0 + t
        n = p + 1
        k = min(n, budget)
        row = got[t]
        ids = row[:k]
        assert np.all(row[k:] == -1), f"{what}: row {t} has ids past its {k} slots"
        assert np.all(ids >= 0) and np.all(ids <= p) and np.all(np.diff(ids) > 0), \
            f"{what}: row {t} ids are not ascending distinct causal cells"
        forced = np.zeros(n, dtype=bool)
        forced[: min(sink, n)] = True
        forced[max(sink, p - local): p] = True
        forced[p] = True
        chosen = np.zeros(n, dtype=bool)
        chosen[ids] = True
        assert np.all(chosen[forced]), f"{what}: row {t} misses a forced cell"
        pick, left = chosen & ~forced, ~chosen & ~forced
        if pick.any() and left.any():
            tol = SCORE_RTOL_A * A[t, :n]
            lo = np.min(S[t, :n][pick] + tol[pick])
            hi = np.max(S[t, :n][left] - tol[left])
            assert lo >= hi, f"{what}: row {t} leaves out a cell that outscores a chosen one beyond the bound"
    return differ
