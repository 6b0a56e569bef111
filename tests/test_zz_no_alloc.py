"""The allocation-free scoring entry point (qsa_score_noalloc).

Some callers cannot allocate device memory when they score: an engine that
owns all device memory and forbids allocation inside its execute callback,
or a serving loop that must not call cudaMalloc (it can synchronise the
device and has no latency bound).  For them the library keeps its scoring
scratch in a fixed built-in array.  This checks, through the C ABI, that
consecutive calls -- the first filling the whole array, the later ones
smaller, so stale rows of an earlier call would show -- give scores bit for
bit equal to the workspace entry point's on the same inputs and within the
score tolerance of the oracle, leave non-causal cells untouched, and that
requests beyond the array are refused.  The file name makes pytest collect it
last.
"""
import numpy as np
import pytest
import torch

from oracle import score, score_abs_bound
from sparse_selected_attention_gb300 import _abi, qsa_score, qsa_score_noalloc, qsa_score_workspace_bytes
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import SENTINEL_BITS, assert_score_close, dev

pytestmark = pytest.mark.gpu

MAXT = _abi.QSA_SCORE_NOALLOC_MAX_TOKENS


def _sentinel(T, ld):
    return torch.full((T, ld), SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)


# (T, pos0, query dtype, query heads, seed): the first call fills the whole
# built-in array (T = its limit), the next two reuse it with fewer tokens.
CALLS = [(MAXT, 5, np.float32, 2, 60), (300, 2000, np.float32, 12, 61), (70, 130, np.float16, 12, 62)]


def test_noalloc_matches_workspace_entry_and_oracle_on_consecutive_calls(cuda_device):
    for i, (T, pos0, dtype, heads, seed) in enumerate(CALLS):
        cache = wl.make_cache(pos0 + T, seed=seed)
        q = wl.queries_f32(T, seed=seed, heads=heads).astype(dtype)
        qd, kq, ksc = dev(q), dev(cache.kq), dev(cache.ksc)
        ld = pos0 + T + 3
        ref = _sentinel(T, ld)
        ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
        qsa_score(qd, kq, ksc, pos0, ref, ws)
        got = _sentinel(T, ld)
        err = torch.zeros(1, dtype=torch.int32, device="cuda")
        qsa_score_noalloc(qd, kq, ksc, pos0, got, err=err)
        torch.cuda.synchronize()
        assert int(err.item()) == 0
        # Same kernels on the same inputs: every element, causal or sentinel,
        # is the same bit pattern.
        assert torch.equal(got.view(torch.int32), ref.view(torch.int32)), f"call {i + 1}: differs from qsa_score"
        causal = torch.arange(ld, device="cuda")[None, :] <= (pos0 + torch.arange(T, device="cuda"))[:, None]
        assert bool(torch.all(got.view(torch.int32)[~causal] == SENTINEL_BITS))
        # And against the oracle, on every row of the small calls and on rows
        # spread over the big one (its first, last and tile-boundary rows).
        if T <= 512:
            rows = np.arange(T)
        else:
            rng = np.random.default_rng(seed)
            rows = np.array(sorted(set(rng.choice(T, 60, replace=False).tolist())
                                   | {0, 63, 64, 127, 128, T - 129, T - 128, T - 65, T - 64, T - 1}))
        r = score(q, cache.kq, cache.ksc, pos0, rows=rows)
        A = score_abs_bound(q, cache.kq, cache.ksc, pos0, rows=rows)
        g = got[torch.as_tensor(rows, device="cuda")].cpu().numpy()[:, : r.shape[1]]
        assert_score_close(g, r, A, f"noalloc call {i + 1} (T={T}) against the oracle")


def test_noalloc_rejects_oversize(cuda_device):
    T = MAXT + 1
    q = torch.zeros((T, 12, 128), dtype=torch.float16, device="cuda")
    kq = torch.zeros((T, 128), dtype=torch.int8, device="cuda")
    ksc = torch.zeros((T, 4), dtype=torch.float16, device="cuda")
    scores = torch.zeros((T, T), dtype=torch.float32, device="cuda")
    with pytest.raises(_abi.QSAError) as ei:
        qsa_score_noalloc(q, kq, ksc, 0, scores)
    assert ei.value.status == _abi.QSA_ERR_INVALID_ARG and str(MAXT) in str(ei.value)
