"""The allocation-free scoring entry point (qsa_score_noalloc).

Some callers cannot allocate device memory when they score (an engine that
owns all device memory, a loop that must not call cudaMalloc); for them the
library keeps its scoring scratch in a fixed built-in array.  This checks,
through the C ABI, that two calls in a row give the same scores as the
workspace entry point (within the score tolerance), leave non-causal cells
untouched, and that oversize requests are refused.  The file name makes
pytest collect it last.
"""
import numpy as np
import pytest
import torch

from oracle import score_abs_bound
from sparse_selected_attention_gb300 import _abi, qsa_score, qsa_score_noalloc, qsa_score_workspace_bytes
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import SENTINEL_BITS, assert_score_close, dev

pytestmark = pytest.mark.gpu


def _sentinel(T, ld):
    return torch.full((T, ld), SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)


@pytest.mark.parametrize("first,second", [((300, 2000, np.float32), (70, 130, np.float16))])
def test_noalloc_matches_workspace_entry_on_two_calls(cuda_device, first, second):
    for i, (T, pos0, dtype) in enumerate((first, second)):
        cache = wl.make_cache(pos0 + T, seed=60 + i)
        q = wl.queries_f32(T, seed=60 + i).astype(dtype)
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
        causal = torch.arange(ld, device="cuda")[None, :] <= (pos0 + torch.arange(T, device="cuda"))[:, None]
        assert bool(torch.all(got.view(torch.int32)[~causal] == SENTINEL_BITS))
        r = ref.cpu().numpy().astype(np.float64)
        r[~causal.cpu().numpy()] = np.nan
        A = score_abs_bound(q, cache.kq, cache.ksc, pos0)
        A = np.pad(A, ((0, 0), (0, ld - A.shape[1])))
        assert_score_close(got.cpu().numpy(), r, A, f"noalloc call {i + 1}")


def test_noalloc_rejects_oversize(cuda_device):
    T = _abi.QSA_SCORE_NOALLOC_MAX_TOKENS + 1
    q = torch.zeros((T, 12, 128), dtype=torch.float16, device="cuda")
    kq = torch.zeros((T, 128), dtype=torch.int8, device="cuda")
    ksc = torch.zeros((T, 4), dtype=torch.float16, device="cuda")
    scores = torch.zeros((T, T), dtype=torch.float32, device="cuda")
    with pytest.raises(_abi.QSAError) as ei:
        qsa_score_noalloc(q, kq, ksc, 0, scores)
    assert ei.value.status == _abi.QSA_ERR_INVALID_ARG and "8192" in str(ei.value)
