"""The time-out path of the score kernel's bounded waits, on the GPU.

Every wait in the tcgen05 score pipeline gives up after a fixed number of
polls, records QSA_DEVERR_TIMEOUT in the caller's error word, and stops every
role in order: the MMA thread waits for the MMAs it has issued, then tensor
memory is freed and the kernel returns.  libqsa_wait0.so is the same source
built with QSA_WAIT_LIMIT=0, so each of those waits gives up at its first
poll; the run below takes that path on purpose, with no fault, trap or hang:
the call must return, set the bit, leave every score cell as the caller
filled it, and leave the context usable for the release library.
"""
import ctypes

import numpy as np
import pytest
import torch

from oracle import score, score_abs_bound
from sparse_selected_attention_gb300 import QSA_DEVERR_TIMEOUT, _abi, qsa_score, qsa_score_workspace_bytes
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import SENTINEL_BITS, assert_score_close, dev

pytestmark = pytest.mark.gpu


def _score_args(q, kq, ksc, pos0, scores, ws, err):
    return _abi.ScoreArgs(ntok=q.shape[0], pos0=pos0, n_q_heads=q.shape[1], head_dim=128, group=32,
                          cache_cells=kq.shape[0], q=q.data_ptr(), q_dtype=_abi.QSA_F32, kq=kq.data_ptr(),
                          ksc=ksc.data_ptr(), scores=scores.data_ptr(), ld=scores.shape[1],
                          workspace=ws.data_ptr(), workspace_bytes=ws.numel(), err=err.data_ptr(),
                          workspace_holds_qbar=0, max_ctas=0)


@pytest.mark.parametrize("T,pos0", [(8, 100), (300, 2000)])
def test_score_wait_timeout_sets_error_and_stops(cuda_device, T, pos0):
    L = _abi.variant("wait0")
    cache = wl.make_cache(pos0 + T, seed=70)
    q = wl.queries_f32(T, seed=70)
    qd, kq, ksc = dev(q), dev(cache.kq), dev(cache.ksc)
    scores = torch.full((T, pos0 + T), SENTINEL_BITS, dtype=torch.int32, device="cuda").view(torch.float32)
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _score_args(qd, kq, ksc, pos0, scores, ws, err)
    st = L.qsa_score(ctypes.byref(a), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _abi.QSA_OK
    torch.cuda.synchronize()
    assert int(err.item()) & QSA_DEVERR_TIMEOUT, "the time-out bit was not set"
    # The epilogue gives up before its first accumulator: nothing is stored.
    assert bool(torch.all(scores.view(torch.int32) == SENTINEL_BITS))

    # The context is still usable: the release library scores the same input.
    good = torch.full_like(scores.view(torch.int32), SENTINEL_BITS).view(torch.float32)
    err.zero_()
    qsa_score(qd, kq, ksc, pos0, good, ws, err=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    rows = np.arange(T)
    ref = score(q, cache.kq, cache.ksc, pos0, rows=rows)
    A = score_abs_bound(q, cache.kq, cache.ksc, pos0, rows=rows)
    assert_score_close(good.cpu().numpy(), ref, A, f"release library after the time-out, T={T}")
