"""The whole hot path in sequence on the GPU (prep -> score -> attention) against
the same sequence in the oracle, on a small long-context case."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, prep as oracle_prep, score, score_abs_bound
from sparse_selected_attention_gb300 import qsa_attn, qsa_prep, qsa_score, qsa_score_workspace_bytes
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import assert_f16_close, assert_score_close, dev

pytestmark = pytest.mark.gpu


def test_prep_score_attn_pipeline(cuda_device):
    T, pos0 = 150, 4000
    C = pos0 + T
    inp = wl.prep_inputs(T, seed=51)
    cache = wl.make_cache(C, seed=51)
    ids = wl.even_ids(T, pos0, width=2048)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    q16 = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    q32 = torch.empty((T, 12, 128), dtype=torch.float32, device="cuda")
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q16,
             q_out_f32=q32)
    scores = torch.full((T, C), float("nan"), device="cuda")
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    qsa_score(q32, kq, ksc, pos0, scores, ws)
    out = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    qsa_attn(q16, kq, vq, ksc, vsc, dev(ids), out)
    torch.cuda.synchronize()

    ref = cache.copy()
    q64, _, _ = oracle_prep(inp.q_in, inp.k_in, inp.v_in, inp.norm_w, pos0, ref.kq, ref.vq, ref.ksc, ref.vsc)
    assert np.array_equal(kq.cpu().numpy(), ref.kq) and np.array_equal(vq.cpu().numpy(), ref.vq)
    # The oracle's score and attention consume the oracle's own prep output.
    S = score(q64, ref.kq, ref.ksc, pos0)
    A = score_abs_bound(q64, ref.kq, ref.ksc, pos0)
    assert_score_close(scores.cpu().numpy(), S, A, "pipeline scores")
    o64, _, _, _ = attention(q64.astype(np.float16), ref.kq, ref.vq, ref.ksc, ref.vsc, ids, 1 / math.sqrt(128))
    assert_f16_close(out.cpu(), o64, "pipeline attention")


def test_bench_step_schedule_full_size(cuda_device):
    """The step as bench.py times it (T = 1984, pos0 = 30000, W = 2048): prep,
    then the score on a second stream beside the attention; outputs checked
    against the oracle on sampled token rows."""
    T, pos0 = wl.SCORE_NTOK, 30000
    C = pos0 + T
    inp = wl.prep_inputs(T, seed=5)
    cache = wl.make_cache(C, seed=5)
    ids = wl.even_ids(T, pos0, width=2048)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    q16 = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    q32 = torch.empty((T, 12, 128), dtype=torch.float32, device="cuda")
    scores = torch.empty((T, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(qsa_score_workspace_bytes(T), dtype=torch.uint8, device="cuda")
    out = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    main, side = torch.cuda.current_stream(), torch.cuda.Stream()
    ev = torch.cuda.Event()
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q16,
             q_out_f32=q32)
    ev.record(main)
    side.wait_event(ev)
    qsa_attn(q16, kq, vq, ksc, vsc, dev(ids), out)
    qsa_score(q32, kq, ksc, pos0, scores, ws, stream=side)
    torch.cuda.synchronize()

    ref = cache.copy()
    q64, _, _ = oracle_prep(inp.q_in, inp.k_in, inp.v_in, inp.norm_w, pos0, ref.kq, ref.vq, ref.ksc, ref.vsc)
    assert np.array_equal(kq.cpu().numpy(), ref.kq) and np.array_equal(vq.cpu().numpy(), ref.vq)
    rows = np.array([0, 1, 63, 64, 500, 1000, 1500, 1983])
    S = score(q64, ref.kq, ref.ksc, pos0, rows=rows)
    A = score_abs_bound(q64, ref.kq, ref.ksc, pos0, rows=rows)
    assert_score_close(scores[torch.as_tensor(rows, device="cuda")].cpu().numpy()[:, : S.shape[1]], S, A,
                       "bench step scores")
    o64, _, _, _ = attention(q64.astype(np.float16), ref.kq, ref.vq, ref.ksc, ref.vsc, ids, 1 / math.sqrt(128),
                             rows=rows)
    assert_f16_close(out[torch.as_tensor(rows, device="cuda")].cpu(), o64, "bench step attention")
