"""Edge cases of every entry point on the GPU: empty batches, the largest
selection rows, id lists wider than the workload's, and prep at positions far
beyond the workload's (angle reduction), each against the oracle."""
import math

import numpy as np
import pytest
import torch

from oracle import attention, prep_queries, quantize_rows, rotate_keys_f32, select_ids
from sparse_selected_attention_gb300 import (QSA_SELECT_MAX_CELLS, qsa_attn, qsa_prep, qsa_score, qsa_score_noalloc,
                                             qsa_score_workspace_bytes, qsa_select)
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import assert_f16_close, cache_dev, dev

pytestmark = pytest.mark.gpu


def test_zero_tokens_every_entry_point(cuda_device):
    cache = wl.make_cache(100, seed=81)
    kq, vq, ksc, vsc = cache_dev(cache)
    before = [x.clone() for x in (kq, vq, ksc, vsc)]
    e = lambda *s, dt=torch.float32: torch.empty(s, dtype=dt, device="cuda")  # noqa: E731
    qsa_prep(e(0, 12, 128), e(0, 1, 128), e(0, 1, 128), e(128), 50, kq, vq, ksc, vsc,
             e(0, 12, 128, dt=torch.float16), q_out_f32=e(0, 12, 128))
    ws = torch.empty(max(1, qsa_score_workspace_bytes(0)), dtype=torch.uint8, device="cuda")
    qsa_score(e(0, 12, 128), kq, ksc, 50, e(0, 100), ws)
    qsa_score_noalloc(e(0, 12, 128), kq, ksc, 50, e(0, 100))
    qsa_select(e(0, 100), 50, e(0, 2048, dt=torch.int32))
    qsa_attn(e(0, 12, 128, dt=torch.float16), kq, vq, ksc, vsc, e(0, 64, dt=torch.int32),
             e(0, 12, 128, dt=torch.float16))
    torch.cuda.synchronize()
    for b, a in zip(before, (kq, vq, ksc, vsc)):
        assert torch.equal(b, a)


@pytest.mark.parametrize("ld_pad", [0, 1])
def test_select_at_the_cell_limit(cuda_device, ld_pad):
    T = 8
    pos0 = QSA_SELECT_MAX_CELLS - T                   # the last row holds 32768 cells
    sc = wl.normal(82, 1, (T, pos0 + T + ld_pad)).astype(np.float32)
    sc[:, 5000:5100] = 1.5                            # a plateau too
    ids = torch.full((T, 2048), -7, dtype=torch.int32, device="cuda")
    qsa_select(dev(sc), pos0, ids)
    torch.cuda.synchronize()
    assert np.array_equal(ids.cpu().numpy(), select_ids(sc, pos0))


def test_attention_wide_id_list(cuda_device):
    # 4096 slots (64 chunks), 3500 valid scattered cells, padding at the end
    # and in the middle.
    cells, T = 20000, 3
    cache = wl.make_cache(cells, seed=83)
    q = wl.queries_f16(T, seed=83)
    ids = np.full((T, 4096), -1, dtype=np.int32)
    for t in range(T):
        keys = wl.random_u64(83, 200 + t, cells)
        ids[t, :3500] = np.argsort(keys, kind="stable")[:3500]
    ids[1, 1000:1200] = -1
    kq, vq, ksc, vsc = cache_dev(cache)
    out = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    qsa_attn(dev(q), kq, vq, ksc, vsc, dev(ids), out)
    torch.cuda.synchronize()
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 1 / math.sqrt(128))
    assert_f16_close(out.cpu(), ref, "W=4096")


@pytest.mark.parametrize("rope_k", [False, True])
def test_prep_far_positions(cuda_device, rope_k):
    # Positions near 2^22: angles up to ~4 M rad.  Only the written rows are
    # compared; the cache is zero elsewhere.
    T, pos0 = 16, (1 << 22) - 16
    inp = wl.prep_inputs(T, seed=84)
    C = pos0 + T
    kq = torch.zeros((C, 128), dtype=torch.int8, device="cuda")
    vq = torch.zeros_like(kq)
    ksc = torch.zeros((C, 4), dtype=torch.float16, device="cuda")
    vsc = torch.zeros_like(ksc)
    q16 = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    q32 = torch.empty((T, 12, 128), dtype=torch.float32, device="cuda")
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q16,
             q_out_f32=q32, rope_k=rope_k)
    torch.cuda.synchronize()
    q64, _, _ = prep_queries(inp.q_in, inp.norm_w, pos0)
    assert_f16_close(q16.cpu(), q64, "q fp16 at far positions")
    np.testing.assert_allclose(q32.cpu().numpy(), q64, atol=2e-5, rtol=0)
    k = rotate_keys_f32(inp.k_in, pos0) if rope_k else inp.k_in
    kc, ks = quantize_rows(k.reshape(T, -1))
    vc, vs = quantize_rows(inp.v_in.reshape(T, -1))
    rows = slice(pos0, pos0 + T)
    assert np.array_equal(kq[rows].cpu().numpy(), kc) and np.array_equal(vq[rows].cpu().numpy(), vc)
    assert np.array_equal(ksc[rows].cpu().numpy().view(np.int16), ks.view(np.int16))
    assert np.array_equal(vsc[rows].cpu().numpy().view(np.int16), vs.view(np.int16))
    assert int(kq[:pos0].abs().sum()) == 0 and int(vq[:pos0].abs().sum()) == 0
