"""qsa_attn at the pages' own shape and with the output gate, on the GPU,
against the oracle on the same seeded inputs.

The shape is that of "round 5 track b: cached residual norms and fused mtp
attention", section "mtp attention" and its actual-verification list. It has
2 KV heads with 12 query heads each, head_dim 256 and fp16 per-64 scales, plus
fp32 gates. The cases cover widths of 1, 31, 64, 65, 128, 319, 320, 321, 384
and 2051 valid cells, with scattered non-contiguous ids and two tokens per
width. Their seed number, 20260701, is reused here.
"""
import numpy as np
import pytest
import torch

from oracle import attention
from sparse_selected_attention_gb300 import qsa_attn
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import assert_f16_close, cache_dev, dev

pytestmark = pytest.mark.gpu

H, HKV, D, GRP, SCALE = wl.PAGES_Q_HEADS, wl.PAGES_KV_HEADS, wl.PAGES_HEAD_DIM, wl.PAGES_GROUP, wl.PAGES_SCALE


def scattered(ntok, cells, valid, width, seed):
    """`valid` distinct cells per token in a seeded random order, then -1."""
    ids = np.full((ntok, width), -1, dtype=np.int32)
    for t in range(ntok):
        keys = wl.random_u64(seed, 100 + t, cells)
        ids[t, :valid] = np.argsort(keys, kind="stable")[:valid]
    return ids


def run(q, cache, ids, scale, gate=None, part=False):
    T, Hq, Dd = q.shape
    kq, vq, ksc, vsc = cache_dev(cache)
    out = torch.full((T, Hq, Dd), float("nan"), dtype=torch.float16, device="cuda")
    nch = ids.shape[1] // 64
    pt = torch.full((T, nch, Hq, Dd + 2), float("nan"), device="cuda") if part else None
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    qsa_attn(dev(q), kq, vq, ksc, vsc, dev(ids), out, scale, part=pt, err=err,
             gate=None if gate is None else dev(gate))
    torch.cuda.synchronize()
    assert int(err.item()) == 0
    return out.cpu(), (pt.cpu().numpy() if part else None)


def check_partials(pt, refpart, d):
    """Chunk partials: m, then l and o rescaled to the oracle's maximum."""
    ref_m, ref_l, ref_o = refpart[..., d], refpart[..., d + 1], refpart[..., :d]
    g_m, g_l, g_o = pt[..., d], pt[..., d + 1], pt[..., :d]
    empty = ~np.isfinite(ref_m)
    assert np.array_equal(np.isfinite(g_m), ~empty)
    assert np.all(g_l[empty] == 0) and np.all(g_o[empty] == 0)
    ne = ~empty
    np.testing.assert_allclose(g_m[ne], ref_m[ne], atol=2e-3, rtol=2e-3)
    np.testing.assert_allclose(g_l[ne] * np.exp(g_m[ne] - ref_m[ne]), ref_l[ne], rtol=2e-3)
    vmax = 127 * 0.0201
    err = np.abs(g_o * np.exp(g_m - np.where(ne, ref_m, 0))[..., None] - ref_o)
    assert np.all(err[ne] <= 2e-3 * (ref_l * vmax)[..., None][ne] + 1e-6)


@pytest.mark.parametrize("valid", [1, 31, 64, 65, 128, 319, 320, 321, 384, 2051])
@pytest.mark.parametrize("gated", [False, True])
def test_pages_shape_width_matrix(cuda_device, valid, gated):
    cells = 6000
    seed = wl.PAGES_SEED
    cache = wl.make_cache(cells, seed=seed, head_dim=D, group=GRP, kv_heads=HKV)
    q = wl.queries_f16(2, seed=seed + valid, heads=H, head_dim=D)
    width = -(-valid // 64) * 64
    ids = scattered(2, cells, valid, width, seed + valid)
    gate = wl.gates_f32(2, seed=seed + valid, heads=H, head_dim=D) if gated else None
    out, _ = run(q, cache, ids, SCALE, gate=gate)
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE, group=GRP, gate=gate)
    assert_f16_close(out, ref, f"pages shape, {valid} valid cells, gated={gated}")


def test_pages_shape_split_path(cuda_device):
    cells, T = 3000, 9
    cache = wl.make_cache(cells, seed=41, head_dim=D, group=GRP, kv_heads=HKV)
    q = wl.queries_f16(T, seed=41, heads=H, head_dim=D)
    ids = scattered(T, cells, 321, 384, 41)
    ids[3, 64:128] = -1                                   # an empty chunk in the middle
    ids[5, :] = -1                                        # a token with no valid cell
    gate = wl.gates_f32(T, seed=41, heads=H, head_dim=D)
    out, pt = run(q, cache, ids, SCALE, gate=gate, part=True)
    ref, _, refpart, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE, group=GRP,
                                   want_part=True, gate=gate)
    assert_f16_close(out, ref, "pages shape, split path")
    check_partials(pt, refpart, D)
    o5 = out[5].numpy()
    assert np.all(o5 == 0) and not np.signbit(o5).any()
    out2, _ = run(q, cache, ids, SCALE, gate=gate)
    assert_f16_close(out2, out.float().numpy().astype(np.float64), "pages shape, fused vs split")


def test_pages_shape_long_context(cuda_device):
    # Prompt-like lists over a 31 K-cell cache: many units per token, the last
    # chunk ragged (2051 of 2112 slots).
    T, pos0 = 24, 30000
    cache = wl.make_cache(pos0 + T, seed=42, head_dim=D, group=GRP, kv_heads=HKV)
    q = wl.queries_f16(T, seed=42, heads=H, head_dim=D)
    ids = wl.even_ids(T, pos0, width=2112, select=2051)
    out, _ = run(q, cache, ids, SCALE)
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, SCALE, group=GRP)
    assert_f16_close(out, ref, "pages shape, long context")


def test_pages_shape_full_size_sampled(cuda_device):
    """The bench's pages-shape workload in its own launch configuration: all
    1984 tokens over 2048 evenly spaced ids of a 31984-cell cache, in one
    call; 128 seeded rows plus the first and last compared with the oracle."""
    T, pos0, W = 1984, 30000, 2048
    cache = wl.make_cache(pos0 + T, seed=wl.PAGES_SEED, head_dim=D, group=GRP, kv_heads=HKV)
    q = wl.queries_f16(T, seed=wl.PAGES_SEED, heads=H, head_dim=D)
    ids = wl.even_ids(T, pos0, W)
    out, _ = run(q, cache, ids, SCALE)
    rows = np.unique(np.concatenate([[0, T - 1], np.argsort(wl.random_u64(wl.PAGES_SEED, 7, T), kind="stable")[:128]]))
    ref, _, _, _ = attention(q[rows], cache.kq, cache.vq, cache.ksc, cache.vsc, ids[rows], SCALE, group=GRP)
    assert_f16_close(out[rows], ref, "pages shape, full size, sampled rows")


@pytest.mark.parametrize("part", [False, True])
def test_gate_on_workload_shape(cuda_device, part):
    cache = wl.make_cache(5000, seed=43)
    q = wl.queries_f16(40, seed=43)
    ids = wl.even_ids(40, 4900, width=2048)
    gate = wl.gates_f32(40, seed=43)
    gate[3] = 0.0                                         # exactly half
    gate[4] = -1e30                                       # fully closed: +0 output
    out, _ = run(q, cache, ids, 1 / np.sqrt(128), gate=gate, part=part)
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 1 / np.sqrt(128), gate=gate)
    assert_f16_close(out, ref, f"gated, part={part}")
    assert np.all(out[4].numpy() == 0)


def test_two_kv_heads_on_workload_dim(cuda_device):
    # head_dim 128 with 2 KV heads of 6 query heads each.
    cache = wl.make_cache(3000, seed=44, kv_heads=2)
    q = wl.queries_f16(17, seed=44, heads=12)
    ids = scattered(17, 3000, 700, 768, 44)
    out, _ = run(q, cache, ids, 1 / np.sqrt(128))
    ref, _, _, _ = attention(q, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 1 / np.sqrt(128))
    assert_f16_close(out, ref, "2 KV heads, head_dim 128")
