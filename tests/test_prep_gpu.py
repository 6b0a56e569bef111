"""qsa_prep on the GPU against the CPU oracle, through the C ABI.

Shapes follow the prep measurements on the pages (P = 0 / 3000, nt = 1, 2, 4,
8, 1984, 2048) plus long-context positions.  Quantised codes and scale bits
must match bit for bit; cache rows outside pos0 .. pos0+T-1 must be untouched.
"""
import numpy as np
import pytest
import torch

from oracle import prep as oracle_prep
from sparse_selected_attention_gb300 import qsa_prep
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import assert_f16_close, dev

pytestmark = pytest.mark.gpu

Q32_ATOL = 2e-5   # fp32 arithmetic on O(1) values: a few ulp of the row scale


def run_case(T, pos0, rope_dims=64, heads=12, extra=7, seed=41, rope_k=False):
    inp = wl.prep_inputs(T, seed=seed, heads=heads)
    C = pos0 + T + extra
    cache = wl.make_cache(C, seed=seed)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    q_out = torch.full((T, heads, 128), float("nan"), dtype=torch.float16, device="cuda")
    q32 = torch.full((T, heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q_out,
             q_out_f32=q32, rope_dims=rope_dims, rope_k=rope_k)
    torch.cuda.synchronize()
    ref_cache = cache.copy()
    q64, _, _ = oracle_prep(inp.q_in, inp.k_in, inp.v_in, inp.norm_w, pos0, ref_cache.kq, ref_cache.vq,
                            ref_cache.ksc, ref_cache.vsc, rope_dims=rope_dims, rope_k=rope_k)
    assert_f16_close(q_out.cpu(), q64, f"q fp16 T={T} pos0={pos0}")
    np.testing.assert_allclose(q32.cpu().numpy(), q64, atol=Q32_ATOL, rtol=0)
    for name, g, r in (("kq", kq, ref_cache.kq), ("vq", vq, ref_cache.vq),
                       ("ksc", ksc, ref_cache.ksc.view(np.int16)), ("vsc", vsc, ref_cache.vsc.view(np.int16))):
        gn = g.cpu().numpy()
        if gn.dtype == np.float16:
            gn = gn.view(np.int16)
        assert np.array_equal(gn, r), f"{name} differs from the oracle (T={T}, pos0={pos0})"


@pytest.mark.parametrize("T,pos0", [(1, 3000), (2, 3000), (4, 3000), (8, 3000), (1984, 0), (1984, 3000),
                                    (2048, 3000), (37, 30000), (5, 31979)])
def test_prep_shapes(cuda_device, T, pos0):
    run_case(T, pos0)


@pytest.mark.parametrize("heads", [1, 2, 4, 5, 7, 8, 16, 29, 30])
def test_prep_head_counts(cuda_device, heads):
    """Query rows are dealt three to a warp: head counts that leave the last
    query warp one or two rows short, and the launcher's maximum of 30."""
    run_case(37, 900, heads=heads, seed=50 + heads)


@pytest.mark.parametrize("rope_dims", [0, 8, 128])
def test_prep_rope_dims(cuda_device, rope_dims):
    run_case(19, 1234, rope_dims=rope_dims)


def test_prep_zero_group_and_large_values(cuda_device):
    T, pos0 = 3, 10
    inp = wl.prep_inputs(T, seed=42)
    inp.k_in[0, 0, 32:64] = 0.0            # a zero group -> scale 0, codes 0
    inp.v_in[1, 0, :] *= 1e4               # large magnitudes
    inp.v_in[2, 0, 96:] = 1e-30            # tiny group -> fp16 scale underflows to 0
    C = pos0 + T
    cache = wl.make_cache(C, seed=42)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    q_out = torch.empty((T, 12, 128), dtype=torch.float16, device="cuda")
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q_out)
    torch.cuda.synchronize()
    ref = cache.copy()
    oracle_prep(inp.q_in, inp.k_in, inp.v_in, inp.norm_w, pos0, ref.kq, ref.vq, ref.ksc, ref.vsc)
    assert np.array_equal(kq.cpu().numpy(), ref.kq) and np.array_equal(vq.cpu().numpy(), ref.vq)
    assert np.array_equal(ksc.cpu().numpy().view(np.int16), ref.ksc.view(np.int16))
    assert np.array_equal(vsc.cpu().numpy().view(np.int16), ref.vsc.view(np.int16))
    assert float(ref.ksc[pos0, 1]) == 0.0 and float(ref.vsc[pos0 + 2, 3]) == 0.0


@pytest.mark.parametrize("T,pos0,rope_dims", [(1984, 30000, 64), (64, 0, 64), (19, 1234, 8), (19, 1234, 128),
                                              (300, 32000, 64)])
def test_prep_rope_k(cuda_device, T, pos0, rope_dims):
    """Key rotation before quantisation: codes and scale bits bit-exact with
    the oracle, at angles up to ~32 K rad."""
    run_case(T, pos0, rope_dims=rope_dims, rope_k=True, seed=47)


@pytest.mark.parametrize("T,heads,wscale", [(150, 12, 1.0), (64, 1, 1.0), (1, 30, 1.0), (150, 12, 1e-6),
                                             (150, 12, 1e6), (70, 12, 1e-25)])
def test_prep_head_sum_feeds_the_score(cuda_device, T, heads, wscale):
    """qsa_prep's qbar_out is the score's own head sum bit for bit (its
    per-token power of two included), a score from it equals the score from
    q_out_f32 bit for bit, and both match the oracle's score of q_out_f32 --
    also with norm weights scaled far up or down, which moves every head sum
    out of the unscaled fp16 range."""
    from oracle import score, score_abs_bound
    from sparse_selected_attention_gb300 import qsa_score, qsa_score_workspace_bytes
    from tests.gpu_helpers import assert_score_close
    pos0 = 3000
    inp = wl.prep_inputs(T, seed=48, heads=heads)
    inp.norm_w = (inp.norm_w.astype(np.float64) * wscale).astype(np.float32)
    cache = wl.make_cache(pos0 + T, seed=48)
    kq, vq, ksc, vsc = dev(cache.kq), dev(cache.vq), dev(cache.ksc), dev(cache.vsc)
    q16 = torch.empty((T, heads, 128), dtype=torch.float16, device="cuda")
    q32 = torch.empty((T, heads, 128), dtype=torch.float32, device="cuda")
    nb = qsa_score_workspace_bytes(T)
    ws_prep = torch.full((nb,), 0x7f, dtype=torch.uint8, device="cuda")
    ws_score = torch.full((nb,), 0x55, dtype=torch.uint8, device="cuda")
    qsa_prep(dev(inp.q_in), dev(inp.k_in), dev(inp.v_in), dev(inp.norm_w), pos0, kq, vq, ksc, vsc, q16,
             q_out_f32=q32, qbar_out=ws_prep)
    s_q = torch.full((T, pos0 + T), -1, dtype=torch.int32, device="cuda").view(torch.float32)
    s_bar = s_q.clone()
    qsa_score(q32, kq, ksc, pos0, s_q, ws_score)
    qsa_score(None, kq, ksc, pos0, s_bar, ws_prep, workspace_holds_qbar=True, n_q_heads=heads)
    torch.cuda.synchronize()
    assert torch.equal(ws_prep, ws_score)                    # padding rows included
    assert torch.equal(s_q.view(torch.int32), s_bar.view(torch.int32))
    q32n = q32.cpu().numpy()
    kqn, kscn = kq.cpu().numpy(), ksc.cpu().numpy()         # with the rows prep just wrote
    rows = np.arange(T)
    ref = score(q32n, kqn, kscn, pos0, rows=rows)
    A = score_abs_bound(q32n, kqn, kscn, pos0, rows=rows)
    assert_score_close(s_bar.cpu().numpy(), ref, A, f"score from prep's head sum, weights x{wscale:g}")
