"""The device bounds-check build (libqsa_check.so) on every entry point.

In that build each kernel tests the index of its global-memory accesses
against the size of its buffer as the call's arguments define it; an index
outside sets a device word (read by qsa_check_word) and the access is skipped.
Every kernel runs here on ragged shapes -- token counts off the tile sizes,
padded and out-of-range ids, row pitches past the causal end, both head
dims -- through the C ABI of both builds on the same inputs: the outputs must
be the same bit for bit, and the check word must stay clear.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from sparse_selected_attention_gb300 import _abi
from sparse_selected_attention_gb300 import workloads as wl
from tests.gpu_helpers import dev

pytestmark = pytest.mark.gpu


def _libs():
    return _abi.lib(), _abi.variant("check")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _check_word(L):
    out = ctypes.c_uint(0xFFFFFFFF)
    assert L.qsa_check_word(ctypes.byref(out)) == _abi.QSA_OK
    return out.value


def _same(a, b, what):
    assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{what}: the check build differs"


def test_prep_and_score_paths(cuda_device):
    rel, chk = _libs()
    assert _check_word(chk) == 0
    T, pos0, H = 150, 3000, 12
    C = pos0 + T + 7
    inp = wl.prep_inputs(T, seed=90)
    cache = wl.make_cache(C, seed=90)
    res = {}
    for name, L in (("rel", rel), ("chk", chk)):
        kq, vq, ksc, vsc = (dev(x) for x in (cache.kq, cache.vq, cache.ksc, cache.vsc))
        qi, ki, vi, nw = (dev(x) for x in (inp.q_in, inp.k_in, inp.v_in, inp.norm_w))
        q16 = torch.empty((T, H, 128), dtype=torch.float16, device="cuda")
        q32 = torch.empty((T, H, 128), dtype=torch.float32, device="cuda")
        ws = torch.zeros(L.qsa_score_workspace_bytes(T, 128), dtype=torch.uint8, device="cuda")
        pa = _abi.PrepArgs(ntok=T, pos0=pos0, n_q_heads=H, n_kv_heads=1, head_dim=128, group=32, rope_dims=64,
                           cache_cells=C, eps=1e-6, rope_theta=1e4, q_in=qi.data_ptr(), k_in=ki.data_ptr(),
                           v_in=vi.data_ptr(), norm_w=nw.data_ptr(), q_out=q16.data_ptr(), q_out_f32=q32.data_ptr(),
                           kq=kq.data_ptr(), vq=vq.data_ptr(), ksc=ksc.data_ptr(), vsc=vsc.data_ptr(), rope_k=1,
                           qbar_out=ws.data_ptr())
        assert L.qsa_prep(ctypes.byref(pa), _stream()) == 0
        ld = pos0 + T + 5
        outs = []
        for holds, qsrc, dt in ((1, None, 0), (0, q32, _abi.QSA_F32), (0, q16, _abi.QSA_F16)):
            sc = torch.full((T, ld), -1, dtype=torch.int32, device="cuda").view(torch.float32)
            w2 = ws if holds else torch.zeros_like(ws)
            sa = _abi.ScoreArgs(ntok=T, pos0=pos0, n_q_heads=H, head_dim=128, group=32, cache_cells=C,
                                q=None if qsrc is None else qsrc.data_ptr(), q_dtype=dt, kq=kq.data_ptr(),
                                ksc=ksc.data_ptr(), scores=sc.data_ptr(), ld=ld, workspace=w2.data_ptr(),
                                workspace_bytes=w2.numel(), err=None, workspace_holds_qbar=holds, max_ctas=0)
            assert L.qsa_score(ctypes.byref(sa), _stream()) == 0
            outs.append(sc)
        sc = torch.full((T, ld), -1, dtype=torch.int32, device="cuda").view(torch.float32)
        sa.scores, sa.workspace, sa.workspace_bytes, sa.q, sa.q_dtype = sc.data_ptr(), None, 0, q32.data_ptr(), 0
        assert L.qsa_score_noalloc(ctypes.byref(sa), _stream()) == 0
        outs.append(sc)
        torch.cuda.synchronize()
        res[name] = (q16, q32, kq, vq, ksc, vsc, ws, outs)
    for i, what in enumerate(("q16", "q32", "kq", "vq", "ksc", "vsc", "workspace")):
        _same(res["rel"][i], res["chk"][i], what)
    for j, what in enumerate(("score (head sum from prep)", "score (fp32 q)", "score (fp16 q)", "score noalloc")):
        _same(res["rel"][7][j], res["chk"][7][j], what)
    assert _check_word(chk) == 0


@pytest.mark.parametrize("pages", [False, True])
def test_attention_fused_and_split(cuda_device, pages):
    rel, chk = _libs()
    if pages:
        hq, hkv, d, grp = wl.PAGES_Q_HEADS, wl.PAGES_KV_HEADS, wl.PAGES_HEAD_DIM, wl.PAGES_GROUP
    else:
        hq, hkv, d, grp = 12, 1, 128, 32
    T, C, W = 33, 5000, 448
    cache = wl.make_cache(C, seed=91, head_dim=d, group=grp, kv_heads=hkv)
    q = wl.queries_f16(T, seed=91, heads=hq, head_dim=d)
    ids = wl.even_ids(T, 4960, width=W, select=400)
    ids[5, 64:128] = -1
    ids[7, 3] = C + 2            # out of range: treated as padding, flagged
    ids[8, 9] = -5
    gate = wl.gates_f32(T, seed=91, heads=hq, head_dim=d)
    res = {}
    for name, L in (("rel", rel), ("chk", chk)):
        kq, vq, ksc, vsc = (dev(x) for x in (cache.kq, cache.vq, cache.ksc, cache.vsc))
        qd, idd, gd = dev(q), dev(ids), dev(gate)
        outs = []
        for split in (False, True):
            out = torch.full((T, hq, d), -1, dtype=torch.int16, device="cuda")
            part = torch.full((T, W // 64, hq, d + 2), -1, dtype=torch.int32, device="cuda") if split else None
            err = torch.zeros(1, dtype=torch.int32, device="cuda")
            a = _abi.AttnArgs(ntok=T, n_q_heads=hq, n_kv_heads=hkv, head_dim=d, group=grp, cache_cells=C, width=W,
                              q=qd.data_ptr(), kq=kq.data_ptr(), vq=vq.data_ptr(), ksc=ksc.data_ptr(),
                              vsc=vsc.data_ptr(), ids=idd.data_ptr(), softmax_scale=1 / math.sqrt(d),
                              out=out.data_ptr(), part=None if part is None else part.data_ptr(), err=err.data_ptr(),
                              gate=gd.data_ptr())
            assert L.qsa_attn(ctypes.byref(a), _stream()) == 0
            outs += [out, err] + ([part] if split else [])
        torch.cuda.synchronize()
        res[name] = outs
    for i, (x, y) in enumerate(zip(res["rel"], res["chk"])):
        _same(x, y, f"attention output {i} (pages shape: {pages})")
    assert int(res["chk"][1].item()) & _abi.QSA_DEVERR_BAD_ID
    assert _check_word(chk) == 0


def test_select_and_id_fills(cuda_device):
    rel, chk = _libs()
    T, pos0 = 40, 5000
    sc = wl.normal(92, 1, (T, pos0 + T + 3)).astype(np.float32)   # odd pitch: rows at every 16-byte offset
    sc[3, 100:2000] = 0.5                                           # a plateau
    res = {}
    for name, L in (("rel", rel), ("chk", chk)):
        s = dev(sc)
        outs = []
        for width, budget, sink, local in ((2048, 2048, 64, 256), (1024, 777, 3, 0)):
            ids = torch.full((T, width), -7, dtype=torch.int32, device="cuda")
            a = _abi.SelectArgs(ntok=T, pos0=pos0, width=width, budget=budget, sink=sink, local=local,
                                scores=s.data_ptr(), ld=sc.shape[1], ids=ids.data_ptr())
            assert L.qsa_select(ctypes.byref(a), _stream()) == 0
            outs.append(ids)
        d1 = torch.full((9, 384), -7, dtype=torch.int32, device="cuda")
        assert L.qsa_fill_ids_decode(9, 30000, 384, 64, 256, ctypes.c_void_p(d1.data_ptr()), _stream()) == 0
        d2 = torch.full((70, 2112), -7, dtype=torch.int32, device="cuda")
        assert L.qsa_fill_ids_even(70, 31900, 2112, 2051, ctypes.c_void_p(d2.data_ptr()), _stream()) == 0
        torch.cuda.synchronize()
        res[name] = outs + [d1, d2]
    for i, (x, y) in enumerate(zip(res["rel"], res["chk"])):
        _same(x, y, f"ids {i}")
    assert _check_word(chk) == 0
