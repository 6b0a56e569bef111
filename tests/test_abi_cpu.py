"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments before any CUDA call."""
import ctypes

import pytest

from sparse_selected_attention_gb300 import _abi, build


@pytest.fixture(scope="module")
def L():
    build.build()
    return _abi.lib()


def test_exports_every_header_function(L):
    names = _abi.header_functions()
    assert {"qsa_prep", "qsa_score", "qsa_attn", "qsa_status_str", "qsa_last_error", "qsa_abi_version",
            "qsa_score_workspace_bytes"} <= set(names)
    for n in names:
        assert hasattr(L, n), n
    assert L.qsa_abi_version() == 3
    assert L.qsa_status_str(0) == b"ok" and L.qsa_status_str(2) == b"unsupported shape"


def test_workspace_bytes(L):
    # per padded token: fp16 hi and lo rows of 128 dims, one int32 exponent
    assert L.qsa_score_workspace_bytes(1, 128) == 64 * 516
    assert L.qsa_score_workspace_bytes(1984, 128) == 1984 * 516
    assert L.qsa_score_workspace_bytes(1985, 128) == 2048 * 516
    assert L.qsa_score_workspace_bytes(10, 64) == 0


FAKE = 1 << 20  # an aligned non-null address; never dereferenced (validation fails first)


def _attn(**kw):
    a = _abi.AttnArgs(ntok=4, n_q_heads=12, n_kv_heads=1, head_dim=128, group=32, cache_cells=100, width=128,
                      q=FAKE, kq=FAKE, vq=FAKE, ksc=FAKE, vsc=FAKE, ids=FAKE, softmax_scale=0.088, out=FAKE,
                      part=None, err=None)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


def _status(L, fn, args):
    # These calls carry fake device addresses and rely on host validation to
    # refuse them; a validation bug must never reach a real GPU with them.
    import torch
    if torch.cuda.is_available():
        pytest.skip("argument-rejection checks use fake device addresses: run them on a machine without a GPU")
    s = getattr(L, fn)(ctypes.byref(args), None)
    return s, L.qsa_last_error().decode()


@pytest.mark.parametrize("kw,want", [
    (dict(width=100), _abi.QSA_ERR_INVALID_ARG),
    (dict(width=0), _abi.QSA_ERR_INVALID_ARG),
    (dict(n_q_heads=17), _abi.QSA_ERR_UNSUPPORTED),
    (dict(head_dim=256), _abi.QSA_ERR_UNSUPPORTED),           # 256 needs 64-dim groups
    (dict(group=64), _abi.QSA_ERR_UNSUPPORTED),               # 128 needs 32-dim groups
    (dict(head_dim=64, group=16), _abi.QSA_ERR_UNSUPPORTED),
    (dict(n_kv_heads=5), _abi.QSA_ERR_UNSUPPORTED),           # 12 heads do not split over 5
    (dict(n_kv_heads=0), _abi.QSA_ERR_UNSUPPORTED),
    (dict(n_q_heads=34, n_kv_heads=2), _abi.QSA_ERR_UNSUPPORTED),  # 17 query heads per KV head
    (dict(gate=FAKE + 2), _abi.QSA_ERR_INVALID_ARG),
    (dict(ids=None), _abi.QSA_ERR_INVALID_ARG),
    (dict(out=FAKE + 2), _abi.QSA_ERR_INVALID_ARG),
    (dict(kq=FAKE + 8), _abi.QSA_ERR_INVALID_ARG),
    (dict(cache_cells=0), _abi.QSA_ERR_INVALID_ARG),
    (dict(softmax_scale=float("inf")), _abi.QSA_ERR_INVALID_ARG),
    (dict(ntok=-1), _abi.QSA_ERR_INVALID_ARG),
])
def test_attn_rejects(L, kw, want):
    s, msg = _status(L, "qsa_attn", _attn(**kw))
    assert s == want and msg.startswith("qsa_attn")


def test_attn_zero_tokens_is_a_no_op(L):
    assert _status(L, "qsa_attn", _attn(ntok=0, q=None, out=None))[0] == _abi.QSA_OK


def _score(**kw):
    a = _abi.ScoreArgs(ntok=64, pos0=10, n_q_heads=12, head_dim=128, group=32, cache_cells=74, q=FAKE,
                       q_dtype=_abi.QSA_F32, kq=FAKE, ksc=FAKE, scores=FAKE, ld=74, workspace=FAKE,
                       workspace_bytes=1 << 20, err=None)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,want", [
    (dict(cache_cells=73), _abi.QSA_ERR_INVALID_ARG),
    (dict(ld=73), _abi.QSA_ERR_INVALID_ARG),
    (dict(q_dtype=7), _abi.QSA_ERR_INVALID_ARG),
    (dict(workspace_bytes=100), _abi.QSA_ERR_INVALID_ARG),
    (dict(workspace=FAKE + 16), _abi.QSA_ERR_INVALID_ARG),
    (dict(workspace=None), _abi.QSA_ERR_INVALID_ARG),
    (dict(head_dim=64), _abi.QSA_ERR_UNSUPPORTED),
    (dict(n_q_heads=0), _abi.QSA_ERR_UNSUPPORTED),
    (dict(ksc=FAKE + 2), _abi.QSA_ERR_INVALID_ARG),
])
def test_score_rejects(L, kw, want):
    s, msg = _status(L, "qsa_score", _score(**kw))
    assert s == want and msg.startswith("qsa_score")


def _prep(**kw):
    a = _abi.PrepArgs(ntok=8, pos0=3000, n_q_heads=12, n_kv_heads=1, head_dim=128, group=32, rope_dims=64,
                      cache_cells=3008, eps=1e-6, rope_theta=10000.0, q_in=FAKE, k_in=FAKE, v_in=FAKE,
                      norm_w=FAKE, q_out=FAKE, q_out_f32=None, kq=FAKE, vq=FAKE, ksc=FAKE, vsc=FAKE)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,want", [
    (dict(cache_cells=3007), _abi.QSA_ERR_INVALID_ARG),
    (dict(rope_dims=60), _abi.QSA_ERR_UNSUPPORTED),
    (dict(rope_dims=136), _abi.QSA_ERR_UNSUPPORTED),
    (dict(n_kv_heads=2), _abi.QSA_ERR_UNSUPPORTED),
    (dict(eps=-1.0), _abi.QSA_ERR_INVALID_ARG),
    (dict(q_in=FAKE + 4), _abi.QSA_ERR_INVALID_ARG),
    (dict(vsc=None), _abi.QSA_ERR_INVALID_ARG),
    (dict(pos0=(1 << 29) - 4, cache_cells=1 << 30), _abi.QSA_ERR_INVALID_ARG),
])
def test_prep_rejects(L, kw, want):
    s, msg = _status(L, "qsa_prep", _prep(**kw))
    assert s == want and msg.startswith("qsa_prep")


def test_null_args_pointer(L):
    for fn in ("qsa_prep", "qsa_score", "qsa_attn"):
        assert getattr(L, fn)(None, None) == _abi.QSA_ERR_INVALID_ARG


def _select(**kw):
    a = _abi.SelectArgs(ntok=8, pos0=3000, width=2048, budget=2048, sink=64, local=256, scores=FAKE, ld=3008,
                        ids=FAKE)
    for k, v in kw.items():
        setattr(a, k, v)
    return a


@pytest.mark.parametrize("kw,want", [
    (dict(width=2000), _abi.QSA_ERR_INVALID_ARG),
    (dict(budget=4096), _abi.QSA_ERR_INVALID_ARG),
    (dict(budget=0), _abi.QSA_ERR_INVALID_ARG),
    (dict(ld=3007), _abi.QSA_ERR_INVALID_ARG),
    (dict(pos0=40000, ld=40008), _abi.QSA_ERR_UNSUPPORTED),
    (dict(width=256, budget=256), _abi.QSA_ERR_INVALID_ARG),
    (dict(ids=None), _abi.QSA_ERR_INVALID_ARG),
    (dict(scores=FAKE + 2), _abi.QSA_ERR_INVALID_ARG),
])
def test_select_rejects(L, kw, want):
    s, msg = _status(L, "qsa_select", _select(**kw))
    assert s == want and msg.startswith("qsa_select")


def test_score_and_prep_head_sum_flags_rejected(L):
    a = _abi.ScoreArgs(ntok=4, pos0=10, n_q_heads=12, head_dim=128, group=32, cache_cells=100, q=FAKE, q_dtype=0,
                       kq=FAKE, ksc=FAKE, scores=FAKE, ld=20, workspace=FAKE, workspace_bytes=1 << 20, err=None,
                       workspace_holds_qbar=2)
    s, msg = _status(L, "qsa_score", a)
    assert s == _abi.QSA_ERR_INVALID_ARG and "workspace_holds_qbar" in msg
    p = _abi.PrepArgs(ntok=4, pos0=10, n_q_heads=12, n_kv_heads=1, head_dim=128, group=32, rope_dims=64,
                      cache_cells=100, eps=1e-6, rope_theta=1e4, q_in=FAKE, k_in=FAKE, v_in=FAKE, norm_w=FAKE,
                      q_out=FAKE, q_out_f32=None, kq=FAKE, vq=FAKE, ksc=FAKE, vsc=FAKE, rope_k=0, qbar_out=FAKE + 16)
    s, msg = _status(L, "qsa_prep", p)
    assert s == _abi.QSA_ERR_INVALID_ARG and "qbar_out" in msg


@pytest.mark.parametrize("fn", ["qsa_score", "qsa_score_noalloc"])
def test_score_rejects_negative_max_ctas(L, fn):
    a = _abi.ScoreArgs(ntok=4, pos0=10, n_q_heads=12, head_dim=128, group=32, cache_cells=100, q=FAKE, q_dtype=0,
                       kq=FAKE, ksc=FAKE, scores=FAKE, ld=20, workspace=FAKE, workspace_bytes=1 << 20, err=None,
                       workspace_holds_qbar=0, max_ctas=-1)
    s, msg = _status(L, fn, a)
    assert s == _abi.QSA_ERR_INVALID_ARG and "max_ctas" in msg


@pytest.mark.parametrize("args", [
    (4, 100, 320, 64, 256, FAKE),      # width below sink + local + 1
    (4, -1, 384, 64, 256, FAKE),
    (4, 100, 384, -1, 256, FAKE),
    (4, 100, 384, 64, 256, None),
    (4, 100, 384, 64, 256, FAKE + 2),
])
def test_fill_ids_decode_rejects(L, args):
    import torch
    if torch.cuda.is_available():
        pytest.skip("argument-rejection checks use fake device addresses: run them on a machine without a GPU")
    assert L.qsa_fill_ids_decode(*args, None) == _abi.QSA_ERR_INVALID_ARG
    assert L.qsa_last_error().decode().startswith("qsa_fill_ids_decode")


@pytest.mark.parametrize("args", [
    (4, 100, 2048, 1, FAKE),           # select below 2
    (4, 100, 1024, 2048, FAKE),        # select above width
    (4, -5, 2048, 2048, FAKE),
    (4, 100, 2048, 2048, None),
])
def test_fill_ids_even_rejects(L, args):
    import torch
    if torch.cuda.is_available():
        pytest.skip("argument-rejection checks use fake device addresses: run them on a machine without a GPU")
    assert L.qsa_fill_ids_even(*args, None) == _abi.QSA_ERR_INVALID_ARG
    assert L.qsa_last_error().decode().startswith("qsa_fill_ids_even")


def test_fill_ids_zero_tokens_is_a_no_op(L):
    assert L.qsa_fill_ids_even(0, 0, 64, 64, None, None) == _abi.QSA_OK
    assert L.qsa_fill_ids_decode(0, 0, 384, 64, 256, None, None) == _abi.QSA_OK


def test_check_word_needs_the_check_build(L):
    out = ctypes.c_uint(7)
    assert L.qsa_check_word(ctypes.byref(out)) == _abi.QSA_ERR_UNSUPPORTED and out.value == 0
    assert L.qsa_check_word(None) == _abi.QSA_ERR_INVALID_ARG
