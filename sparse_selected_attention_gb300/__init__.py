"""GB300-native QSA (sparse selected attention) hot path.

Python binding of the C ABI in include/qsa.h: each function marshals torch
CUDA tensors into the argument struct and calls the library on the current
CUDA stream.  All computation runs in libqsa.so's kernels; tensors on the CPU
are rejected rather than computed elsewhere.

    qsa_prep   query RMS-norm + RoPE, K/V int8 quantisation into the cache
    qsa_score  head-reduced fp32 scores of every causal cache cell
    qsa_select per-token selected cell ids from the scores
    qsa_attn   chunked attention over per-token selected cell ids
    qsa_fill_ids_decode / qsa_fill_ids_even  the workloads' id lists, on the device
"""
from __future__ import annotations

import ctypes
import math

from . import _abi
from ._abi import (QSA_DEVERR_BAD_ID, QSA_DEVERR_TIMEOUT, QSA_SCORE_NOALLOC_MAX_TOKENS,  # noqa: F401
                   QSA_SELECT_MAX_CELLS, QSAError, lib)

__all__ = ["qsa_prep", "qsa_score", "qsa_score_noalloc", "qsa_select", "qsa_attn", "qsa_score_workspace_bytes",
           "qsa_fill_ids_decode", "qsa_fill_ids_even", "qsa_abi_version",
           "QSAError", "QSA_DEVERR_BAD_ID", "QSA_DEVERR_TIMEOUT", "QSA_SCORE_NOALLOC_MAX_TOKENS",
           "QSA_SELECT_MAX_CELLS", "lib"]


def _ptr(t, name, dtype=None, optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the QSA path runs only on the GPU)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def qsa_abi_version() -> int:
    return lib().qsa_abi_version()


def qsa_score_workspace_bytes(ntok: int, head_dim: int = 128) -> int:
    return int(lib().qsa_score_workspace_bytes(ntok, head_dim))


def qsa_prep(q_in, k_in, v_in, norm_w, pos0, kq, vq, ksc, vsc, q_out, q_out_f32=None,
             eps=1e-6, rope_theta=10000.0, rope_dims=64, rope_k=False, qbar_out=None, stream=None):
    """Normalise + rotate q_in into q_out (fp16) / q_out_f32 and quantise k_in,
    v_in into cache rows pos0 .. pos0+ntok-1 (with rope_k, the key rows are
    rotated first).  Shapes: q_in [T, Hq, D] fp32, k_in / v_in [T, 1, D]
    fp32, norm_w [D], kq / vq [C, D] int8, ksc / vsc [C, D/32] fp16.
    qbar_out, if given, is a qsa_score workspace (qsa_score_workspace_bytes(T)
    bytes) that receives the score's head sum, for a qsa_score call with
    workspace_holds_qbar=True."""
    import torch
    T, H, D = q_in.shape
    a = _abi.PrepArgs(ntok=T, pos0=int(pos0), n_q_heads=H, n_kv_heads=k_in.shape[1], head_dim=D, group=32,
                      rope_dims=int(rope_dims), cache_cells=kq.shape[0], eps=float(eps),
                      rope_theta=float(rope_theta),
                      q_in=_ptr(q_in, "q_in", torch.float32), k_in=_ptr(k_in, "k_in", torch.float32),
                      v_in=_ptr(v_in, "v_in", torch.float32), norm_w=_ptr(norm_w, "norm_w", torch.float32),
                      q_out=_ptr(q_out, "q_out", torch.float16),
                      q_out_f32=_ptr(q_out_f32, "q_out_f32", torch.float32, optional=True),
                      kq=_ptr(kq, "kq", torch.int8), vq=_ptr(vq, "vq", torch.int8),
                      ksc=_ptr(ksc, "ksc", torch.float16), vsc=_ptr(vsc, "vsc", torch.float16),
                      rope_k=1 if rope_k else 0, qbar_out=_ptr(qbar_out, "qbar_out", optional=True))
    _abi.check(lib().qsa_prep(ctypes.byref(a), _stream(stream)))


def qsa_score(q, kq, ksc, pos0, scores, workspace, err=None, stream=None, workspace_holds_qbar=False,
              n_q_heads=12, max_ctas=0):
    """scores[t, c] for c <= pos0 + t (others untouched).  q [T, Hq, D] fp32 or
    fp16; scores [T, ld] fp32 with ld >= pos0 + T; workspace a uint8 CUDA
    tensor of at least qsa_score_workspace_bytes(T) bytes.  With
    workspace_holds_qbar=True the workspace was filled by qsa_prep(qbar_out=)
    for these tokens and q may be None (T is then scores.shape[0]).
    max_ctas > 0 caps the persistent CTAs (one per SM when 0), leaving the
    other SMs to kernels on other streams."""
    import torch
    if q is None:
        if not workspace_holds_qbar:
            raise ValueError("q is required unless the workspace holds the head sum")
        T, H, D = scores.shape[0], int(n_q_heads), 128
        qp, qdt = None, _abi.QSA_F32
    else:
        T, H, D = q.shape
        if q.dtype not in (torch.float32, torch.float16):
            raise ValueError("q must be float32 or float16")
        qp, qdt = _ptr(q, "q"), (_abi.QSA_F16 if q.dtype == torch.float16 else _abi.QSA_F32)
    if scores.dim() != 2 or scores.shape[0] < T:
        raise ValueError("scores must be [T, ld]")
    a = _abi.ScoreArgs(ntok=T, pos0=int(pos0), n_q_heads=H, head_dim=D, group=32, cache_cells=kq.shape[0],
                       q=qp, q_dtype=qdt, workspace_holds_qbar=1 if workspace_holds_qbar else 0,
                       kq=_ptr(kq, "kq", torch.int8), ksc=_ptr(ksc, "ksc", torch.float16),
                       scores=_ptr(scores, "scores", torch.float32), ld=scores.shape[1],
                       workspace=_ptr(workspace, "workspace"),
                       workspace_bytes=workspace.numel() * workspace.element_size(),
                       err=_ptr(err, "err", torch.int32, optional=True), max_ctas=int(max_ctas))
    _abi.check(lib().qsa_score(ctypes.byref(a), _stream(stream)))


def qsa_score_noalloc(q, kq, ksc, pos0, scores, err=None, stream=None, max_ctas=0):
    """qsa_score without a caller workspace, for callers that cannot allocate
    device memory when they score.  It uses the library's built-in scratch
    (at most 8192 tokens), so calls must not overlap on the GPU."""
    import torch
    T, H, D = q.shape
    if q.dtype not in (torch.float32, torch.float16):
        raise ValueError("q must be float32 or float16")
    if scores.dim() != 2 or scores.shape[0] < T:
        raise ValueError("scores must be [T, ld]")
    a = _abi.ScoreArgs(ntok=T, pos0=int(pos0), n_q_heads=H, head_dim=D, group=32, cache_cells=kq.shape[0],
                       q=_ptr(q, "q"), q_dtype=_abi.QSA_F16 if q.dtype == torch.float16 else _abi.QSA_F32,
                       kq=_ptr(kq, "kq", torch.int8), ksc=_ptr(ksc, "ksc", torch.float16),
                       scores=_ptr(scores, "scores", torch.float32), ld=scores.shape[1],
                       workspace=None, workspace_bytes=0, err=_ptr(err, "err", torch.int32, optional=True),
                       max_ctas=int(max_ctas))
    _abi.check(lib().qsa_score_noalloc(ctypes.byref(a), _stream(stream)))


def qsa_select(scores, pos0, ids, budget=2048, sink=64, local=256, stream=None):
    """ids [T, W] int32 <- the forced decode window plus the top-scoring causal
    cells of each row of scores [T, ld] fp32 (ties to the lower id), ascending,
    -1 padded."""
    import torch
    T = ids.shape[0]
    if scores.dim() != 2 or scores.shape[0] < T:
        raise ValueError("scores must be [T, ld]")
    a = _abi.SelectArgs(ntok=T, pos0=int(pos0), width=ids.shape[1], budget=int(budget), sink=int(sink),
                        local=int(local), scores=_ptr(scores, "scores", torch.float32), ld=scores.shape[1],
                        ids=_ptr(ids, "ids", torch.int32))
    _abi.check(lib().qsa_select(ctypes.byref(a), _stream(stream)))


def qsa_fill_ids_decode(ids, pos0, sink=64, local=256, stream=None):
    """ids [T, W] int32 <- each token's decode window (sink cells, the
    previous `local` cells, its own cell p = pos0 + t), ascending, -1 padded."""
    import torch
    T, W = ids.shape
    _abi.check(lib().qsa_fill_ids_decode(T, int(pos0), W, int(sink), int(local),
                                         _ptr(ids, "ids", torch.int32), _stream(stream)))


def qsa_fill_ids_even(ids, pos0, select=2048, stream=None):
    """ids [T, W] int32 <- up to `select` evenly spaced causal cells of each
    token (always 0 and p = pos0 + t), ascending, -1 padded."""
    import torch
    T, W = ids.shape
    _abi.check(lib().qsa_fill_ids_even(T, int(pos0), W, int(select), _ptr(ids, "ids", torch.int32),
                                       _stream(stream)))


def qsa_attn(q, kq, vq, ksc, vsc, ids, out, softmax_scale=None, part=None, err=None, gate=None, stream=None):
    """Chunked attention of q [T, Hq, D] fp16 over ids [T, W] int32 (-1 =
    padding, W a multiple of 64) into out [T, Hq, D] fp16.  kq/vq are
    [cells, D] (one KV head) or [cells, Hkv, D] int8, scales [cells, (Hkv,)
    4] fp16; D is 128 (32-dim groups) or 256 (64-dim groups).  gate, if
    given, is [T, Hq, D] fp32 logits: out = fp16(O * sigmoid(gate)).  part,
    if given, is [T, W/64, Hq, D+2] fp32 and selects the split per-chunk +
    merge path."""
    import torch
    T, H, D = q.shape
    hkv = 1 if kq.dim() == 2 else kq.shape[1]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    a = _abi.AttnArgs(ntok=T, n_q_heads=H, n_kv_heads=hkv, head_dim=D, group=D // 4, cache_cells=kq.shape[0],
                      width=ids.shape[1], q=_ptr(q, "q", torch.float16), kq=_ptr(kq, "kq", torch.int8),
                      vq=_ptr(vq, "vq", torch.int8), ksc=_ptr(ksc, "ksc", torch.float16),
                      vsc=_ptr(vsc, "vsc", torch.float16), ids=_ptr(ids, "ids", torch.int32),
                      softmax_scale=float(softmax_scale), out=_ptr(out, "out", torch.float16),
                      part=_ptr(part, "part", torch.float32, optional=True),
                      err=_ptr(err, "err", torch.int32, optional=True),
                      gate=_ptr(gate, "gate", torch.float32, optional=True))
    _abi.check(lib().qsa_attn(ctypes.byref(a), _stream(stream)))
