"""ctypes mirror of include/qsa.h and the loader of libqsa.so.

Only argument marshalling lives here: every step of the hot path runs in the
library's CUDA kernels.  A missing library is an error, never a fallback.
"""
from __future__ import annotations

import ctypes
import os
import re

_HERE = os.path.dirname(os.path.abspath(__file__))
# QSA_LIB names another build of the same library (the sanitizer tests load
# libqsa_asan.so this way); there is no fallback when it is missing.
LIB_PATH = os.environ.get("QSA_LIB") or os.path.join(_HERE, "libqsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "qsa.h")

QSA_OK, QSA_ERR_INVALID_ARG, QSA_ERR_UNSUPPORTED, QSA_ERR_CUDA = 0, 1, 2, 3
QSA_DEVERR_BAD_ID, QSA_DEVERR_TIMEOUT = 1, 2
QSA_F32, QSA_F16 = 0, 1
QSA_SCORE_NOALLOC_MAX_TOKENS = 8192
QSA_SELECT_MAX_CELLS = 32768

_c_int, _c_float, _vp = ctypes.c_int, ctypes.c_float, ctypes.c_void_p


class PrepArgs(ctypes.Structure):
    _fields_ = [("ntok", _c_int), ("pos0", _c_int), ("n_q_heads", _c_int), ("n_kv_heads", _c_int),
                ("head_dim", _c_int), ("group", _c_int), ("rope_dims", _c_int), ("cache_cells", _c_int),
                ("eps", _c_float), ("rope_theta", _c_float),
                ("q_in", _vp), ("k_in", _vp), ("v_in", _vp), ("norm_w", _vp),
                ("q_out", _vp), ("q_out_f32", _vp), ("kq", _vp), ("vq", _vp), ("ksc", _vp), ("vsc", _vp),
                ("rope_k", _c_int), ("qbar_out", _vp)]


class ScoreArgs(ctypes.Structure):
    _fields_ = [("ntok", _c_int), ("pos0", _c_int), ("n_q_heads", _c_int), ("head_dim", _c_int),
                ("group", _c_int), ("cache_cells", _c_int),
                ("q", _vp), ("q_dtype", _c_int), ("kq", _vp), ("ksc", _vp), ("scores", _vp),
                ("ld", ctypes.c_int64), ("workspace", _vp), ("workspace_bytes", ctypes.c_size_t), ("err", _vp),
                ("workspace_holds_qbar", _c_int), ("max_ctas", _c_int)]


class SelectArgs(ctypes.Structure):
    _fields_ = [("ntok", _c_int), ("pos0", _c_int), ("width", _c_int), ("budget", _c_int), ("sink", _c_int),
                ("local", _c_int), ("scores", _vp), ("ld", ctypes.c_int64), ("ids", _vp)]


class AttnArgs(ctypes.Structure):
    _fields_ = [("ntok", _c_int), ("n_q_heads", _c_int), ("n_kv_heads", _c_int), ("head_dim", _c_int),
                ("group", _c_int), ("cache_cells", _c_int), ("width", _c_int),
                ("q", _vp), ("kq", _vp), ("vq", _vp), ("ksc", _vp), ("vsc", _vp), ("ids", _vp),
                ("softmax_scale", _c_float), ("out", _vp), ("part", _vp), ("err", _vp), ("gate", _vp)]


class QSAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"QSA status {status}: {message}")
        self.status = status


ABI_VERSION = 3  # the struct layouts above
_lib = None


def _load(path: str) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m sparse_selected_attention_gb300.build --all` "
            "(the QSA path has no fallback)")
    L = ctypes.CDLL(path)
    _declare(L, path)
    return L


_variants = {}


def variant(name: str) -> ctypes.CDLL:
    """A test variant of the library (see build.VARIANTS), loaded beside the
    release one with its own symbols; its functions take the same structs."""
    if name not in _variants:
        from .build import lib_path
        _variants[name] = _load(lib_path(name))
    return _variants[name]


def lib() -> ctypes.CDLL:
    """The loaded libqsa.so; raises if it has not been built."""
    global _lib
    if _lib is None:
        _lib = _load(LIB_PATH)
    return _lib


def _declare(L: ctypes.CDLL, path: str) -> None:
    for name, argt in (("qsa_prep", PrepArgs), ("qsa_score", ScoreArgs), ("qsa_attn", AttnArgs),
                       ("qsa_score_noalloc", ScoreArgs), ("qsa_select", SelectArgs)):
        f = getattr(L, name)
        f.argtypes = [ctypes.POINTER(argt), _vp]
        f.restype = _c_int
    L.qsa_fill_ids_decode.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _vp, _vp]
    L.qsa_fill_ids_decode.restype = _c_int
    L.qsa_fill_ids_even.argtypes = [_c_int, _c_int, _c_int, _c_int, _vp, _vp]
    L.qsa_fill_ids_even.restype = _c_int
    L.qsa_check_word.argtypes = [_vp]
    L.qsa_check_word.restype = _c_int
    L.qsa_score_workspace_bytes.argtypes = [_c_int, _c_int]
    L.qsa_score_workspace_bytes.restype = ctypes.c_size_t
    L.qsa_status_str.argtypes = [_c_int]
    L.qsa_status_str.restype = ctypes.c_char_p
    L.qsa_last_error.argtypes = []
    L.qsa_last_error.restype = ctypes.c_char_p
    L.qsa_abi_version.argtypes = []
    L.qsa_abi_version.restype = _c_int
    if L.qsa_abi_version() != ABI_VERSION:
        raise RuntimeError(f"{path} has ABI version {L.qsa_abi_version()}, these bindings expect "
                           f"{ABI_VERSION}: rebuild it")


def check(status: int) -> None:
    if status != QSA_OK:
        L = lib()
        msg = (L.qsa_last_error() or b"").decode() or L.qsa_status_str(status).decode()
        raise QSAError(status, msg)


def header_functions(path: str = HEADER):
    """Names of the functions include/qsa.h declares."""
    with open(path) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_0-9]+)\s*\(", text)))
