"""Seeded synthetic inputs for the QSA attention hot path.

This module holds the input recipes only: random draws, the structure of the
selected-id lists and the named workload shapes.  It contains none of the
method's arithmetic (no normalisation, rotation, quantisation, scoring or
softmax), so the CUDA path and the CPU oracle can both consume its output
without sharing any of the computation they are compared on.

Random numbers come from a counter-based SplitMix64 generator (Steele, Lea and
Flood, "Fast splittable pseudorandom number generators", OOPSLA 2014) written
out here, so a seed gives the same integers on every platform and numpy
version.  Floating-point draws are derived from those integers (uniforms by
the top 53 bits, normals by the Box-Muller transform).

Workload shapes follow the audit pages on sparse selected attention: a
12-query-head / 1-KV-head layout with head_dim 128 and one fp16 scale per
32-dim group; decode windows of 64 sink + 256 local + 1 current cell
("sol_r5_mtp_qsa", mtp attention section); prompt lists of evenly spaced
unique causal cells padded with -1 ("sol_r11_qsa", boundaries and provenance).
"""
from __future__ import annotations

import dataclasses

import numpy as np

# SplitMix64 constants (golden-ratio increment and the two mixing multipliers).
_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_MIX1 = np.uint64(0xBF58476D1CE4E5B9)
_MIX2 = np.uint64(0x94D049BB133111EB)

N_Q_HEADS = 12
N_KV_HEADS = 1
HEAD_DIM = 128
GROUP = 32
SINK = 64
LOCAL = 256
DECODE_WIDTH = 384
PROMPT_SELECT = 2048


def _mix(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _MIX1
    z = (z ^ (z >> np.uint64(27))) * _MIX2
    return z ^ (z >> np.uint64(31))


def _stream_key(seed: int, stream: int) -> np.uint64:
    base = np.array([(int(seed) & 0xFFFFFFFF) << 16 | (int(stream) & 0xFFFF)], dtype=np.uint64)
    return _mix(base * _GAMMA + _GAMMA)[0]


def random_u64(seed: int, stream: int, n: int) -> np.ndarray:
    """n SplitMix64 outputs of the (seed, stream) sequence."""
    key = _stream_key(seed, stream)
    with np.errstate(over="ignore"):
        ctr = (np.arange(1, n + 1, dtype=np.uint64) * _GAMMA) + key
        return _mix(ctr)


def uniform(seed: int, stream: int, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    n = int(np.prod(shape))
    u = (random_u64(seed, stream, n) >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return (lo + (hi - lo) * u).reshape(shape)


def normal(seed: int, stream: int, shape) -> np.ndarray:
    n = int(np.prod(shape))
    m = (n + 1) // 2
    u = uniform(seed, stream, (2 * m,))
    u1 = 1.0 - u[:m]  # (0, 1]
    u2 = u[m:]
    r = np.sqrt(-2.0 * np.log(u1))
    z = np.concatenate([r * np.cos(2.0 * np.pi * u2), r * np.sin(2.0 * np.pi * u2)])
    return z[:n].reshape(shape)


def int8_uniform(seed: int, stream: int, shape) -> np.ndarray:
    """Integers uniform on [-127, 127] (the cache's code range)."""
    u = uniform(seed, stream, shape)
    return (np.floor(u * 255.0) - 127.0).astype(np.int8)


# Stream numbers: one per drawn tensor, so changing one shape leaves the others.
_S_KQ, _S_VQ, _S_KSC, _S_VSC, _S_Q16, _S_Q32, _S_QIN, _S_KIN, _S_VIN, _S_G, _S_EDGE, _S_GATE = range(1, 13)


@dataclasses.dataclass
class Cache:
    """An int8 K/V cache with one fp16 scale per (cell, 32-dim group)."""

    kq: np.ndarray   # int8 [C, D]
    vq: np.ndarray   # int8 [C, D]
    ksc: np.ndarray  # float16 [C, D // GROUP]
    vsc: np.ndarray  # float16 [C, D // GROUP]

    @property
    def cells(self) -> int:
        return self.kq.shape[0]

    def copy(self) -> "Cache":
        return Cache(self.kq.copy(), self.vq.copy(), self.ksc.copy(), self.vsc.copy())


def make_cache(cells: int, seed: int = 5, head_dim: int = HEAD_DIM, group: int = GROUP,
               scale_lo: float = 1e-3, scale_hi: float = 2e-2, kv_heads: int = 1) -> Cache:
    """Cache of `cells` rows: codes uniform on [-127,127], scales fp16(U[lo,hi]).
    One KV head: kq/vq [cells, D], scales [cells, D/group]; more: kq/vq
    [cells, kv_heads, D], scales [cells, kv_heads, D/group]."""
    ng = head_dim // group
    row = (cells, head_dim) if kv_heads == 1 else (cells, kv_heads, head_dim)
    srow = (cells, ng) if kv_heads == 1 else (cells, kv_heads, ng)
    return Cache(
        kq=int8_uniform(seed, _S_KQ, row),
        vq=int8_uniform(seed, _S_VQ, row),
        ksc=uniform(seed, _S_KSC, srow, scale_lo, scale_hi).astype(np.float16),
        vsc=uniform(seed, _S_VSC, srow, scale_lo, scale_hi).astype(np.float16),
    )


# The pages' own attention shape ("round 5 track b: cached residual norms and
# fused mtp attention", section "mtp attention": two KV heads per token, 24
# heads of 256 + 2 partial floats, fp16 per-64 scales, seed 20260701) and
# the matching softmax scale 1/sqrt(256).
PAGES_KV_HEADS, PAGES_Q_HEADS, PAGES_HEAD_DIM, PAGES_GROUP = 2, 24, 256, 64
PAGES_SCALE = 0.0625
PAGES_SEED = 20260701


def gates_f32(ntok: int, seed: int = 5, heads: int = N_Q_HEADS, head_dim: int = HEAD_DIM) -> np.ndarray:
    """fp32 output-gate logits, 2 * N(0,1) (so some saturate). [ntok, heads, D]."""
    return (2.0 * normal(seed, _S_GATE, (ntok, heads, head_dim))).astype(np.float32)


def queries_f16(ntok: int, seed: int = 5, heads: int = N_Q_HEADS, head_dim: int = HEAD_DIM) -> np.ndarray:
    """fp16 attention queries, fp16 round-to-nearest of N(0,1) draws. [ntok, heads, D]."""
    return normal(seed, _S_Q16, (ntok, heads, head_dim)).astype(np.float16)


def queries_f32(ntok: int, seed: int = 5, heads: int = N_Q_HEADS, head_dim: int = HEAD_DIM) -> np.ndarray:
    """fp32 score-pass queries, N(0,1). [ntok, heads, D]."""
    return normal(seed, _S_Q32, (ntok, heads, head_dim)).astype(np.float32)


@dataclasses.dataclass
class PrepInputs:
    q_in: np.ndarray    # fp32 [T, Hq, D]
    k_in: np.ndarray    # fp32 [T, Hkv, D]
    v_in: np.ndarray    # fp32 [T, Hkv, D]
    norm_w: np.ndarray  # fp32 [D]


def prep_inputs(ntok: int, seed: int = 5, heads: int = N_Q_HEADS, kv_heads: int = N_KV_HEADS,
                head_dim: int = HEAD_DIM) -> PrepInputs:
    """Un-normalised fp32 rows N(0,1) and an RMS-norm weight U[0.5, 1.5]."""
    return PrepInputs(
        q_in=normal(seed, _S_QIN, (ntok, heads, head_dim)).astype(np.float32),
        k_in=normal(seed, _S_KIN, (ntok, kv_heads, head_dim)).astype(np.float32),
        v_in=normal(seed, _S_VIN, (ntok, kv_heads, head_dim)).astype(np.float32),
        norm_w=uniform(seed, _S_G, (head_dim,), 0.5, 1.5).astype(np.float32),
    )


def decode_ids(ntok: int, pos0: int, width: int = DECODE_WIDTH, sink: int = SINK,
               local: int = LOCAL) -> np.ndarray:
    """Per-token decode window: sink cells, the previous `local` cells and the
    token's own cell p = pos0 + t, ascending and causal, then -1 up to `width`."""
    ids = np.full((ntok, width), -1, dtype=np.int32)
    for t in range(ntok):
        p = pos0 + t
        cells = sorted(set(range(0, min(sink, p))) | set(range(max(sink, p - local), p)) | {p})
        if len(cells) > width:
            raise ValueError("decode window wider than the id list")
        ids[t, : len(cells)] = cells
    return ids


def even_ids(ntok: int, pos0: int, width: int = PROMPT_SELECT, select: int = PROMPT_SELECT) -> np.ndarray:
    """Per-token prompt list: up to `select` evenly spaced unique causal cells of
    0..p (p = pos0 + t), always containing 0 and p, ascending, then -1."""
    ids = np.full((ntok, width), -1, dtype=np.int32)
    for t in range(ntok):
        n = pos0 + t + 1
        k = min(n, select)
        if k > width:
            raise ValueError("selection wider than the id list")
        if k == n:
            ids[t, :k] = np.arange(n, dtype=np.int64)
        else:
            j = np.arange(k, dtype=np.int64)
            ids[t, :k] = (j * (n - 1)) // (k - 1)
    return ids


def edge_signed_zero(q: np.ndarray) -> np.ndarray:
    """Signed-zero edge mode: tokens t = 0 (mod 7) get q = +0 and tokens
    t = 3 (mod 7) get q = -0 on every head."""
    q = q.copy()
    q[0::7] = np.float16(0.0)
    q[3::7] = np.float16(-0.0)
    return q


def edge_cancellation(q: np.ndarray, cache: Cache, seed: int = 5):
    """Tiny-cancellation edge mode: for tokens t = 5 (mod 7) the second half of
    each query head is minus the first half plus fp16(1e-3 N(0,1)); every
    cache row repeats its first 64 key codes and first two key scales in its
    second half, so those tokens' dot products nearly cancel."""
    q = q.copy()
    cache = cache.copy()
    half = q.shape[-1] // 2
    sel = q[5::7]
    noise = (1e-3 * normal(seed, _S_EDGE, sel[..., :half].shape)).astype(np.float16)
    sel[..., half:] = (-sel[..., :half].astype(np.float32) + noise.astype(np.float32)).astype(np.float16)
    q[5::7] = sel
    cache.kq[:, half:] = cache.kq[:, :half]
    ng = cache.ksc.shape[1]
    cache.ksc[:, ng // 2:] = cache.ksc[:, : ng // 2]
    return q, cache


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    ntok: int
    pos0: int
    width: int
    ids: str          # "decode" | "even" | "none"
    seed: int = 5

    @property
    def cells(self) -> int:
        return self.pos0 + self.ntok

    def make_ids(self) -> np.ndarray:
        if self.ids == "decode":
            return decode_ids(self.ntok, self.pos0, self.width)
        if self.ids == "even":
            return even_ids(self.ntok, self.pos0, self.width)
        raise ValueError(self.ids)


# The five workloads the method is specified on (names describe the shapes).
TINY_DECODE = Workload("tiny decode: ntok=1 pos0=320 W=384", 1, 320, DECODE_WIDTH, "decode")
MTP_DECODE = Workload("MTP decode window: ntok=8 pos0=30000 W=384", 8, 30000, DECODE_WIDTH, "decode")
PROMPT_SHORT = Workload("prompt attention short context: T=1984 pos0=0 W=2048", 1984, 0, PROMPT_SELECT, "even")
PROMPT_LONG = Workload("prompt attention long context: T=1984 pos0=30000 W=2048", 1984, 30000, PROMPT_SELECT, "even")
SCORE_POS0 = (0, 2048, 8192, 30000)
SCORE_NTOK = 1984
