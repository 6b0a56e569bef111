"""The algorithmic bytes and pairs behind bench.py's roofline figures, against
closed forms worked out by hand from the workload definitions (no GPU).

Attention moves 272 B per valid selected cell (128 + 128 int8 code bytes and
2 x 4 fp16 group scales), 4 B per id slot, and the fp16 q and output rows.
The score writes one fp32 value per causal (token, cell) pair.  Selection
reads every free causal score once and writes W ids per token.
"""
import numpy as np
import pytest

import bench
from sparse_selected_attention_gb300 import workloads as wl

T, W = 1984, 2048
QOUT = 2 * T * 12 * 128 * 2  # fp16 q in and fp16 out


def test_long_context_attention_bytes():
    ids = wl.even_ids(T, 30000, W)
    nbytes, valid = bench.attn_bytes(ids, T)
    assert valid == T * W                       # every token selects 2048 of its 30001+ cells
    assert nbytes == T * W * 272 + T * W * 4 + QOUT == 1_133_641_728


def test_short_context_attention_bytes():
    ids = wl.even_ids(T, 0, W)
    nbytes, valid = bench.attn_bytes(ids, T)
    assert valid == T * (T + 1) // 2 == 1_969_120  # token t sees cells 0..t
    assert nbytes == valid * 272 + T * W * 4 + QOUT


@pytest.mark.parametrize("pos0", [0, 2048, 8192, 30000])
def test_score_pairs(pos0):
    # token t (position pos0 + t) scores cells 0 .. pos0 + t
    assert bench.score_pairs(T, pos0) == sum(pos0 + t + 1 for t in range(T)) == T * pos0 + 1_969_120


def test_selection_bytes():
    # p = pos0 + t >= 320: the free range is [64, p - 256), p - 320 cells
    free = sum(p - 320 for p in range(30000, 30000 + T))
    assert free == 60_852_256
    assert bench.select_bytes(T, 30000) == 4 * free + 4 * T * W == 259_661_952
    # short rows: no free cells below p = 320
    assert bench.select_bytes(1, 100) == 4 * W


def test_pages_shape_attention_bytes():
    ids = wl.even_ids(T, 30000, W)
    nbytes, valid = bench.attn_bytes(ids, T, hkv=2, hq=24, d=256)
    per_cell = 2 * (2 * 256 + 2 * 4 * 2)        # two KV heads x (K and V codes + 4 scales each)
    assert per_cell == 1056
    assert nbytes == valid * per_cell + T * W * 4 + 2 * T * 24 * 256 * 2


def test_prep_bytes_per_token():
    per = 12 * 128 * (4 + 2) + 2 * 128 * 4 + 2 * (128 + 2 * 4)   # q in/out, k and v in, codes + scales out
    pad = -(-T // 64) * 64
    assert bench.prep_bytes(T) == T * per + pad * (2 * 128 * 2 + 4) + 128 * 4
    assert bench.prep_bytes(T) == pytest.approx(21.87e6, rel=1e-3)


def test_score_tiles_and_executed_flops():
    # pos0 = 0: token tile tt (tokens 128 tt .. 128 tt + 127) reaches cell
    # 128 tt + 127, i.e. tt + 1 cell tiles; the last tile (tokens 1920..1983)
    # reaches cell 1983, 16 cell tiles: 1 + 2 + ... + 15 + 16 = 136.
    assert bench.score_tiles(T, 0) == 136
    # pos0 = 30000: tile tt's last token sits at 30000 + 128 tt + 127, so
    # (30127 + 128 tt) // 128 + 1 = 235 + tt + 1 cell tiles for tt < 15
    # (30127 = 235 * 128 + 47) and (30000 + 1983) // 128 + 1 = 250 for the
    # last: 15 * 236 + (0 + 1 + ... + 14) + 250.
    assert bench.score_tiles(T, 30000) == 15 * 236 + 105 + 250 == 3895
    # three 128 x 128 x 128 fp16 products per tile, 2 flops per multiply-add
    assert bench.score_flops_executed(T, 30000) == 3895 * 3 * 2 * 128 ** 3


def test_score_bytes():
    # head sum: 1984 padded tokens x (2 fp16 rows of 128 + one int32 exponent);
    # cache: 31984 cells x (128 code bytes + 4 fp16 scales); scores: 4 B per
    # causal pair (1984 * 30000 + 1 + 2 + ... + 1984 = 61,489,120 pairs)
    assert bench.score_bytes(T, 30000, 31984) == 1984 * 516 + 31984 * 136 + 4 * 61_489_120 == 251_330_048
