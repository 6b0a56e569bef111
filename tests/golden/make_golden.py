"""Writes tests/golden/oracle_regression.json from the oracle alone.

The pages print no worked values, so this fixture is a regression record of
the pinned oracle on tiny seeded inputs: it guards the oracle against
unintended changes.  It calls only oracle/ and the seeded input recipes.
Run from the repository root:  python tests/golden/make_golden.py
"""
import json
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from oracle import attention, prep_queries, quantize_rows, rotate_keys_f32, score, select_ids  # noqa: E402
from sparse_selected_attention_gb300 import workloads as wl  # noqa: E402


def build():
    inp = wl.prep_inputs(2, seed=21)
    q64, q16, _ = prep_queries(inp.q_in, inp.norm_w, pos0=30000)
    codes, scales = quantize_rows(inp.k_in.reshape(2, -1))
    cache = wl.make_cache(70, seed=21)
    qs = wl.queries_f32(2, seed=21)
    S = score(qs, cache.kq, cache.ksc, pos0=68)
    qa = wl.queries_f16(2, seed=21)
    ids = wl.even_ids(2, 68, width=128, select=40)
    out64, out16, _, _ = attention(qa, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 1.0 / math.sqrt(128.0))
    # the gate, the pages' shape (2 KV heads, d = 256, per-64 scales), key
    # rotation before quantising, and the selection
    gate = wl.gates_f32(2, seed=21)
    g64, _, _, _ = attention(qa, cache.kq, cache.vq, cache.ksc, cache.vsc, ids, 1.0 / math.sqrt(128.0), gate=gate)
    pc = wl.make_cache(70, seed=22, head_dim=256, group=64, kv_heads=2)
    pq = wl.queries_f16(2, seed=22, heads=24, head_dim=256)
    p64, _, _, _ = attention(pq, pc.kq, pc.vq, pc.ksc, pc.vsc, ids, 0.0625, group=64)
    rk_codes, rk_scales = quantize_rows(rotate_keys_f32(inp.k_in, 30000).reshape(2, -1))
    sc = wl.normal(23, 1, (3, 3003)).astype(np.float32)
    sel = select_ids(sc, 3000, width=384, budget=330)
    return {
        "inputs": "workloads.prep_inputs(2, seed=21) at pos0=30000; make_cache(70, seed=21); "
                  "queries_f32/f16(2, seed=21); even_ids(2, 68, width=128, select=40); gates_f32(2, seed=21); "
                  "pages' shape make_cache(70, seed=22, d=256, group=64, 2 KV heads), queries_f16(2, seed=22, "
                  "24 heads); selection over normal(23, 1, (3, 3003)) at pos0=3000, width 384, budget 330",
        "prep_q_f64_t1_h5_d0_8": q64[1, 5, :8].tolist(),
        "prep_q_f16_bits_t0_h0_d60_68": q16[0, 0, 60:68].view(np.uint16).tolist(),
        "quant_codes_t1_d0_16": codes[1, :16].tolist(),
        "quant_scale_bits_t1": scales[1].view(np.uint16).tolist(),
        "score_t1_c60_70": S[1, 60:70].tolist(),
        "attn_f64_t1_h11_d120_128": out64[1, 11, 120:128].tolist(),
        "attn_f16_bits_t0_h3_d0_8": out16[0, 3, :8].view(np.uint16).tolist(),
        "attn_gated_f64_t1_h7_d0_8": g64[1, 7, :8].tolist(),
        "attn_pages_shape_f64_t0_h17_d248_256": p64[0, 17, 248:256].tolist(),
        "rope_k_codes_t1_d24_40": rk_codes[1, 24:40].tolist(),
        "rope_k_scale_bits_t1": rk_scales[1].view(np.uint16).tolist(),
        "select_ids_t2_free_part": sel[2, 64:73].tolist(),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(build(), f, indent=1)
    print("wrote", path)
