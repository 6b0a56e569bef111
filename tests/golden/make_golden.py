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

from oracle import attention, prep_queries, quantize_rows, score  # noqa: E402
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
    return {
        "inputs": "workloads.prep_inputs(2, seed=21) at pos0=30000; make_cache(70, seed=21); "
                  "queries_f32/f16(2, seed=21); even_ids(2, 68, width=128, select=40)",
        "prep_q_f64_t1_h5_d0_8": q64[1, 5, :8].tolist(),
        "prep_q_f16_bits_t0_h0_d60_68": q16[0, 0, 60:68].view(np.uint16).tolist(),
        "quant_codes_t1_d0_16": codes[1, :16].tolist(),
        "quant_scale_bits_t1": scales[1].view(np.uint16).tolist(),
        "score_t1_c60_70": S[1, 60:70].tolist(),
        "attn_f64_t1_h11_d120_128": out64[1, 11, 120:128].tolist(),
        "attn_f16_bits_t0_h3_d0_8": out16[0, 3, :8].view(np.uint16).tolist(),
    }


if __name__ == "__main__":
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_regression.json")
    with open(path, "w") as f:
        json.dump(build(), f, indent=1)
    print("wrote", path)
