"""CPU oracle for the QSA hot path: test infrastructure only (see qsa_oracle)."""
from .qsa_oracle import (attention, prep, prep_queries, quantize_rows, rope_inv_freq, rotate_keys_f32,  # noqa: F401
                         score, score_abs_bound, select_ids, CHUNK)
