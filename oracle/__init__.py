"""CPU oracle for parallel constrained decoding -- test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg use this
package.  The library's compute path never imports it, and it shares no code
with the CUDA path.
"""
from .pcd_oracle import (  # noqa: F401
    Oracle, KVCache, FieldResult,
    rms_norm, rope_cos_sin, apply_rope, attention, silu, swiglu,
    logsumexp64, scores_to_result, combine_spellings, first_token_result,
    length_normalised_scores, per_level_scores, field_scores, SCORINGS,
    kv_bytes_per_token,
)
