"""fp64 CPU oracle for one MLA decode step — test infrastructure only.

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. The CUDA library never calls it and shares no code with it.
"""
from .mla import (  # noqa: F401
    rope_inv_freq, rope, cache_rows, absorbed_query, latent_attention,
    output_projection, decode_materialised, decode_absorbed, scale_of,
    per_token_cache_elems, rms_norm, premerged_query_weights, premerged_output_weights,
    materialised_kv, materialised_query, mha_attention, prefill_materialised,
)
