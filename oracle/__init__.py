"""fp64 CPU oracle for paged varlen attention (test infrastructure only).

Only tests, the smoke check and the benchmark's CPU-baseline leg use this
package; the CUDA library never imports or links it.
"""
from .paged_attention import (  # noqa: F401
    reshape_and_cache,
    gather_kv,
    attend_dense,
    varlen_attention,
    merge_attn_states,
    merge_attn_states_n,
    dcp_decode_attention,
    cascade_attention,
    cascade_attention_steps,
    e4m3_decode,
    e4m3_encode,
    e4m3_round,
    quantize_e4m3,
    dequantize_e4m3,
    reshape_and_cache_e4m3,
    varlen_attention_e4m3,
)
