"""fp64 CPU oracle (test infrastructure only; see ``mla_oracle``)."""
from .mla_oracle import (  # noqa: F401
    D_QK, D_V, LN2, LOG2E, LSE_BASE2, LSE_NATURAL, attend, bf16_to_f64, dcp_local_metadata,
    decode_full, decode_partial_causal,
    decode_partial, dequant_rows, e4m3_to_f64, f32_to_e4m3, gather_rows, kv_append, local_len,
    lse_combine, lse_to_base, lse_to_natural, owned_tokens,
)
