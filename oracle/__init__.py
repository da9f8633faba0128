"""Float64 CPU oracle of the SP-TP FFN boundary (test infrastructure only)."""
from . import fp8_oracle
from .sptp_oracle import (attn_qkv_boundary, dtp_ffn_stack_forward, dtp_ffn_stack_forward_permuted,
                          permute_ffn_neurons, reduce_partials, rel_max_error, rms_norm, rowparallel_projection,
                          shard_ffn, silu, sptp_ffn_forward)

__all__ = ["fp8_oracle", "attn_qkv_boundary", "dtp_ffn_stack_forward", "dtp_ffn_stack_forward_permuted",
           "permute_ffn_neurons", "reduce_partials", "rel_max_error", "rms_norm", "rowparallel_projection",
           "shard_ffn", "silu", "sptp_ffn_forward"]
