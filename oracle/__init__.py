"""Float64 CPU oracle of the SP-TP FFN boundary (test infrastructure only)."""
from .sptp_oracle import (dtp_ffn_stack_forward, reduce_partials, rel_max_error, rms_norm,
                          shard_ffn, silu, sptp_ffn_forward)

__all__ = ["dtp_ffn_stack_forward", "reduce_partials", "rel_max_error", "rms_norm",
           "shard_ffn", "silu", "sptp_ffn_forward"]
