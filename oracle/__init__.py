"""CPU oracle (test infrastructure only): see sampler_oracle."""
from .sampler_oracle import (bf16_bits_to_f64, entropy_accept, row_stats, soft_embed,
                             sum_partials)

__all__ = ["bf16_bits_to_f64", "entropy_accept", "row_stats", "soft_embed", "sum_partials"]
