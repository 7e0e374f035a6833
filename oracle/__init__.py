"""CPU oracle (test infrastructure only): see sampler_oracle and sampling_oracle."""
from .sampler_oracle import (bf16_bits_to_f64, entropy_accept, row_stats, soft_embed,
                             sum_partials)
from .sampling_oracle import philox4x32_10, row_sample, uniforms

__all__ = ["bf16_bits_to_f64", "entropy_accept", "row_stats", "soft_embed", "sum_partials",
           "philox4x32_10", "row_sample", "uniforms"]
