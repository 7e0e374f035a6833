"""CPU oracle (test infrastructure only): see sampler_oracle, sampling_oracle, loop_oracle,
partition_oracle and quant_oracle."""
from .sampler_oracle import (bf16_bits_to_f64, entropy_accept, row_stats, soft_embed,
                             sum_partials)
from .sampling_oracle import candidate_kappa, philox4x32_10, row_sample, uniforms
from .loop_oracle import entropy_accept_eligible, loop_update, new_loop_state
from .partition_oracle import row_stats_combine, row_stats_partial
from .quant_oracle import (dequantize_rows_e4m3, e4m3_decode, e4m3_round, quantize_rows_e4m3,
                           soft_embed_e4m3)

__all__ = ["bf16_bits_to_f64", "entropy_accept", "row_stats", "soft_embed", "sum_partials",
           "candidate_kappa", "philox4x32_10", "row_sample", "uniforms",
           "entropy_accept_eligible", "loop_update", "new_loop_state",
           "row_stats_combine", "row_stats_partial",
           "dequantize_rows_e4m3", "e4m3_decode", "e4m3_round", "quantize_rows_e4m3", "soft_embed_e4m3"]
