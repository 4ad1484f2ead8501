"""Float64 CPU oracle (test infrastructure only; never part of the product path)."""
from .verify_ref import (  # noqa: F401
    bf16_bits_to_f64,
    e4m3_bits_to_f64,
    gate_factor,
    gather_latent_rows,
    ref_attention_partials,
    ref_greedy_verify,
    ref_kv_append,
    ref_lse_combine,
    ref_verify_attention,
    ref_verify_step,
    ref_wuv_project,
    sigmoid,
)
from .sampled_ref import inverse_cdf, ref_sampled_verify, target_probs  # noqa: F401
