"""GB300-native speculative-decoding verify step for gated NoPE MLA.

The compute lives in ``libspecverify.so`` (hand-written sm_103a CUDA, C ABI in
``include/specverify.h``); this package is the thin Python binding.
"""
from .binding import (  # noqa: F401
    EXPORTED_SYMBOLS,
    SV_DEV_BAD_BOUND,
    SV_DEV_BAD_PAGE,
    SV_DEV_TIMEOUT,
    FORM_AUTO,
    FORM_STACKED,
    FORM_TWO_CTA,
    SV_SPLITS_BALANCED,
    SV_SPLITS_WAVE,
    SpecVerifyError,
    attention_workspace_bytes,
    greedy_workspace,
    greedy_workspace_bytes,
    load_library,
    mla_kv_append,
    mla_lse_combine,
    mla_verify_decode,
    mla_wuv_project,
    num_splits_for,
    sampled_workspace,
    sampled_workspace_bytes,
    spec_verify_greedy,
    spec_verify_sampled,
    status_string,
)
from .step import StagedInputs, VerifyStep  # noqa: F401
