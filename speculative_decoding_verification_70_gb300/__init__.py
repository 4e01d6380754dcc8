"""GB300-native verify-and-recover step of speculative decoding and of
Speculative Speculative Decoding (SSD).

The compute lives in libssd_gb300.so (C ABI: include/ssd.h, CUDA kernels for
sm_103a); this package is its thin Python binding plus the seeded synthetic
workloads.  Calls take CUDA torch tensors and run on the current stream.
"""
from ._binding import (  # noqa: F401
    DEVERR_BAD_LOGITS,
    DEVERR_BAD_TEMPERATURE,
    DEVERR_BAD_TOKEN,
    DEVERR_CACHE_FULL,
    DEVERR_FILTER_BAND,
    DEVERR_TIMEOUT,
    SIGNATURES,
    SSDError,
    SpecCache,
    get_device_error,
    load_library,
    new_workspace,
    profile_begin,
    profile_end,
    selftest_exp2,
    set_split,
    set_chain_batch,
    set_step_schedule,
    softmax_workspace_bytes,
    ssd_draft_sample,
    ssd_forked_recovery,
    ssd_sample_residual,
    ssd_softmax_temp,
    ssd_verify,
    ssd_verify_fork,
    ssd_verify_fork_cache,
    ssd_verify_topk,
    ssd_verify_tree,
    workspace_bytes,
)

__all__ = [
    "ssd_softmax_temp", "ssd_verify", "ssd_sample_residual", "ssd_forked_recovery",
    "ssd_verify_fork", "SpecCache", "workspace_bytes", "softmax_workspace_bytes",
    "new_workspace", "get_device_error", "load_library", "selftest_exp2", "SSDError",
]
