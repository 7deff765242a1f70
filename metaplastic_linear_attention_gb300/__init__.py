"""GB300-native Palimpsa dual-state recurrence (metaplastic linear attention).

Per head the recurrence keeps a memory mean mu and an elementwise precision I
(both d_v x d_k); each token makes a beta-weighted write whose per-element
plasticity is set by I, the gate alpha = exp(-A d_t) discounts I toward
I_prior, and the output is y_t = mu_t q_t (Bonnet et al., "Learning to
Remember, Learn, and Forget in Attention-Based Models", Eq. (5)).

The computation lives in ``libpalimpsa.so`` (hand-written sm_103a kernels
behind the C ABI of ``include/palimpsa.h``); this package is its thin binding
plus the seeded synthetic-input generator.
"""
from .binding import (  # noqa: F401
    PALIMPSA_BF16,
    PALIMPSA_F32,
    PALIMPSA_FUSE_QK_NORM,
    PALIMPSA_FUSE_V_STAR,
    PalimpsaError,
    library_path,
    load_library,
    palimpsa_abi_version,
    palimpsa_backward,
    palimpsa_checkpoint_bytes,
    palimpsa_debug_withhold_first_copy,
    palimpsa_forward_checkpointed,
    palimpsa_forward_chunked,
    palimpsa_forward_fused,
    palimpsa_forward_plan,
    palimpsa_forward_varlen,
    palimpsa_forward_varlen_fused,
    palimpsa_forward_varlen_checkpointed,
    palimpsa_backward_varlen,
    palimpsa_checkpoint_bytes_varlen,
    packed_checkpoint_shape,
    palimpsa_forward_without_meta,
    palimpsa_get_device_status,
    palimpsa_probe_issue_rate,
    palimpsa_release_scratch,
    palimpsa_scratch_reserved_bytes,
    palimpsa_segment_summary,
    palimpsa_set_forward_segments,
    palimpsa_set_scratch_retention,
    palimpsa_set_step_l2_keep_bytes,
    palimpsa_set_wait_timeout_ns,
    palimpsa_state_combine,
    palimpsa_status_string,
    palimpsa_step,
    palimpsa_step_fused,
)
