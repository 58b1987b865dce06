"""GB300-native slot-indexed recurrent-state cache for KDA/GDN linear-attention layers.

The compute runs in librsc.so (hand-written sm_103a CUDA kernels behind the C ABI of
include/rsc.h); this package is its ctypes binding plus the seeded workload inputs.
"""
from .binding import (  # noqa: F401
    BF16, COMMIT, F32, GDN, KDA, VERIFY, ReplayRings, RscError, SlotAllocator, SlotPool,
    kda_decode_step, max_running_requests, track_plan,
    kda_decode_step_ex, kda_decode_step_gated, kda_decode_step_track, kda_prefill_chunk, kda_prefill_workspace_size, kda_replay_verify_commit,
    kda_spec_verify_commit, lib,
    rsc_get_device_error, ssm_pool_bytes, ssm_slot_copy, status_string,
)
