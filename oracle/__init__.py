"""CPU oracle for the DDP gradient-synchronisation hot path.

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline / reference leg.  The product library never imports
it and never falls back to it.  See ddp_oracle.py for the definitions and the
passages each one follows.

Every function is pinned by tests/test_oracle_*.py; none is "parity unpinned".
"""
from .ddp_oracle import (  # noqa: F401
    PLAN_CAP,
    PLAN_DEEP_FIRST,
    WALK_CAP,
    accumulate,
    any_nonfinite,
    bf16_bits_to_f32,
    bn_fold_inference,
    bn_running_update,
    clip_coefficient,
    dist_sampler_indices,
    f32_to_bf16_rne,
    f64_to_bf16_rne,
    feistel_encrypt,
    feistel_round_keys,
    grad_mean,
    grad_global_norm,
    grad_mean_tree,
    keyed_perm,
    keyed_perm_all,
    murmur3_fmix32,
    plan_buckets,
    ring_allreduce_mean,
    sampler_num_samples,
    sgd_from_grad,
    sgd_step,
    splitmix64_mix,
    splitmix64_stream,
    syncbn,
    syncbn_stats,
    syncbn_stats_at,
)
