"""GB300-native Kimi Delta Attention (KDA) recurrent decode.

The decode entry points of libkda, with the C names:

    kda_recurrent_decode   T=1, split q/k/v, softplus or bounded gate
    kda_packed_decode      Kimi K3 packed QKV, T=1, bf16 state
    kda_fused_decode       short conv + SiLU, KDA step, gated RMSNorm
    kda_spec_decode        ragged speculative rows, T >= 1 tokens each
    kda_spec_verify_decode the same from a read-only state, with commit caches
    kda_packed_fused_decode fused conv + KDA + RMSNorm over ragged speculative
                           rows, with per-token conv and state checkpoints

Build the library with ``python -m linear_attention_decode_02_gb300.build``.
"""

from .binding import (SCHED_AUTO, SCHED_SPLIT, SCHED_STREAM, KdaError, kda_device_error,  # noqa: F401
                      kda_fused_decode, kda_packed_decode, kda_packed_fused_decode, kda_plan_schedule, kda_plan_split,
                      kda_recurrent_decode, kda_set_schedule_override, kda_set_split_override,
                      kda_spec_decode, kda_spec_verify_decode, kda_version, library)
