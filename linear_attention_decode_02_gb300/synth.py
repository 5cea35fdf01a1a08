"""Seeded synthetic inputs for the KDA decode paths.

This module only draws random numbers and lays them out in the shapes,
dtypes and strides of the decode contracts; it holds none of the method's
arithmetic.  The tests feed the same CPU tensors to the CUDA library (after a
copy to the device) and to the float64 oracle (after an exact upcast).

Recipes (all seeded, all CPU ``torch.Generator``):

* recurrent: q, k, v, raw gate, raw beta ~ N(0, 1); A_log ~ U(-2, 0) per
  head; dt_bias ~ N(0, 0.1) per key channel; state pool ~ N(0, 0.1);
  live rows take distinct random slots in [1, num_slots).
* packed (Kimi K3, H=12): packed QKV [B, 4608], raw gate [B, 1536], raw beta
  [B, 12] ~ N(0, 1); bf16 pool; floor(null_frac * B) rows set to -1.
* fused: x ~ N(0, 1) [rows, 3*H*128]; conv weight ~ N(0, 0.5) [3, 4, H*128];
  conv cache ~ N(0, 1) in the [slot][tap][channel] layout; output gate ~
  N(0, 1); norm weight 1 + N(0, 0.1); some rows null (a mix of 0 and -1).
* spec: per-row lengths uniform in [1, T_max] with one row at T_max and
  about 1/8 of the rows empty; q, k, v, beta logits ~ N(0, 1) in bf16;
  log-decay gates ~ U(-5, 0) in fp32; pool of 4*N slots.
"""

from __future__ import annotations

import math

import torch

D = 128


def _gen(seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def _normal(gen, shape, std=1.0, mean=0.0, dtype=torch.float32):
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    if mean != 0.0:
        t.add_(mean)
    return t.to(dtype)


def _uniform(gen, shape, lo, hi, dtype=torch.float32):
    t = torch.rand(*shape, generator=gen, dtype=torch.float32)
    return (t * (hi - lo) + lo).to(dtype)


def distinct_slots(gen, count, num_slots):
    """`count` distinct slot ids drawn from [1, num_slots)."""
    if count > num_slots - 1:
        raise ValueError("not enough slots for distinct live rows")
    return (torch.randperm(num_slots - 1, generator=gen)[:count] + 1).to(torch.int32)


def state_pool(gen, num_slots, heads, dtype, std=0.1):
    """State pool [num_slots, H, 128, 128] ~ N(0, std)."""
    return _normal(gen, (num_slots, heads, D, D), std=std, dtype=dtype)


def with_nulls(gen, slots, null_count, null_values=(-1,)):
    """Replace `null_count` random positions of `slots` by null values."""
    slots = slots.clone()
    if null_count > 0:
        pos = torch.randperm(slots.numel(), generator=gen)[:null_count]
        vals = torch.tensor(null_values, dtype=torch.int32)
        pick = torch.randint(0, len(null_values), (null_count,), generator=gen)
        slots[pos] = vals[pick]
    return slots


def recurrent_case(B, H, num_slots, seed=0, in_dtype=torch.bfloat16,
                   state_dtype=torch.float32, state_indices=None, null_count=0, make_state=True):
    """Inputs of the split q/k/v T=1 path (``kda_recurrent_decode``)."""
    gen = _gen(seed)
    case = {
        "q": _normal(gen, (B, H, D), dtype=in_dtype),
        "k": _normal(gen, (B, H, D), dtype=in_dtype),
        "v": _normal(gen, (B, H, D), dtype=in_dtype),
        "raw_gate": _normal(gen, (B, H, D), dtype=in_dtype),
        "raw_beta": _normal(gen, (B, H), dtype=in_dtype),
        "A_log": _uniform(gen, (H,), -2.0, 0.0),
        "dt_bias": _normal(gen, (H * D,), std=0.1),
    }
    if state_indices is None:
        idx = with_nulls(gen, distinct_slots(gen, B, num_slots), null_count)
    else:
        idx = torch.tensor(state_indices, dtype=torch.int32)
    case["state_indices"] = idx
    if make_state:
        case["state"] = state_pool(gen, num_slots, H, state_dtype)
    return case


def tiny_recurrent_case(seed=0):
    """B=4, H=4, fp32 everything, 8 slots, state_indices [3, 1, -1, 6]."""
    return recurrent_case(4, 4, 8, seed=seed, in_dtype=torch.float32,
                          state_dtype=torch.float32, state_indices=[3, 1, -1, 6])


def packed_case(B, num_slots=2048, seed=0, null_frac=0.1, heads=12, make_state=True):
    """Inputs of the Kimi K3 packed T=1 path (``kda_packed_decode``)."""
    gen = _gen(seed)
    HD = heads * D
    case = {
        "mixed_qkv": _normal(gen, (B, 3 * HD), dtype=torch.bfloat16),
        "raw_gate": _normal(gen, (B, HD), dtype=torch.bfloat16),
        "raw_beta": _normal(gen, (B, heads), dtype=torch.bfloat16),
        "A_log": _uniform(gen, (heads,), -2.0, 0.0),
        "dt_bias": _normal(gen, (HD,), std=0.1),
    }
    n_null = int(math.floor(null_frac * B))
    case["state_indices"] = with_nulls(gen, distinct_slots(gen, B, num_slots), n_null)
    if make_state:
        case["state"] = state_pool(gen, num_slots, heads, torch.bfloat16)
    return case


def conv_cache(gen, num_slots, channels):
    """Conv cache of logical shape [slots, C, 3] stored as [slot][tap][channel].

    Its strides are [3*C, 1, C]: channel stride 1, tap stride C.
    """
    phys = _normal(gen, (num_slots, 3, channels), dtype=torch.bfloat16)
    return phys.permute(0, 2, 1)


def fused_case(H, rows, seed=0, state_dtype=torch.float32, null_frac=0.1,
               num_slots=None, gate_4d=True, make_state=True):
    """Inputs of the fused conv + KDA + gated RMSNorm path (``kda_fused_decode``)."""
    gen = _gen(seed)
    HD = H * D
    if num_slots is None:
        num_slots = 2 * rows + 1
    case = {
        "x": _normal(gen, (rows, 3 * HD), dtype=torch.bfloat16),
        "conv_weight": _normal(gen, (3, 4, HD), std=0.5),
        "raw_gate": _normal(gen, (1, rows, H, D), dtype=torch.bfloat16),
        "raw_beta": _normal(gen, (1, rows, H), dtype=torch.bfloat16),
        "A_log": _uniform(gen, (H,), -2.0, 0.0),
        "dt_bias": _normal(gen, (HD,), std=0.1),
    }
    n_null = int(math.floor(null_frac * rows))
    case["state_indices"] = with_nulls(gen, distinct_slots(gen, rows, num_slots), n_null,
                                       null_values=(0, -1))
    if make_state:
        case["conv_state"] = conv_cache(gen, num_slots, 3 * HD)
        case["state"] = state_pool(gen, num_slots, H, state_dtype)
    og = _normal(gen, (rows, H, D), dtype=torch.bfloat16)
    case["output_gate"] = og.unsqueeze(0) if gate_4d else og
    case["norm_weight"] = _normal(gen, (D,), std=0.1, mean=1.0)
    return case


def spec_lengths(gen, N, t_max, empty_frac=0.125):
    """Ragged lengths in [1, t_max], one row at t_max, about empty_frac rows empty."""
    lens = torch.randint(1, t_max + 1, (N,), generator=gen, dtype=torch.int32)
    lens[torch.randint(0, N, (1,), generator=gen)] = t_max
    n_empty = int(round(empty_frac * N))
    if N > 1 and n_empty > 0:
        full = int((lens == t_max).nonzero()[0])
        cand = torch.tensor([i for i in range(N) if i != full])
        pick = cand[torch.randperm(cand.numel(), generator=gen)[:n_empty]]
        lens[pick] = 0
    return lens


def spec_case(N, t_max, seed=0, H=16, lengths=None, pad_rows=0, null_count=0,
              state_dtype=torch.float32, num_slots=None, make_state=True):
    """Inputs of the packed speculative path (``kda_spec_decode``).

    Token rows [cu[N], cu[N] + pad_rows) are graph padding past the last row.
    """
    gen = _gen(seed)
    if lengths is None:
        lens = spec_lengths(gen, N, t_max)
    else:
        lens = torch.tensor(lengths, dtype=torch.int32)
    cu = torch.zeros(N + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0)
    R = int(cu[-1]) + pad_rows
    if num_slots is None:
        num_slots = 4 * N
    case = {
        "q": _normal(gen, (R, H, D), dtype=torch.bfloat16),
        "k": _normal(gen, (R, H, D), dtype=torch.bfloat16),
        "v": _normal(gen, (R, H, D), dtype=torch.bfloat16),
        "g": _uniform(gen, (R, H, D), -5.0, 0.0),
        "beta": _normal(gen, (R, H), dtype=torch.bfloat16),
        "cu_seqlens": cu,
        "lengths": lens,
        "t_max": int(t_max),
    }
    case["state_indices"] = with_nulls(gen, distinct_slots(gen, N, num_slots), null_count)
    if make_state:
        case["state"] = state_pool(gen, num_slots, H, state_dtype)
    return case


def packed_fused_case(N, t_max, H=12, seed=0, lengths=None, cols=None, accepted=None, pad_rows=0,
                      null_count=0, state_dtype=torch.float32, num_slots=None, make_state=True):
    """Inputs of the packed fused speculative path (``kda_packed_fused_decode``).

    Sequence n owns token rows qsl[n] .. qsl[n+1]-1 and the `cols` distinct
    checkpoint slots state_indices[n, :]; it starts from column
    num_accepted_tokens[n] - 1 (random in 1..cols unless `accepted` is given).
    `null_count` sequences get a null start slot (0 or -1).  Token rows past
    qsl[N] are `pad_rows` of graph padding.
    """
    gen = _gen(seed)
    cols = cols or t_max
    HD = H * D
    if lengths is None:
        lens = spec_lengths(gen, N, t_max)
    else:
        lens = torch.tensor(lengths, dtype=torch.int32)
    qsl = torch.zeros(N + 1, dtype=torch.int32)
    qsl[1:] = torch.cumsum(lens, 0)
    R = int(qsl[-1]) + pad_rows
    if num_slots is None:
        num_slots = N * cols + 1
    case = {
        "x": _normal(gen, (R, 3 * HD), dtype=torch.bfloat16),
        "conv_weight": _normal(gen, (3, 4, HD), std=0.5),
        "raw_gate": _normal(gen, (R, H, D), dtype=torch.bfloat16),
        "raw_beta": _normal(gen, (R, H), dtype=torch.bfloat16),
        "A_log": _uniform(gen, (H,), -2.0, 0.0),
        "dt_bias": _normal(gen, (HD,), std=0.1),
        "query_start_loc": qsl,
        "lengths": lens,
        "t_max": int(t_max),
    }
    idx = distinct_slots(gen, N * cols, num_slots).reshape(N, cols)
    if accepted is None:
        acc = torch.randint(1, cols + 1, (N,), generator=gen, dtype=torch.int32)
    else:
        acc = torch.as_tensor(accepted, dtype=torch.int32).expand(N).clone()
    if null_count > 0:
        pick = torch.randperm(N, generator=gen)[:null_count]
        for n in pick.tolist():
            idx[n, int(acc[n]) - 1] = int(torch.randint(-1, 1, (1,), generator=gen))
    case["state_indices"] = idx
    case["num_accepted_tokens"] = acc
    if make_state:
        case["conv_state"] = conv_cache(gen, num_slots, 3 * HD)
        case["state"] = state_pool(gen, num_slots, H, state_dtype)
    case["output_gate"] = _normal(gen, (R, H, D), dtype=torch.bfloat16)
    case["norm_weight"] = _normal(gen, (D,), std=0.1, mean=1.0)
    return case


def to_f64(t):
    """Exact upcast of a stored tensor to a float64 numpy array (bf16 is exact in f64)."""
    return t.detach().to("cpu").to(torch.float64).numpy()
