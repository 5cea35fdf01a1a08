"""The C-ABI library: builds, loads, exports every declared symbol, and
rejects contract breaches on the host before any CUDA call (CPU only).

Descriptors here point at host memory: validation never dereferences data,
so a breach returns its status without touching a GPU.  A call that passes
validation on a machine without a GPU stops at the device query instead
(KDA_ERR_CUDA or KDA_ERR_UNSUPPORTED), never at a launch.
"""

import ctypes
import os
import re

import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build
from linear_attention_decode_02_gb300.binding import KdaTensor, desc

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
OK, INVALID, UNSUPPORTED, ALIAS, CUDA = 0, 1, 2, 3, 4
# Descriptors here point at host memory.  A call that passes validation
# would launch a kernel on them when a GPU is present, so those calls are
# made only on machines without one (validation failures never launch).
NO_GPU = not torch.cuda.is_available()


def _passes_validation(status):
    """Without a GPU a valid call stops at the device query."""
    return status in (CUDA, UNSUPPORTED)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.library()


def test_every_declared_symbol_is_exported(lib):
    with open(os.path.join(ROOT, "include", "kda.h")) as f:
        text = f.read()
    declared = set(re.findall(r"^(?:kda_status|int32_t|const char\*)\s+(kda_\w+)\(", text, re.M))
    assert declared == set(binding.EXPORTS)
    for name in declared:
        assert hasattr(lib, name), name


def test_status_strings_and_version(lib):
    assert lib.kda_status_string(0) == b"KDA_OK"
    assert lib.kda_status_string(3) == b"KDA_ERR_ALIAS"
    assert b"sm_103a" in lib.kda_version()


def test_plan_split_policy(lib):
    # split kernel: 16 slabs per unit below half the SM count, 8 up to five
    # units per SM, 4 above; speculative rows always 2
    assert binding.kda_plan_split(0, 16384, 0, 1, 152) == 4
    assert binding.kda_plan_split(0, 32, 0, 1, 152) == 16
    assert binding.kda_plan_split(0, 76, 0, 1, 152) == 16
    assert binding.kda_plan_split(0, 77, 0, 1, 152) == 8
    assert binding.kda_plan_split(0, 759, 0, 1, 152) == 8
    assert binding.kda_plan_split(0, 760, 0, 1, 152) == 4
    assert binding.kda_plan_split(3, 2048, 0, 6, 152) == 2
    assert binding.kda_plan_split(3, 16, 0, 6, 152) == 2
    for units in (1, 8, 38, 76, 77, 16384):  # fused: one CTA per unit unless a cluster is forced
        assert binding.kda_plan_split(2, units, 0, 1, 152) == 1
    assert binding.kda_plan_split(0, 1, 5, 1, 152) == 0  # bad dtype
    assert binding.kda_plan_split(9, 1, 0, 1, 152) == 0  # bad op
    for units in (1, 3, 12, 100, 1000, 100000):
        s = binding.kda_plan_split(1, units, 1, 1, 152)
        assert s in (1, 2, 4, 8, 16)


def test_split_override(lib):
    assert lib.kda_set_split_override(3) == INVALID
    assert lib.kda_set_split_override(4) == OK
    assert binding.kda_plan_split(0, 16384, 0, 1, 152) == 4
    assert binding.kda_plan_split(2, 16384, 0, 1, 152) == 4
    assert lib.kda_set_split_override(16) == OK
    assert binding.kda_plan_split(2, 16384, 0, 1, 152) == 4  # a forced 8 or 16 runs as 4
    assert lib.kda_set_split_override(0) == OK
    assert binding.kda_plan_split(0, 16384, 0, 1, 152) == 4


def _recurrent_args(B=2, H=2, N=4, qkv=torch.bfloat16, state=torch.float32):
    t = dict(
        q=torch.zeros(B, H, 128, dtype=qkv), k=torch.zeros(B, H, 128, dtype=qkv),
        v=torch.zeros(B, H, 128, dtype=qkv), raw_gate=torch.zeros(B, H, 128, dtype=qkv),
        raw_beta=torch.zeros(B, H, dtype=qkv), A_log=torch.zeros(H), dt_bias=torch.zeros(H * 128),
        state_indices=torch.ones(B, dtype=torch.int32), state=torch.zeros(N, H, 128, 128, dtype=state),
        out=torch.zeros(B, H, 128, dtype=torch.bfloat16))
    return t


def test_cached_descriptors_equal_fresh_ones():
    # the marshalling cache is keyed on everything a descriptor holds
    base = torch.zeros(6, 4, 128, dtype=torch.bfloat16)
    views = [base, base[1:], base[:, ::2], base.transpose(0, 1), torch.zeros(3, dtype=torch.int32),
             torch.zeros(2, 3, 128, 128), torch.zeros(0, 4, dtype=torch.float32)]
    for _ in range(2):
        for t in views:
            assert bytes(binding._ref(t)._obj) == bytes(desc(t))
    for i in range(binding._DESC_CACHE_MAX + 8):
        binding._ref(torch.zeros(1 + i % 7, 3)[: 1 + i % 5])
    assert len(binding._DESC_CACHE) <= binding._DESC_CACHE_MAX


def _call_recurrent(lib, t, has_lb=0, lb=0.0, scale=0.088):
    names = ["q", "k", "v", "raw_gate", "raw_beta", "A_log", "dt_bias", "state_indices", "state", "out"]
    ds = [desc(t[n]) if isinstance(t[n], torch.Tensor) else t[n] for n in names]
    return lib.kda_recurrent_decode(*[ctypes.byref(d) for d in ds], has_lb, lb, scale, None)


def _msg(lib):
    return lib.kda_last_error_message().decode()


@pytest.mark.skipif(not NO_GPU, reason="a GPU is present: a valid call would launch on host memory")
def test_recurrent_valid_args_reach_the_device_query(lib):
    st = _call_recurrent(lib, _recurrent_args())
    assert _passes_validation(st), _msg(lib)


@pytest.mark.parametrize("mutate,expect,text", [
    (lambda t: t.update(q=torch.zeros(2, 2, 64, dtype=torch.bfloat16)), INVALID, "q: axis 2"),
    (lambda t: t.update(k=torch.zeros(2, 2, 128, dtype=torch.float32)), INVALID, "dtype must match q"),
    (lambda t: t.update(state_indices=torch.ones(2, dtype=torch.float32)), INVALID, "state_indices: dtype"),
    (lambda t: t.update(state=torch.zeros(4, 3, 128, 128)), INVALID, "state: axis 1"),
    (lambda t: t.update(state=torch.zeros(4, 2, 128, 128, dtype=torch.int32)), INVALID, "state: dtype"),
    (lambda t: t.update(state=torch.zeros(4, 2, 128, 256)[..., :128]), INVALID, "contiguous"),
    (lambda t: t.update(out=torch.zeros(2, 2, 128, dtype=torch.float32)), INVALID, "out: dtype"),
    (lambda t: t.update(out=torch.zeros(2, 128, 2, dtype=torch.bfloat16).transpose(1, 2)), INVALID, "contiguous"),
    (lambda t: t.update(q=torch.zeros(2, 2, 130, dtype=torch.bfloat16)[..., 1:129]), INVALID, "multiple of 4"),
    (lambda t: t.update(q=torch.zeros(2, 2, 132, dtype=torch.bfloat16)[..., 2:130]), INVALID, "aligned"),
    (lambda t: t.update(A_log=torch.zeros(3)), INVALID, "A_log"),
    (lambda t: t.update(dt_bias=torch.zeros(2 * 64)), INVALID, "dt_bias"),
    (lambda t: t.update(raw_beta=torch.zeros(2, 3, dtype=torch.bfloat16)), INVALID, "raw_beta"),
])
def test_recurrent_rejects_breaches(lib, mutate, expect, text):
    t = _recurrent_args()
    mutate(t)
    assert _call_recurrent(lib, t) == expect
    assert text in _msg(lib)


def test_recurrent_rejects_aliasing_out_and_state(lib):
    t = _recurrent_args()
    t["out"] = t["state"].view(-1)[: 2 * 2 * 128].view(torch.bfloat16)[: 2 * 2 * 128].view(2, 2, 128)
    assert _call_recurrent(lib, t) == ALIAS
    assert "overlaps" in _msg(lib)
    t = _recurrent_args()
    t["state"] = torch.zeros(4, 2, 128, 128)
    t["q"] = t["state"].view(torch.bfloat16).view(-1)[: 2 * 2 * 128].view(2, 2, 128)
    assert _call_recurrent(lib, t) == ALIAS


def test_recurrent_rejects_bad_gate_and_scale(lib):
    assert _call_recurrent(lib, _recurrent_args(), has_lb=1, lb=1.0) == INVALID
    assert _call_recurrent(lib, _recurrent_args(), has_lb=2, lb=-5.0) == INVALID
    assert _call_recurrent(lib, _recurrent_args(), scale=0.0) == INVALID
    assert _call_recurrent(lib, _recurrent_args(), scale=float("nan")) == INVALID


def test_null_descriptor_is_rejected(lib):
    t = _recurrent_args()
    names = ["q", "k", "v", "raw_gate", "raw_beta", "A_log", "dt_bias", "state_indices", "state", "out"]
    ptrs = [ctypes.byref(desc(t[n])) for n in names]
    ptrs[4] = None
    assert lib.kda_recurrent_decode(*ptrs, 0, 0.0, 0.088, None) == INVALID
    assert "raw_beta: null" in _msg(lib)


def test_empty_batch_launches_nothing(lib):
    t = _recurrent_args(B=0)
    assert _call_recurrent(lib, t) == OK


def _packed_args(B=3, N=4):
    return dict(mixed_qkv=torch.zeros(B, 4608, dtype=torch.bfloat16),
                raw_gate=torch.zeros(B, 1536, dtype=torch.bfloat16),
                raw_beta=torch.zeros(B, 12, dtype=torch.bfloat16), A_log=torch.zeros(12),
                dt_bias=torch.zeros(1536), state_indices=torch.ones(B, dtype=torch.int32),
                state=torch.zeros(N, 12, 128, 128, dtype=torch.bfloat16),
                out=torch.zeros(B, 1, 12, 128, dtype=torch.bfloat16))


def _call_packed(lib, t):
    names = ["mixed_qkv", "raw_gate", "raw_beta", "A_log", "dt_bias", "state_indices", "state", "out"]
    return lib.kda_packed_decode(*[ctypes.byref(desc(t[n])) for n in names], None)


def test_packed_contract(lib):
    if NO_GPU:
        assert _passes_validation(_call_packed(lib, _packed_args())), _msg(lib)
    for key, val, text in [
        ("mixed_qkv", torch.zeros(3, 4096, dtype=torch.bfloat16), "mixed_qkv: axis 1"),
        ("state", torch.zeros(4, 12, 128, 128), "bfloat16 pool"),
        ("raw_gate", torch.zeros(3, 1536), "raw_gate: dtype"),
        ("out", torch.zeros(3, 1, 8, 128, dtype=torch.bfloat16), "out: axis 1"),
    ]:
        t = _packed_args()
        t[key] = val
        assert _call_packed(lib, t) == INVALID
        assert text in _msg(lib)
    # a padded packed row (row stride > 4608) is accepted by validation
    t = _packed_args()
    t["mixed_qkv"] = torch.zeros(3, 4608 + 64, dtype=torch.bfloat16)[:, :4608]
    if NO_GPU:
        assert _passes_validation(_call_packed(lib, t)), _msg(lib)


def test_empty_packed_and_fused_batches_launch_nothing(lib):
    # zero rows pass validation and return before any device query
    assert _call_packed(lib, _packed_args(B=0)) == OK, _msg(lib)
    assert _call_fused(lib, _fused_args(rows=0)) == OK, _msg(lib)


def _fused_args(H=8, rows=4, N=9, state=torch.float32):
    HD = H * 128
    return dict(x=torch.zeros(rows, 3 * HD, dtype=torch.bfloat16), conv_weight=torch.zeros(3, 4, HD),
                conv_state=torch.zeros(N, 3, 3 * HD, dtype=torch.bfloat16).permute(0, 2, 1),
                raw_gate=torch.zeros(1, rows, H, 128, dtype=torch.bfloat16),
                raw_beta=torch.zeros(1, rows, H, dtype=torch.bfloat16), A_log=torch.zeros(H),
                dt_bias=torch.zeros(HD), state_indices=torch.ones(rows, dtype=torch.int32),
                state=torch.zeros(N, H, 128, 128, dtype=state),
                output_gate=torch.zeros(rows, H, 128, dtype=torch.bfloat16), norm_weight=torch.ones(128),
                out=torch.zeros(1, rows, H, 128, dtype=torch.bfloat16))


def _call_fused(lib, t, has_lb=1, lb=-5.0, eps=1e-5):
    names = ["x", "conv_weight", "conv_state", "raw_gate", "raw_beta", "A_log", "dt_bias",
             "state_indices", "state", "output_gate", "norm_weight"]
    ds = [ctypes.byref(desc(t[n])) for n in names]
    return lib.kda_fused_decode(*ds, has_lb, lb, eps, ctypes.byref(desc(t["out"])), None)


def test_fused_contract(lib):
    if NO_GPU:
        assert _passes_validation(_call_fused(lib, _fused_args())), _msg(lib)
    t = _fused_args()
    t["conv_state"] = torch.zeros(9, 3 * 1024, 3, dtype=torch.bfloat16)  # tap-contiguous layout
    assert _call_fused(lib, t) == INVALID
    assert "conv_state: strides" in _msg(lib)
    t = _fused_args()
    t["conv_state"] = torch.zeros(5, 3, 3 * 1024, dtype=torch.bfloat16).permute(0, 2, 1)
    assert _call_fused(lib, t) == INVALID  # num_slots differ
    t = _fused_args()
    t["norm_weight"] = torch.ones(64)
    assert _call_fused(lib, t) == INVALID
    assert _call_fused(lib, _fused_args(), eps=-1.0) == INVALID
    t = _fused_args()
    t["out"] = t["x"].view(-1)[: 4 * 8 * 128].view(1, 4, 8, 128)
    assert _call_fused(lib, t) == ALIAS
    t = _fused_args()
    buf = torch.zeros(9 * 3 * 3 * 1024, dtype=torch.bfloat16)
    t["x"] = buf[: 4 * 3 * 1024].view(4, 3 * 1024)
    t["conv_state"] = buf.view(9, 3, 3 * 1024).permute(0, 2, 1)
    assert _call_fused(lib, t) == ALIAS
    assert "conv_state overlaps x" in _msg(lib)


def _spec_args(R=7, N=3, H=2, M=12):
    return dict(q=torch.zeros(R, H, 128, dtype=torch.bfloat16), k=torch.zeros(R, H, 128, dtype=torch.bfloat16),
                v=torch.zeros(R, H, 128, dtype=torch.bfloat16), g=torch.zeros(R, H, 128),
                beta=torch.zeros(R, H, dtype=torch.bfloat16),
                cu_seqlens=torch.tensor([0, 2, 5, 7], dtype=torch.int32)[: N + 1],
                state_indices=torch.ones(N, dtype=torch.int32), state=torch.zeros(M, H, 128, 128),
                out=torch.zeros(R, H, 128, dtype=torch.bfloat16))


def _call_spec(lib, t, t_max=3, logit=1, scale=0.088):
    d = {n: ctypes.byref(desc(v)) for n, v in t.items()}
    return lib.kda_spec_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], logit, d["cu_seqlens"], t_max,
                               d["state_indices"], d["state"], d["out"], scale, None)


def test_spec_contract(lib):
    if NO_GPU:
        assert _passes_validation(_call_spec(lib, _spec_args())), _msg(lib)
    t = _spec_args()
    t["g"] = torch.zeros(7, 2, 128, dtype=torch.bfloat16)
    assert _call_spec(lib, t) == INVALID
    t = _spec_args()
    t["state_indices"] = torch.ones(4, dtype=torch.int32)
    assert _call_spec(lib, t) == INVALID
    assert _call_spec(lib, _spec_args(), t_max=0) == INVALID
    assert _call_spec(lib, _spec_args(), logit=3) == INVALID
    t = _spec_args(R=0)
    t["cu_seqlens"] = torch.zeros(4, dtype=torch.int32)
    assert _call_spec(lib, t) == OK  # no token rows: nothing to launch


def _call_verify(lib, t, corr=None, kg=None, t_max=3):
    d = {n: ctypes.byref(desc(v)) for n, v in t.items()}
    c = ctypes.byref(desc(corr)) if corr is not None else None
    g = ctypes.byref(desc(kg)) if kg is not None else None
    return lib.kda_spec_verify_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], 1, d["cu_seqlens"], t_max,
                                      d["state_indices"], d["state"], d["out"], c, g, 0.088, None)


def test_spec_verify_contract(lib):
    M, H = 12, 2
    if NO_GPU:
        assert _passes_validation(_call_verify(lib, _spec_args())), _msg(lib)
        assert _passes_validation(_call_verify(lib, _spec_args(), torch.zeros(M, H, 4, 128),
                                               torch.zeros(M, H, 4, 256))), _msg(lib)
    assert _call_verify(lib, _spec_args(), t_max=17) == UNSUPPORTED
    assert _call_verify(lib, _spec_args(), torch.zeros(M, H, 4, 128), torch.zeros(M, H, 5, 256)) == INVALID
    assert "token capacity" in _msg(lib)
    assert _call_verify(lib, _spec_args(), torch.zeros(M, H, 17, 128)) == INVALID
    assert _call_verify(lib, _spec_args(), torch.zeros(M + 1, H, 4, 128)) == INVALID
    assert _call_verify(lib, _spec_args(), None, torch.zeros(M, H, 4, 128)) == INVALID
    assert _call_verify(lib, _spec_args(), torch.zeros(M, H, 4, 128, dtype=torch.bfloat16)) == INVALID
    assert _call_verify(lib, _spec_args(), torch.zeros(M, H, 128, 4).transpose(2, 3)) == INVALID
    both = torch.zeros(M, H, 4, 384)
    assert _call_verify(lib, _spec_args(), both[..., :128], both[..., 128:]) == INVALID  # not contiguous
    buf = torch.zeros(M * H * 4 * 256)
    assert _call_verify(lib, _spec_args(), buf[: M * H * 4 * 128].view(M, H, 4, 128),
                        buf.view(M, H, 4, 256)) == ALIAS
    t = _spec_args()
    flat = t["state"].view(-1)
    assert _call_verify(lib, t, flat[: M * H * 4 * 128].view(M, H, 4, 128)) == ALIAS


def _pf_args(R=5, N=3, C=2, H=2, M=9):
    HD = H * 128
    return dict(x=torch.zeros(R, 3 * HD, dtype=torch.bfloat16), conv_weight=torch.zeros(3, 4, HD),
                conv_state=torch.zeros(M, 3, 3 * HD, dtype=torch.bfloat16).permute(0, 2, 1),
                raw_gate=torch.zeros(R, H, 128, dtype=torch.bfloat16), raw_beta=torch.zeros(R, H, dtype=torch.bfloat16),
                A_log=torch.zeros(H), dt_bias=torch.zeros(HD),
                state_indices=torch.arange(1, N * C + 1, dtype=torch.int32).view(N, C),
                query_start_loc=torch.tensor([0, 2, 4, 5], dtype=torch.int32)[: N + 1],
                num_accepted_tokens=torch.ones(N, dtype=torch.int32), state=torch.zeros(M, H, 128, 128),
                output_gate=torch.zeros(R, H, 128, dtype=torch.bfloat16), norm_weight=torch.ones(128),
                out=torch.zeros(R, H, 128, dtype=torch.bfloat16))


def _call_pf(lib, t, eps=1e-5):
    d = {n: ctypes.byref(desc(v)) for n, v in t.items()}
    return lib.kda_packed_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"], d["raw_beta"],
                                       d["A_log"], d["dt_bias"], d["state_indices"], d["query_start_loc"],
                                       d["num_accepted_tokens"], d["state"], d["output_gate"], d["norm_weight"],
                                       1, -5.0, eps, d["out"], None)


def test_empty_token_rows_launch_nothing(lib):
    # no token rows: the speculative and packed fused entry points return
    # before any device query, whatever the sequence count
    t = _spec_args(R=0, N=0)
    t["cu_seqlens"] = torch.zeros(1, dtype=torch.int32)
    t["state_indices"] = torch.zeros(0, dtype=torch.int32)
    assert _call_spec(lib, t) == OK, _msg(lib)
    t = _pf_args(R=0, N=2)
    t["query_start_loc"] = torch.zeros(3, dtype=torch.int32)
    assert _call_pf(lib, t) == OK, _msg(lib)


def test_packed_fused_contract(lib):
    if NO_GPU:
        assert _passes_validation(_call_pf(lib, _pf_args())), _msg(lib)
    t = _pf_args()
    t["state_indices"] = torch.ones(3, dtype=torch.int32)  # rank 1: needs [N, C]
    assert _call_pf(lib, t) == INVALID
    t = _pf_args()
    t["state_indices"] = torch.ones(2, 3, dtype=torch.int32).t()  # column stride 2
    assert _call_pf(lib, t) == INVALID
    t = _pf_args()
    t["query_start_loc"] = torch.zeros(3, dtype=torch.int32)  # needs N+1
    assert _call_pf(lib, t) == INVALID
    t = _pf_args()
    t["num_accepted_tokens"] = torch.ones(2, dtype=torch.int32)
    assert _call_pf(lib, t) == INVALID
    t = _pf_args()
    t["conv_state"] = torch.zeros(9, 3 * 256, 3, dtype=torch.bfloat16)  # tap-innermost layout
    assert _call_pf(lib, t) == INVALID
    t = _pf_args()
    t["raw_gate"] = torch.zeros(4, 2, 128, dtype=torch.bfloat16)  # R mismatch
    assert _call_pf(lib, t) == INVALID
    assert _call_pf(lib, _pf_args(), eps=float("nan")) == INVALID
    t = _pf_args()
    t["x"] = torch.zeros(5, 3 * 256 + 4, dtype=torch.bfloat16)[:, : 3 * 256]  # rows 8 bytes off 16
    assert _call_pf(lib, t) == UNSUPPORTED
    assert "16-byte" in _msg(lib)
    t = _pf_args()
    t["out"] = t["output_gate"]
    assert _call_pf(lib, t) == ALIAS
    t = _pf_args()
    t["x"] = torch.zeros(0, 768, dtype=torch.bfloat16)
    for key in ("raw_gate", "output_gate", "out"):
        t[key] = torch.zeros(0, 2, 128, dtype=torch.bfloat16)
    t["raw_beta"] = torch.zeros(0, 2, dtype=torch.bfloat16)
    t["query_start_loc"] = torch.zeros(4, dtype=torch.int32)
    assert _call_pf(lib, t) == OK  # no token rows: nothing to launch


def test_packed_fused_cluster_policy(lib):
    # measured policy: fp32 4 CTAs at the smallest batches, then 2, then 1; bf16 2, then 1 (8 only when forced)
    assert binding.kda_plan_split(4, 12, 0, 1, 152) == 4  # fp32: 4 CTAs while 6 units <= SMs
    assert binding.kda_plan_split(4, 25, 0, 1, 152) == 4
    assert binding.kda_plan_split(4, 26, 0, 1, 152) == 2  # then 2 while 4 units <= SMs
    assert binding.kda_plan_split(4, 38, 0, 1, 152) == 2
    assert binding.kda_plan_split(4, 39, 0, 1, 152) == 1
    assert binding.kda_plan_split(4, 12, 1, 1, 152) == 2  # bf16: 2 while 4 units <= SMs
    assert binding.kda_plan_split(4, 38, 1, 1, 152) == 2
    assert binding.kda_plan_split(4, 39, 1, 1, 152) == 1
    assert binding.kda_plan_split(4, 96, 0, 1, 152) == 1
    assert binding.kda_plan_split(4, 1536, 1, 1, 152) == 1
    assert binding.kda_plan_schedule(4, 12, 0, 1, 152) == 1
    assert binding.kda_plan_split(5, 12, 0, 1, 152) == 0  # unknown op
    assert lib.kda_set_split_override(16) == OK
    assert binding.kda_plan_split(4, 12, 0, 1, 152) == 8  # a forced 16 runs as 8
    assert lib.kda_set_split_override(0) == OK


def test_schedule_override_and_plan(lib):
    assert lib.kda_set_schedule_override(7) == INVALID
    assert lib.kda_set_schedule_override(2) == OK
    assert binding.kda_plan_schedule(0, 1, 0, 1, 152) == 2
    assert binding.kda_plan_schedule(3, 1, 0, 1, 152) == 1  # stream does not apply to spec rows
    assert lib.kda_set_schedule_override(3) == OK  # tensor-core chunked form: spec rows only
    assert binding.kda_plan_schedule(3, 2048, 1, 6, 152) == 3
    assert binding.kda_plan_schedule(0, 16384, 1, 1, 152) == 2  # T=1 ignores it
    assert binding.kda_plan_schedule(4, 12, 0, 1, 152) == 1
    assert lib.kda_set_schedule_override(0) == OK
    assert binding.kda_plan_schedule(1, 6144, 1, 1, 152) == 2  # bf16 packed: stream
    assert binding.kda_plan_schedule(1, 12, 1, 1, 152) == 1
    assert binding.kda_plan_schedule(0, 16384, 0, 1, 152) == 1  # fp32: split kernel
    assert binding.kda_plan_schedule(0, 16384, 1, 1, 152) == 2  # bf16 state: stream
    assert binding.kda_plan_schedule(2, 8192, 0, 1, 152) == 2  # fused, many units
    assert binding.kda_plan_schedule(2, 1024, 0, 1, 152) == 2
    assert binding.kda_plan_schedule(2, 380, 0, 1, 152) == 2  # from 2.5 units per SM
    assert binding.kda_plan_schedule(2, 379, 1, 1, 152) == 1
    assert binding.kda_plan_schedule(2, 256, 0, 1, 152) == 1
    # speculative rows: the tensor-core form for a bf16 state with t_max >= 14
    assert binding.kda_plan_schedule(3, 2048, 1, 14, 152) == 3
    assert binding.kda_plan_schedule(3, 2048, 1, 16, 152) == 3
    assert binding.kda_plan_schedule(3, 2048, 1, 13, 152) == 1
    assert binding.kda_plan_schedule(3, 2048, 0, 16, 152) == 1  # fp32 state: split kernel
    assert lib.kda_set_split_override(8) == OK  # a forced split implies the split schedule
    assert binding.kda_plan_schedule(1, 6144, 1, 1, 152) == 1
    assert binding.kda_plan_schedule(3, 2048, 1, 16, 152) == 1
    assert lib.kda_set_split_override(0) == OK
    assert lib.kda_set_schedule_override(2) == OK
    assert binding.kda_plan_schedule(3, 2048, 1, 16, 152) == 1  # stream does not apply to spec rows
    assert lib.kda_set_schedule_override(0) == OK
    assert binding.kda_plan_schedule(9, 6144, 1, 1, 152) == 0


def test_device_error_query_needs_a_pointer(lib):
    assert lib.kda_device_error(None, 0) == INVALID


def test_error_messages_are_per_thread(lib):
    """Two host threads make failing calls at the same time (ctypes releases
    the GIL for the call): each reads back only its own call's message."""
    import threading

    null_args = [None] * 10
    t = binding.KdaTensor()
    t.ndim = 0
    rank0_args = [ctypes.byref(t)] * 10
    failures = []

    def worker(args, expect):
        for _ in range(2000):
            st = lib.kda_recurrent_decode(*args, 0, 0.0, 0.088, None)
            msg = lib.kda_last_error_message().decode()
            if st != INVALID or expect not in msg:
                failures.append((st, msg))
                return

    threads = [threading.Thread(target=worker, args=(null_args, "null tensor descriptor")),
               threading.Thread(target=worker, args=(rank0_args, "ndim 0"))]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not failures, failures[:3]
