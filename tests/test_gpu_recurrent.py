"""GPU parity of kda_recurrent_decode and kda_packed_decode against the oracle.

Shapes: the tiny 4-row case, Kimi-Linear H=32 fp32 state (B up to 512 over a
1024-slot pool, rows sampled at the largest size) and the packed Kimi K3
contract (H=12, bf16 state, 10% padding rows, B from 1 to 512).
"""

import os
import numpy as np
import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P

pytestmark = pytest.mark.gpu
SPLITS = [0, 1, 2, 4, 8, 16]


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    yield binding.library()
    binding.kda_set_split_override(0)
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


def _run_recurrent(d, lower_bound=None, out=None):
    return binding.kda_recurrent_decode(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["A_log"],
                                        d["dt_bias"], d["state_indices"], d["state"], out=out,
                                        lower_bound=lower_bound)


def _check_recurrent(case, d, before, out, rows=None, lower_bound=None):
    ref_out, ref_state = P.oracle_recurrent(case, rows=rows, lower_bound=lower_bound)
    r = list(range(out.shape[0])) if rows is None else list(rows)
    P.assert_out_close(out.reshape(out.shape[0], -1, 128)[r], ref_out)
    for s, S in ref_state.items():
        P.assert_state_close(d["state"][s], S)
    P.assert_untouched(before, d["state"], P.live_slots(case["state_indices"], case["state"].shape[0]))
    idx = case["state_indices"]
    null = [i for i in r if not (0 < int(idx[i]) < case["state"].shape[0])]
    if null:
        assert torch.count_nonzero(out.reshape(out.shape[0], -1)[null]) == 0


@pytest.mark.parametrize("split", SPLITS)
def test_tiny_case_every_split(split):
    binding.kda_set_split_override(split)
    case = synth.tiny_recurrent_case()
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out)
    binding.kda_set_split_override(0)


@pytest.mark.parametrize("split", SPLITS)
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lower_bound", [None, -5.0])
def test_kimi_linear_small_pool(split, state_dtype, lower_bound):
    binding.kda_set_split_override(split)
    case = synth.recurrent_case(24, 32, 40, seed=1, state_dtype=state_dtype, null_count=3)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_recurrent(d, lower_bound=lower_bound)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out, lower_bound=lower_bound)
    binding.kda_set_split_override(0)


@pytest.mark.parametrize("B", [1, 8, 32, 128, 512])
def test_kimi_linear_full_pool(B):
    """H=32 fp32 pool [1024, 32, 128, 128], distinct slots, auto split."""
    case = synth.recurrent_case(B, 32, 1024, seed=2)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out)  # every row and slot against the oracle


def test_strided_views_into_one_projection_row():
    """q, k, v as views into one padded projection row; raw gate / beta with their own row strides."""
    B, H = 6, 4
    base = synth.recurrent_case(B, H, 10, seed=3)
    proj = torch.zeros(B, 3 * H * 128 + 64, dtype=torch.bfloat16)
    proj[:, : H * 128] = base["q"].reshape(B, -1)
    proj[:, H * 128: 2 * H * 128] = base["k"].reshape(B, -1)
    proj[:, 2 * H * 128: 3 * H * 128] = base["v"].reshape(B, -1)
    gbuf = torch.zeros(B, H * 128 + 256, dtype=torch.bfloat16)
    gbuf[:, : H * 128] = base["raw_gate"].reshape(B, -1)
    bbuf = torch.zeros(B, 7, dtype=torch.bfloat16)
    bbuf[:, :H] = base["raw_beta"]
    pd, gd, bd = proj.cuda(), gbuf.cuda(), bbuf.cuda()
    d = P.to_device(base)
    d["q"] = pd[:, : H * 128].view(B, H, 128)
    d["k"] = pd[:, H * 128: 2 * H * 128].view(B, H, 128)
    d["v"] = pd[:, 2 * H * 128: 3 * H * 128].view(B, H, 128)
    d["raw_gate"] = gd[:, : H * 128].view(B, H, 128)
    d["raw_beta"] = bd[:, :H]
    assert d["q"].stride(0) == 3 * H * 128 + 64 and d["raw_beta"].stride(0) == 7
    before = d["state"].clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    _check_recurrent(base, d, before, out)


def test_guard_bands_between_slots_stay_untouched():
    """Slot stride larger than the slot block: the gaps must not be written."""
    B, H, N = 5, 3, 8
    case = synth.recurrent_case(B, H, N, seed=4, in_dtype=torch.float32)
    block = H * 128 * 128
    stride = block + 4096
    buf = torch.full((N * stride,), 7.25, dtype=torch.float32, device="cuda")
    pool = torch.as_strided(buf, (N, H, 128, 128), (stride, 128 * 128, 128, 1))
    pool.copy_(case["state"].cuda())
    d = P.to_device(case)
    d["state"] = pool
    gaps = buf.view(N, stride)[:, block:].clone()
    before = pool.clone()
    out = torch.full((B, H, 128), 3.0, dtype=torch.bfloat16, device="cuda")
    _run_recurrent(d, out=out)
    torch.cuda.synchronize()
    assert torch.equal(buf.view(N, stride)[:, block:], gaps)
    _check_recurrent(case, d, before, out)


def test_current_stream_and_graph_replay_with_new_indices():
    """Captured once; replays see changed inputs and indices (null rows included)."""
    B, H, N = 8, 32, 64
    c1 = synth.recurrent_case(B, H, N, seed=5, null_count=1)
    d = P.to_device(c1)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run_recurrent(d, out=out)  # warm-up on a side stream
    torch.cuda.current_stream().wait_stream(s)
    fresh = P.dev(c1["state"])
    d["state"].copy_(fresh)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run_recurrent(d, out=out)
    for seed in (6, 7):
        c2 = synth.recurrent_case(B, H, N, seed=seed, null_count=2)
        c2["state"] = c1["state"]
        for key in ("q", "k", "v", "raw_gate", "raw_beta", "A_log", "dt_bias", "state_indices"):
            d[key].copy_(c2[key].cuda())
        d["state"].copy_(fresh)
        before = d["state"].clone()
        g.replay()
        torch.cuda.synchronize()
        _check_recurrent(c2, d, before, out)


def test_repeated_calls_are_deterministic():
    case = synth.recurrent_case(16, 32, 64, seed=8)
    outs, states = [], []
    for _ in range(2):
        d = P.to_device(case)
        outs.append(_run_recurrent(d))
        states.append(d["state"])
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1]) and torch.equal(states[0], states[1])


# ---- packed Kimi K3 -------------------------------------------------------------

def _run_packed(d, out=None):
    return binding.kda_packed_decode(d["mixed_qkv"], d["raw_gate"], d["raw_beta"], d["A_log"], d["dt_bias"],
                                     d["state_indices"], d["state"], out=out)


def _check_packed(case, d, before, out, rows=None):
    ref_out, ref_state = P.oracle_packed(case, rows=rows)
    r = list(range(out.shape[0])) if rows is None else list(rows)
    P.assert_out_close(out.reshape(out.shape[0], 12, 128)[r], ref_out)
    for s, S in ref_state.items():
        P.assert_state_close(d["state"][s], S)
    P.assert_untouched(before, d["state"], P.live_slots(case["state_indices"], case["state"].shape[0]))
    idx = case["state_indices"]
    pad = [i for i in range(out.shape[0]) if int(idx[i]) <= 0]
    if pad:
        assert torch.count_nonzero(out.reshape(out.shape[0], -1)[pad]) == 0


@pytest.mark.parametrize("B", [1, 8, 16, 31, 32, 64, 128, 256, 512])
def test_packed_batch_sweep(B):
    case = synth.packed_case(B, num_slots=2048, seed=B)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_packed(d)
    torch.cuda.synchronize()
    _check_packed(case, d, before, out)  # every row and slot against the oracle


@pytest.mark.parametrize("split", SPLITS)
def test_packed_every_split_with_padded_rows(split):
    binding.kda_set_split_override(split)
    case = synth.packed_case(20, num_slots=64, seed=11, null_frac=0.25)
    d = P.to_device(case)
    wide = torch.zeros(20, 4608 + 128, dtype=torch.bfloat16, device="cuda")
    wide[:, :4608] = d["mixed_qkv"]
    d["mixed_qkv"] = wide[:, :4608]
    before = d["state"].clone()
    out = torch.full((20, 1, 12, 128), 9.0, dtype=torch.bfloat16, device="cuda")
    _run_packed(d, out=out)
    torch.cuda.synchronize()
    _check_packed(case, d, before, out)
    binding.kda_set_split_override(0)


def test_packed_long_run_drift_stays_bounded():
    """64 chained steps on the same slots, GPU bf16 state vs the float64 oracle
    carried in float64 (reported bound, not bit parity: the GPU rounds the
    state every step)."""
    B = 4
    case = synth.packed_case(B, num_slots=8, seed=12, null_frac=0.0)
    d = P.to_device(case)
    ref_state = {s: P.f64(case["state"][s]) for s in case["state_indices"].tolist()}
    from oracle import kda_oracle as ko
    worst = 0.0
    for step in range(64):
        step_case = synth.packed_case(B, num_slots=8, seed=100 + step, null_frac=0.0)
        for key in ("mixed_qkv", "raw_gate", "raw_beta"):
            d[key].copy_(step_case[key].cuda())
        out = _run_packed(d)
        idx = case["state_indices"].numpy()
        pool = np.zeros((9, 12, 128, 128))
        for s in ref_state:
            pool[s] = ref_state[s]
        ref_out, st = ko.packed_decode(P.f64(step_case["mixed_qkv"]), P.f64(step_case["raw_gate"]),
                                       P.f64(step_case["raw_beta"]), P.f64(case["A_log"]), P.f64(case["dt_bias"]),
                                       idx, pool)
        for s in ref_state:
            ref_state[s] = st[s]
        worst = max(worst, float(np.abs(out.double().cpu().numpy().reshape(B, 12, 128) - ref_out).max()))
    assert worst <= P.OUT_ATOL


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_long_run_drift_512_steps(state_dtype):
    """Drift diagnostic: 512 chained T=1 steps on the same slots (H=4, 4 rows,
    fresh activations every step), the GPU state carried in the pool's dtype
    against the oracle carried in float64.  The curve (max abs error of the
    outputs and of the state at steps 1, 2, 4, ..., 512) is reported in the
    test session's summary; the gate only catches a blow-up."""
    from oracle import kda_oracle as ko
    B, H, M = 4, 4, 8
    case = synth.recurrent_case(B, H, M, seed=13, state_dtype=state_dtype, null_count=0)
    d = P.to_device(case)
    idx = case["state_indices"].numpy()
    pool = P.f64(case["state"])
    curve = []
    for step in range(1, 513):
        sc = synth.recurrent_case(B, H, M, seed=1000 + step, state_dtype=state_dtype, null_count=0)
        for key in ("q", "k", "v", "raw_gate", "raw_beta"):
            d[key].copy_(sc[key].cuda())
        out = _run_recurrent(d)
        ref_out, pool = ko.recurrent_decode(P.f64(sc["q"]), P.f64(sc["k"]), P.f64(sc["v"]), P.f64(sc["raw_gate"]),
                                            P.f64(sc["raw_beta"]), P.f64(case["A_log"]), P.f64(case["dt_bias"]),
                                            idx, pool)
        if step & (step - 1) == 0:
            torch.cuda.synchronize()
            e_out = float(np.abs(out.double().cpu().numpy() - ref_out).max())
            e_st = float(np.abs(d["state"].double().cpu().numpy()[idx] - pool[idx]).max())
            curve.append((step, e_out, e_st))
    P.DRIFT[f"recurrent H=4 {str(state_dtype).split('.')[-1]} state"] = curve
    assert all(np.isfinite(e) for _, a, b in curve for e in (a, b))
    assert max(a for _, a, _ in curve) <= 10 * P.OUT_ATOL


# ---- persistent streaming schedule (bulk copies into shared-memory stages) -----------

@pytest.fixture
def stream_schedule():
    binding.kda_set_schedule_override(binding.SCHED_STREAM)
    yield
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("in_dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("lower_bound", [None, -5.0])
@pytest.mark.parametrize("B,H,N,nulls", [(3, 2, 8, 1), (37, 5, 60, 4)])
def test_stream_schedule_parity(stream_schedule, state_dtype, in_dtype, lower_bound, B, H, N, nulls):
    case = synth.recurrent_case(B, H, N, seed=B + H, in_dtype=in_dtype, state_dtype=state_dtype, null_count=nulls)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_recurrent(d, lower_bound=lower_bound)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out, lower_bound=lower_bound)
    assert binding.kda_device_error() == 0


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_stream_many_units_per_cta(stream_schedule, state_dtype):
    """Thousands of units: every stage is refilled many times."""
    case = synth.recurrent_case(300, 12, 400, seed=21, state_dtype=state_dtype, null_count=30)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out)
    assert binding.kda_device_error() == 0


def test_stream_needs_aligned_head_vectors(stream_schedule):
    """Forced streaming on 8-byte-aligned rows is refused; the policy uses the split kernel instead."""
    B, H = 40, 16
    case = synth.recurrent_case(B, H, 64, seed=22)
    d = P.to_device(case)
    wide = torch.zeros(B, H * 128 + 4, dtype=torch.bfloat16, device="cuda")
    wide[:, : H * 128] = d["q"].reshape(B, -1)
    d["q"] = wide[:, : H * 128].view(B, H, 128)
    assert (d["q"].stride(0) * 2) % 16 == 8
    with pytest.raises(binding.KdaError) as e:
        _run_recurrent(d)
    assert e.value.status == 2
    binding.kda_set_schedule_override(binding.SCHED_AUTO)
    before = d["state"].clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    _check_recurrent(case, d, before, out)


def test_stream_graph_replay(stream_schedule):
    B, H, N = 64, 32, 200
    c1 = synth.recurrent_case(B, H, N, seed=23, null_count=5)
    d = P.to_device(c1)
    out = torch.empty(B, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run_recurrent(d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    fresh = P.dev(c1["state"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run_recurrent(d, out=out)
    c2 = synth.recurrent_case(B, H, N, seed=24, null_count=9)
    for key in ("q", "k", "v", "raw_gate", "raw_beta", "state_indices"):
        d[key].copy_(c2[key].cuda())
    c2["state"], c2["A_log"], c2["dt_bias"] = c1["state"], c1["A_log"], c1["dt_bias"]
    d["state"].copy_(fresh)
    before = d["state"].clone()
    g.replay()
    torch.cuda.synchronize()
    _check_recurrent(c2, d, before, out)


@pytest.mark.parametrize("B", [5, 100])
def test_packed_stream_schedule(stream_schedule, B):
    case = synth.packed_case(B, num_slots=256, seed=25 + B)
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run_packed(d)
    torch.cuda.synchronize()
    _check_packed(case, d, before, out)
    assert binding.kda_device_error() == 0


@pytest.mark.parametrize("B", [8, 100])
def test_packed_graph_replay_with_new_inputs(B):
    """Captured once (split schedule at B=8, streaming at B=100); the replay
    sees new activations and slot indices, null rows included."""
    N = 512
    c1 = synth.packed_case(B, num_slots=N, seed=40 + B)
    d = P.to_device(c1)
    out = torch.empty(B, 1, 12, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run_packed(d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    fresh = P.dev(c1["state"])
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run_packed(d, out=out)
    c2 = synth.packed_case(B, num_slots=N, seed=41 + B, make_state=False)
    for key in ("mixed_qkv", "raw_gate", "raw_beta", "state_indices"):
        d[key].copy_(c2[key].cuda())
    c2["state"], c2["A_log"], c2["dt_bias"] = c1["state"], c1["A_log"], c1["dt_bias"]
    d["state"].copy_(fresh)
    before = d["state"].clone()
    out.fill_(7.0)
    g.replay()
    torch.cuda.synchronize()
    _check_packed(c2, d, before, out)


def test_schedule_policy_queries():
    assert binding.kda_plan_schedule(0, 16384, 0, 1, 152) == binding.SCHED_SPLIT
    assert binding.kda_plan_schedule(1, 6144, 1, 1, 152) == binding.SCHED_STREAM
    assert binding.kda_plan_schedule(0, 32, 1, 1, 152) == binding.SCHED_SPLIT
    assert binding.kda_plan_schedule(2, 16384, 0, 1, 152) == binding.SCHED_STREAM
    assert binding.kda_plan_schedule(3, 16384, 0, 1, 152) == binding.SCHED_SPLIT


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_stream_guard_bands_between_slots(stream_schedule, state_dtype):
    """Stream schedule on a pool whose slot stride exceeds the slot block (tensor-map strides)."""
    B, H, N = 40, 6, 50
    case = synth.recurrent_case(B, H, N, seed=26, state_dtype=state_dtype, null_count=3)
    block = H * 128 * 128
    stride = block + 8192
    buf = torch.full((N * stride,), 7.25, dtype=state_dtype, device="cuda")
    pool = torch.as_strided(buf, (N, H, 128, 128), (stride, 128 * 128, 128, 1))
    pool.copy_(case["state"].cuda())
    d = P.to_device(case)
    d["state"] = pool
    gaps = buf.view(N, stride)[:, block:].clone()
    before = pool.clone()
    out = _run_recurrent(d)
    torch.cuda.synchronize()
    assert torch.equal(buf.view(N, stride)[:, block:], gaps)
    _check_recurrent(case, d, before, out)
    assert binding.kda_device_error() == 0


def test_readme_example_runs():
    """The usage example in the README executes and updates the state in place."""
    import re as _re
    with open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "README.md")) as f:
        blocks = _re.findall(r"```python\n(.*?)```", f.read(), _re.S)
    assert len(blocks) == 1
    scope = {}
    exec(compile(blocks[0], "README.md", "exec"), scope)
    torch.cuda.synchronize()
    out, state = scope["out"], scope["state"]
    assert out.shape == (8, 32, 128) and out.dtype == torch.bfloat16
    assert torch.isfinite(out.float()).all()
    assert torch.count_nonzero(state[1:9]) > 0 and torch.count_nonzero(state[0]) == 0
