"""GPU parity of kda_fused_decode (short conv + SiLU, KDA step, gated RMSNorm).

Heads {8, 12, 32, 96}, rows {1, 32, 256}, bounded (-5) and softplus gates,
float32 and bfloat16 state, a mix of 0 and -1 null rows.  The conv cache is
data movement and must match the oracle bit for bit.
"""

import numpy as np
import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.library()


def _run(d, lower_bound=-5.0, out=None, norm_eps=1e-5):
    return binding.kda_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"], d["raw_beta"],
                                    d["A_log"], d["dt_bias"], d["state_indices"], d["state"], d["output_gate"],
                                    d["norm_weight"], lower_bound=lower_bound, norm_eps=norm_eps, out=out)


def _device_case(case):
    d = P.to_device(case)
    phys = case["conv_state"].permute(0, 2, 1).contiguous().cuda()
    d["conv_state"] = phys.permute(0, 2, 1)
    assert d["conv_state"].stride()[1:] == (1, case["conv_state"].shape[1])
    return d


def _check(case, d, before, cbefore, out, rows=None, lower_bound=-5.0):
    ref_out, ref_state, ref_conv = P.oracle_fused(case, rows=rows, lower_bound=lower_bound)
    n = out.shape[1]
    r = list(range(n)) if rows is None else list(rows)
    P.assert_out_close_or_ulp(out[0][r], ref_out)
    for s, S in ref_state.items():
        P.assert_state_close(d["state"][s], S)
    for s, C in ref_conv.items():
        got = d["conv_state"][s].double().cpu().numpy()
        np.testing.assert_array_equal(got, C)
    touched = P.live_slots(case["state_indices"], case["state"].shape[0])
    P.assert_untouched(before, d["state"], touched)
    P.assert_untouched(cbefore, d["conv_state"], touched)
    idx = case["state_indices"]
    null = [i for i in range(n) if int(idx[i]) <= 0]
    if null:
        assert torch.count_nonzero(out[0][null]) == 0


@pytest.mark.parametrize("H", [8, 12, 32, 96])
@pytest.mark.parametrize("rows", [1, 32, 256])
def test_fused_config_sweep(H, rows):
    case = synth.fused_case(H, rows, seed=H * 1000 + rows)
    d = _device_case(case)
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    out = _run(d)
    torch.cuda.synchronize()
    _check(case, d, before, cbefore, out)  # every row and slot


@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_fused_gate_and_state_dtype(lower_bound, state_dtype):
    case = synth.fused_case(12, 20, seed=5, state_dtype=state_dtype, null_frac=0.3, gate_4d=False)
    d = _device_case(case)
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    out = _run(d, lower_bound=lower_bound)
    torch.cuda.synchronize()
    _check(case, d, before, cbefore, out, lower_bound=lower_bound)


def test_fused_two_windows_chain():
    """Two consecutive calls on the same slots: conv cache and state carry over."""
    H, rows = 8, 6
    case = synth.fused_case(H, rows, seed=9, null_frac=0.0)
    d = _device_case(case)
    _run(d)
    torch.cuda.synchronize()
    mid = dict(case)
    mid["state"] = d["state"].cpu()
    mid["conv_state"] = d["conv_state"].cpu()
    step2 = synth.fused_case(H, rows, seed=10, null_frac=0.0)
    for key in ("x", "raw_gate", "raw_beta", "output_gate"):
        mid[key] = step2[key]
        d[key].copy_(step2[key].cuda())
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    out = _run(d)
    torch.cuda.synchronize()
    _check(mid, d, before, cbefore, out)


def test_fused_graph_replay_with_null_rows():
    H, rows = 12, 16
    case = synth.fused_case(H, rows, seed=11)
    d = _device_case(case)
    out = torch.empty(1, rows, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(d, out=out)
    c2 = synth.fused_case(H, rows, seed=12, null_frac=0.25)
    for key in ("x", "raw_gate", "raw_beta", "output_gate", "state_indices", "state"):
        d[key].copy_(c2[key].cuda())
    d["conv_state"].copy_(c2["conv_state"].cuda())
    c2["conv_weight"], c2["A_log"], c2["dt_bias"], c2["norm_weight"] = (
        case["conv_weight"], case["A_log"], case["dt_bias"], case["norm_weight"])
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    g.replay()
    torch.cuda.synchronize()
    _check(c2, d, before, cbefore, out)


# ---- persistent streaming schedule -------------------------------------------------

@pytest.fixture
def stream_schedule():
    binding.kda_set_schedule_override(binding.SCHED_STREAM)
    yield
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
@pytest.mark.parametrize("H,rows", [(8, 3), (12, 40), (32, 64)])
def test_fused_stream_parity(stream_schedule, state_dtype, lower_bound, H, rows):
    case = synth.fused_case(H, rows, seed=H + rows, state_dtype=state_dtype, null_frac=0.2)
    d = _device_case(case)
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    out = torch.full((1, rows, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    _run(d, lower_bound=lower_bound, out=out)
    torch.cuda.synchronize()
    _check(case, d, before, cbefore, out, lower_bound=lower_bound)
    assert binding.kda_device_error() == 0


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_fused_stream_many_units_and_graph(stream_schedule, state_dtype):
    """Many rounds through both rings (about 16 units a CTA: the activation
    entries run ahead of the state stages and wrap several times), under
    graph replay with new inputs."""
    H, rows = 8, 300
    c1 = synth.fused_case(H, rows, seed=31, null_frac=0.1, state_dtype=state_dtype)
    d = _device_case(c1)
    out = torch.empty(1, rows, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(d, out=out)
    c2 = synth.fused_case(H, rows, seed=32, null_frac=0.15, state_dtype=state_dtype)
    for key in ("x", "raw_gate", "raw_beta", "output_gate", "state_indices", "state"):
        d[key].copy_(c2[key].cuda())
    d["conv_state"].copy_(c2["conv_state"].cuda())
    c2["conv_weight"], c2["A_log"], c2["dt_bias"], c2["norm_weight"] = (
        c1["conv_weight"], c1["A_log"], c1["dt_bias"], c1["norm_weight"])
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    g.replay()
    torch.cuda.synchronize()
    _check(c2, d, before, cbefore, out)
    assert binding.kda_device_error() == 0


def test_fused_stream_rejects_unaligned_rows(stream_schedule):
    H, rows = 8, 4
    case = synth.fused_case(H, rows, seed=33)
    d = _device_case(case)
    wide = torch.zeros(rows, 3 * H * 128 + 4, dtype=torch.bfloat16, device="cuda")
    wide[:, : 3 * H * 128] = d["x"]
    d["x"] = wide[:, : 3 * H * 128]
    with pytest.raises(binding.KdaError) as e:
        _run(d)
    assert e.value.status == 2


def _unaligned_weight(d):
    flat = torch.zeros(d["conv_weight"].numel() + 1, dtype=torch.float32, device="cuda")
    flat[1:] = d["conv_weight"].reshape(-1)
    w = flat[1:].view(d["conv_weight"].shape)
    assert w.data_ptr() % 16 != 0
    return w


def test_fused_stream_rejects_unaligned_conv_weight(stream_schedule):
    """The streaming prologue reads four weights per lane at once."""
    case = synth.fused_case(8, 4, seed=34)
    d = _device_case(case)
    d["conv_weight"] = _unaligned_weight(d)
    with pytest.raises(binding.KdaError) as e:
        _run(d)
    assert e.value.status == 2


def test_fused_unaligned_conv_weight_falls_back_to_split():
    """A batch the dispatcher would stream (32 x 32 units), with conv_weight
    4 bytes off a 16-byte boundary: the call takes the split kernel."""
    H, rows = 32, 32
    case = synth.fused_case(H, rows, seed=35, null_frac=0.1)
    d = _device_case(case)
    d["conv_weight"] = _unaligned_weight(d)
    before, cbefore = d["state"].clone(), d["conv_state"].clone()
    out = _run(d)
    torch.cuda.synchronize()
    _check(case, d, before, cbefore, out)
    assert binding.kda_device_error() == 0


@pytest.mark.parametrize("cluster", [1, 2, 4])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("lower_bound", [-5.0, None])
def test_fused_every_cluster_size(cluster, state_dtype, lower_bound):
    """The split schedule with 1, 2 or 4 CTAs per (row, head): each CTA owns a
    slab of the value columns, the RMSNorm sums meet through distributed
    shared memory, and each conv-cache channel is shifted by exactly one CTA."""
    binding.kda_set_split_override(cluster)
    try:
        case = synth.fused_case(12, 7, seed=70 + cluster, state_dtype=state_dtype, null_frac=0.3)
        d = _device_case(case)
        before, cbefore = d["state"].clone(), d["conv_state"].clone()
        out = torch.full((1, 7, 12, 128), 7.0, dtype=torch.bfloat16, device="cuda")
        _run(d, lower_bound=lower_bound, out=out)
        torch.cuda.synchronize()
    finally:
        binding.kda_set_split_override(0)
    _check(case, d, before, cbefore, out, lower_bound=lower_bound)


@pytest.mark.parametrize("cluster", [2, 4])
def test_fused_cluster_repeated_calls_are_identical(cluster):
    """Every CTA of a cluster reads the conv history of all q and k channels
    while the owning CTA shifts it: fifty calls from the same caches must give
    the same outputs and caches bit for bit."""
    binding.kda_set_split_override(cluster)
    try:
        case = synth.fused_case(8, 3, seed=80 + cluster, null_frac=0.0)
        d = _device_case(case)
        st0, cs0 = d["state"].clone(), d["conv_state"].clone()
        first = None
        for _ in range(50):
            d["state"].copy_(st0)
            d["conv_state"].copy_(cs0)
            out = _run(d)
            torch.cuda.synchronize()
            got = (out.clone(), d["state"].clone(), d["conv_state"].clone())
            if first is None:
                first = got
                _check(case, d, st0, cs0, out)
            else:
                assert all(torch.equal(x, y) for x, y in zip(got, first))
    finally:
        binding.kda_set_split_override(0)
