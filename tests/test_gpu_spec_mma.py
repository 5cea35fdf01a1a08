"""GPU parity of the tensor-core (tcgen05) chunked form of the speculative
entry points, bfloat16 state: kda_spec_decode and kda_spec_verify_decode with
the MMA schedule forced, against the float64 oracle and against the
per-token CUDA-core kernel.
"""

import numpy as np
import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P
from tests import test_gpu_spec as TS
from tests import test_gpu_verify as TV

pytestmark = pytest.mark.gpu
BF16 = torch.bfloat16


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    yield binding.library()
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.fixture
def mma():
    binding.kda_set_schedule_override(binding.SCHED_MMA)
    yield
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


def _spec(case, t_max, beta_is_logit=True):
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full(case["q"].shape, 5.0, dtype=BF16, device="cuda")
    TS._run(d, t_max, out=out, beta_is_logit=beta_is_logit)
    torch.cuda.synchronize()
    TS._check(case, d, before, out, beta_is_logit=beta_is_logit)
    assert binding.kda_device_error() == 0
    return d, out


@pytest.mark.parametrize("N", [1, 16, 128])
@pytest.mark.parametrize("t_max", [2, 4, 5, 6])
def test_mma_spec_config_sweep(mma, N, t_max):
    case = synth.spec_case(N, t_max, seed=300 + N * 10 + t_max, null_count=N // 16, state_dtype=BF16)
    _spec(case, t_max)


@pytest.mark.parametrize("H", [1, 3, 16])
def test_mma_spec_head_counts_padding_and_null_rows(mma, H):
    case = synth.spec_case(9, 5, seed=310 + H, H=H, null_count=2, pad_rows=3, state_dtype=BF16)
    _spec(case, 5)


def test_mma_spec_one_token_rows(mma):
    case = synth.spec_case(40, 1, seed=320, H=8, null_count=3, state_dtype=BF16)
    _spec(case, 1)


def test_mma_spec_rows_longer_than_a_chunk(mma):
    """Rows of 9..25 tokens run two to four chunks with the state carried on
    chip (bf16 high part plus low part) between them."""
    case = synth.spec_case(5, 25, seed=321, H=4, lengths=[25, 9, 0, 17, 16], state_dtype=BF16)
    _spec(case, 25)


def test_mma_spec_strong_and_zero_decay(mma):
    case = synth.spec_case(4, 12, seed=322, H=2, lengths=[12, 6, 3, 10], state_dtype=BF16)
    gen = torch.Generator().manual_seed(5)
    g = -(40.0 + 15.0 * torch.rand(case["g"].shape, generator=gen))
    g[: case["g"].shape[0] // 2] = 0.0  # no decay on the first half of the token rows
    case["g"] = g
    _spec(case, 12)


def test_mma_spec_precomputed_beta(mma):
    case = synth.spec_case(6, 6, seed=323, H=3, state_dtype=BF16)
    case["beta"] = torch.rand(case["beta"].shape, generator=torch.Generator().manual_seed(2))
    _spec(case, 6, beta_is_logit=False)


def test_mma_spec_many_units_per_cta(mma):
    """4800 units: every CTA's stage ring and operand buffers wrap many times."""
    case = synth.spec_case(300, 4, seed=324, H=16, null_count=20, state_dtype=BF16)
    _spec(case, 4)


def test_mma_spec_fp32_state_is_refused(mma):
    case = synth.spec_case(3, 2, seed=325, H=2)
    d = P.to_device(case)
    with pytest.raises(binding.KdaError) as e:
        TS._run(d, 2)
    assert e.value.status == 2


def test_mma_spec_matches_the_cuda_core_kernel():
    """Same call on both schedules: outputs within the output tolerance,
    states within one bf16 ulp of each other's float32 value."""
    case = synth.spec_case(64, 6, seed=326, H=16, null_count=4, state_dtype=BF16)
    outs, states = [], []
    for sched in (binding.SCHED_SPLIT, binding.SCHED_MMA):
        binding.kda_set_schedule_override(sched)
        try:
            d = P.to_device(case)
            outs.append(TS._run(d, 6))
            torch.cuda.synchronize()
            states.append(d["state"].double())
        finally:
            binding.kda_set_schedule_override(binding.SCHED_AUTO)
    assert (outs[0].double() - outs[1].double()).abs().max().item() <= P.OUT_ATOL
    ulp = torch.from_numpy(np.maximum(P.ko.bf16_ulp(states[0].cpu().numpy()), P.BF16_STATE_FLOOR)).cuda()
    assert bool(((states[0] - states[1]).abs() <= 2 * ulp).all())


def test_mma_spec_graph_replay_with_dynamic_cu_seqlens(mma):
    H = 12
    case = synth.spec_case(3, 2, seed=327, H=H, lengths=[2, 2, 2], num_slots=8, state_dtype=BF16)
    case["state_indices"] = torch.tensor([1, 2, 3], dtype=torch.int32)
    d = P.to_device(case)
    fresh = d["state"].clone()
    out = torch.zeros(case["q"].shape, dtype=BF16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        TS._run(d, 2, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        TS._run(d, 2, out=out)
    d["state"].copy_(fresh)
    new_cu = torch.tensor([0, 2, 2, 4], dtype=torch.int32)
    d["cu_seqlens"].copy_(new_cu)
    case["cu_seqlens"] = new_cu
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    TS._check(case, d, fresh, out)
    assert torch.equal(fresh[2], d["state"][2]) and torch.count_nonzero(out[4:]) == 0


def test_mma_spec_no_rows_all_padding(mma):
    case = synth.spec_case(1, 1, seed=328, H=2, lengths=[0], pad_rows=4, num_slots=4, state_dtype=BF16)
    case["state_indices"] = case["state_indices"][:0]
    case["cu_seqlens"] = torch.zeros(1, dtype=torch.int32)
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full((4, 2, 128), 5.0, dtype=BF16, device="cuda")
    TS._run(d, 1, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert torch.equal(before, d["state"])


def test_mma_spec_chained_calls_track_the_oracle(mma):
    """Eight chained calls on the same slots with fresh tokens each time: the
    state each call leaves feeds the next, compared with the oracle after
    every call."""
    lens = [5, 3, 0, 4, 1, 5]
    case = synth.spec_case(6, 5, seed=329, H=4, lengths=lens, state_dtype=BF16)
    d = P.to_device(case)
    for step in range(8):
        sc = synth.spec_case(6, 5, seed=400 + step, H=4, lengths=lens, make_state=False)
        for key in ("q", "k", "v", "g", "beta"):
            d[key].copy_(sc[key].cuda())
            case[key] = sc[key]
        case["state"] = d["state"].cpu()
        before = d["state"].clone()
        out = torch.full(case["q"].shape, 5.0, dtype=BF16, device="cuda")
        TS._run(d, 5, out=out)
        torch.cuda.synchronize()
        TS._check(case, d, before, out)


@pytest.mark.parametrize("N,t_max", [(1, 4), (16, 6), (9, 16)])
def test_mma_verify(mma, N, t_max):
    """Verify mode on the tensor cores: outputs, correction and key/gate
    caches, the state untouched; up to 16 tokens (two chunks)."""
    case = synth.spec_case(N, t_max, seed=330 + N + t_max, H=6, null_count=N // 8, state_dtype=BF16)
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = TV._caches(case["state"].shape[0], 6, t_max)
    out = torch.full(case["q"].shape, 5.0, dtype=BF16, device="cuda")
    TV._run(d, t_max, corr, kg, out=out)
    torch.cuda.synchronize()
    TV._check(case, d, before, out, corr, kg, t_max)
    assert binding.kda_device_error() == 0


def test_mma_verify_then_decode_agree(mma):
    case = synth.spec_case(20, 6, seed=340, H=8, state_dtype=BF16)
    d = P.to_device(case)
    corr, kg = TV._caches(case["state"].shape[0], 8, 6)
    out_v = TV._run(d, 6, corr, kg)
    out_d = TS._run(d, 6)
    torch.cuda.synchronize()
    assert torch.equal(out_v, out_d)


def test_auto_schedule_takes_the_tensor_core_form_for_long_bf16_rows():
    """With a bf16 pool and t_max >= 14 the dispatcher picks the tensor-core
    form on its own; the rows (two chunks each, some ragged) match the
    oracle like the forced schedule does."""
    assert binding.kda_plan_schedule(binding.OP_SPEC, 20 * 4, 1, 16, 152) == binding.SCHED_MMA
    assert binding.kda_plan_schedule(binding.OP_SPEC, 20 * 4, 1, 13, 152) == binding.SCHED_SPLIT
    case = synth.spec_case(20, 16, seed=341, H=4, null_count=2, state_dtype=BF16)
    _spec(case, 16)
