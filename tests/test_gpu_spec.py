"""GPU parity of kda_spec_decode: ragged speculative rows (T >= 1 tokens),
precomputed fp32 log-decay gates in [-5, 0], H=16, pool of 4N slots.
"""

import json
import os

import numpy as np
import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    yield binding.library()
    binding.kda_set_split_override(0)


def _run(d, t_max, out=None, beta_is_logit=True):
    return binding.kda_spec_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                   d["state_indices"], d["state"], t_max, out=out, beta_is_logit=beta_is_logit)


def _check(case, d, before, out, rows=None, beta_is_logit=True):
    ref_tok, ref_state = P.oracle_spec(case, rows=rows, beta_is_logit=beta_is_logit)
    if ref_tok:
        toks = sorted(ref_tok)
        P.assert_out_close(out[toks], np.stack([ref_tok[t] for t in toks]))
    for s, S in ref_state.items():
        P.assert_state_close(d["state"][s], S)
    idx, cu = case["state_indices"], case["cu_seqlens"]
    M = case["state"].shape[0]
    touched = [int(idx[n]) for n in range(idx.shape[0])
               if 0 < int(idx[n]) < M and int(cu[n + 1]) > int(cu[n])]
    P.assert_untouched(before, d["state"], touched)
    # rows of null sequences and padding rows are zero
    R = out.shape[0]
    covered = set()
    for n in range(idx.shape[0]):
        if 0 < int(idx[n]) < M:
            covered |= set(range(max(int(cu[n]), 0), min(int(cu[n + 1]), R)))
    zero = [t for t in range(R) if t not in covered]
    if zero:
        assert torch.count_nonzero(out[zero]) == 0


@pytest.mark.parametrize("N", [1, 16, 128])
@pytest.mark.parametrize("t_max", [2, 4, 5, 6])
def test_spec_config_sweep(N, t_max):
    case = synth.spec_case(N, t_max, seed=N * 10 + t_max, null_count=N // 16)
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full(case["q"].shape, 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, t_max, out=out)
    torch.cuda.synchronize()
    _check(case, d, before, out)


@pytest.mark.parametrize("split", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_spec_every_split(split, state_dtype):
    binding.kda_set_split_override(split)
    case = synth.spec_case(9, 5, seed=split, H=4, null_count=1, pad_rows=3, state_dtype=state_dtype)
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full(case["q"].shape, 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, 5, out=out)
    torch.cuda.synchronize()
    _check(case, d, before, out)
    binding.kda_set_split_override(0)


def test_spec_long_rows_span_several_token_chunks():
    case = synth.spec_case(4, 19, seed=3, H=2, lengths=[19, 9, 0, 17])
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run(d, 19)
    torch.cuda.synchronize()
    _check(case, d, before, out)


def test_spec_strong_decay_splits_chunks():
    """Log decays near the clamp force one-token chunks; results stay at parity."""
    case = synth.spec_case(3, 6, seed=9, H=2, lengths=[6, 3, 5])
    gen = torch.Generator().manual_seed(3)
    case["g"] = -(40.0 + 15.0 * torch.rand(case["g"].shape, generator=gen))
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run(d, 6)
    torch.cuda.synchronize()
    _check(case, d, before, out)


def test_spec_precomputed_beta():
    case = synth.spec_case(6, 3, seed=4, H=3)
    case["beta"] = torch.rand(case["beta"].shape, generator=torch.Generator().manual_seed(1))
    d = P.to_device(case)
    before = d["state"].clone()
    out = _run(d, 3, beta_is_logit=False)
    torch.cuda.synchronize()
    _check(case, d, before, out, beta_is_logit=False)


@pytest.mark.parametrize("split", [8, 0])
def test_spec_equals_sequential_single_token_calls(split):
    """One T-token call == T calls of one token per row, within the fp32 state
    and output tolerances (the T-token call defers the decay within a token
    chunk, a different rounding order from T single-token calls)."""
    binding.kda_set_split_override(split)
    case = synth.spec_case(12, 6, seed=5, H=16)
    lens, cu = case["lengths"], case["cu_seqlens"]
    d = P.to_device(case)
    out_all = _run(d, 6)
    d2 = P.to_device(case)
    out_seq = torch.zeros_like(out_all)
    for t in range(6):
        rows = [n for n in range(12) if int(lens[n]) > t]
        tok = torch.tensor([int(cu[n]) + t for n in rows], dtype=torch.long)
        sub = {k: d2[k][tok.cuda()] for k in ("q", "k", "v", "g", "beta")}
        sub["cu_seqlens"] = torch.arange(len(rows) + 1, dtype=torch.int32, device="cuda")
        sub["state_indices"] = d2["state_indices"][torch.tensor(rows, device="cuda")]
        sub["state"] = d2["state"]
        o = _run(sub, 1)
        out_seq[tok.cuda()] = o
    torch.cuda.synchronize()
    binding.kda_set_split_override(0)
    assert (d["state"] - d2["state"]).abs().max().item() <= P.F32_STATE_ATOL
    assert (out_all.float() - out_seq.float()).abs().max().item() <= P.OUT_ATOL


def test_spec_trailing_empty_rows_golden():
    with open(os.path.join(GOLDEN, "spec_trailing_empty.json")) as f:
        fx = json.load(f)
    case = synth.spec_case(4, 1, seed=6, H=12, lengths=[1, 1, 0, 0], pad_rows=2, num_slots=8)
    case["state_indices"] = torch.tensor(fx["state_indices"], dtype=torch.int32)
    assert case["cu_seqlens"].tolist() == fx["cu_seqlens"]
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full((fx["num_token_rows"], 12, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(d, 1, out=out)
    torch.cuda.synchronize()
    mutated = [s for s in range(8) if not torch.equal(before[s], d["state"][s])]
    assert mutated == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert torch.count_nonzero(out[r]) == 0
    _check(case, d, before, out)


def test_spec_graph_replay_with_dynamic_cu_seqlens():
    """Captured with every row active; replayed with an empty middle row."""
    H = 12
    case = synth.spec_case(3, 1, seed=7, H=H, lengths=[1, 1, 1], num_slots=8)
    case["state_indices"] = torch.tensor([1, 2, 3], dtype=torch.int32)
    d = P.to_device(case)
    fresh = d["state"].clone()
    out = torch.zeros(3, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(d, 1, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(d, 1, out=out)
    d["state"].copy_(fresh)
    d["cu_seqlens"].copy_(torch.tensor([0, 1, 1, 2], dtype=torch.int32))
    case["cu_seqlens"] = torch.tensor([0, 1, 1, 2], dtype=torch.int32)
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    _check(case, d, fresh, out)
    # token row 1 belongs to sequence 2 (slot 3); row 2 is padding
    assert not torch.equal(fresh[3], d["state"][3]) and torch.equal(fresh[2], d["state"][2])
    assert torch.count_nonzero(out[2]) == 0


def test_spec_no_rows_all_token_rows_padding():
    case = synth.spec_case(1, 1, seed=12, H=2, lengths=[0], pad_rows=4, num_slots=4)
    case["state_indices"] = case["state_indices"][:0]
    case["cu_seqlens"] = torch.zeros(1, dtype=torch.int32)
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full((4, 2, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, 1, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert torch.equal(before, d["state"])


@pytest.mark.parametrize("state_dtype,t_max,fixed", [(torch.float32, 6, False), (torch.bfloat16, 6, False),
                                                     (torch.bfloat16, 16, False), (torch.bfloat16, 16, True)])
def test_spec_full_size_every_row(state_dtype, t_max, fixed):
    """The timed size (N=128, T <= 6, H=16) with either state dtype, and with
    a bf16 pool rows of up to and of exactly 16 tokens (the dispatcher's
    tensor-core form, two chunks a row): every token row and every live slot
    against the oracle."""
    case = synth.spec_case(128, t_max, seed=21, null_count=8, state_dtype=state_dtype,
                           lengths=[t_max] * 128 if fixed else None)
    d = P.to_device(case)
    before = d["state"].clone()
    out = torch.full(case["q"].shape, float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(d, t_max, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()
    _check(case, d, before, out)
    assert binding.kda_device_error() == 0
