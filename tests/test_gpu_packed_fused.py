"""GPU parity of kda_packed_fused_decode: packed speculative sequences through
the fused conv + KDA + gated RMSNorm step, with per-token conv and recurrent
checkpoints, against the float64 oracle.
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


def _run(d, out=None, lower_bound=-5.0):
    return binding.kda_packed_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"], d["raw_beta"],
                                           d["A_log"], d["dt_bias"], d["state_indices"], d["query_start_loc"],
                                           d["num_accepted_tokens"], d["state"], d["output_gate"],
                                           d["norm_weight"], lower_bound=lower_bound, out=out)


def _check(case, d, st0, cs0, out, seqs=None, lower_bound=-5.0):
    ref_tok, ref_st, ref_cs = P.oracle_packed_fused(case, seqs=seqs, lower_bound=lower_bound)
    if ref_tok:
        toks = sorted(ref_tok)
        P.assert_out_close_or_ulp(out[toks], np.stack([ref_tok[t] for t in toks]))
    for s, S in ref_st.items():
        P.assert_state_close(d["state"][s], S)
        got = d["conv_state"][s].double().cpu().numpy()
        assert np.array_equal(got, ref_cs[s]), f"conv checkpoint of slot {s} differs"
    written = P.packed_fused_written_slots(case)
    if seqs is None:
        assert set(ref_st) == written
    P.assert_untouched(st0, d["state"], sorted(written))
    P.assert_untouched(cs0, d["conv_state"], sorted(written))
    # rows of null or padding sequences are zero
    idx, qsl, acc = case["state_indices"], case["query_start_loc"], case["num_accepted_tokens"]
    M, R = case["state"].shape[0], case["x"].shape[0]
    live_rows = set()
    for n in range(idx.shape[0]):
        a = int(acc[n])
        if 1 <= a <= idx.shape[1] and 0 < int(idx[n, a - 1]) < M:
            live_rows |= set(range(max(int(qsl[n]), 0), min(int(qsl[n + 1]), R)))
    zero = [t for t in range(R) if t not in live_rows]
    if zero:
        assert torch.count_nonzero(out[zero]) == 0


def _setup(case):
    d = P.to_device(case)
    return d, d["state"].clone(), d["conv_state"].clone()


@pytest.mark.parametrize("N", [1, 8, 33])
@pytest.mark.parametrize("t_max", [1, 3, 5])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_packed_fused_config_sweep(N, t_max, state_dtype):
    case = synth.packed_fused_case(N, t_max, H=12, seed=N * 10 + t_max, null_count=N // 8,
                                   state_dtype=state_dtype, pad_rows=2)
    d, st0, cs0 = _setup(case)
    out = torch.full((case["x"].shape[0], 12, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, out=out)
    torch.cuda.synchronize()
    _check(case, d, st0, cs0, out)


@pytest.mark.parametrize("cluster", [1, 2, 4, 8])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_packed_fused_every_cluster_size(cluster, state_dtype):
    binding.kda_set_split_override(cluster)
    try:
        case = synth.packed_fused_case(7, 5, H=3, seed=60 + cluster, null_count=1, pad_rows=3,
                                       state_dtype=state_dtype)
        case["state_indices"][0, 2] = -1  # one skipped checkpoint
        d, st0, cs0 = _setup(case)
        out = torch.full((case["x"].shape[0], 3, 128), 5.0, dtype=torch.bfloat16, device="cuda")
        _run(d, out=out)
        torch.cuda.synchronize()
    finally:
        binding.kda_set_split_override(0)
    _check(case, d, st0, cs0, out)


@pytest.mark.parametrize("cluster", [1, 8])
def test_packed_fused_long_sequences_every_cluster_extreme(cluster):
    binding.kda_set_split_override(cluster)
    try:
        case = synth.packed_fused_case(3, 17, H=2, seed=70 + cluster, lengths=[17, 9, 12], cols=10,
                                       accepted=[1, 10, 4])
        d, st0, cs0 = _setup(case)
        out = _run(d)
        torch.cuda.synchronize()
    finally:
        binding.kda_set_split_override(0)
    _check(case, d, st0, cs0, out)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_packed_fused_long_sequences_span_token_chunks(state_dtype):
    """Sequences of up to 19 tokens (three chunks) with 12 checkpoint columns:
    tokens past column 11 decode but write no checkpoint."""
    case = synth.packed_fused_case(4, 19, H=2, seed=31, lengths=[19, 9, 0, 13], cols=12, accepted=[1, 12, 3, 7],
                                   state_dtype=state_dtype)
    d, st0, cs0 = _setup(case)
    out = _run(d)
    torch.cuda.synchronize()
    _check(case, d, st0, cs0, out)


def test_packed_fused_softplus_gate_and_head_counts():
    for H in (1, 8, 32):
        case = synth.packed_fused_case(5, 4, H=H, seed=40 + H, null_count=1)
        d, st0, cs0 = _setup(case)
        out = _run(d, lower_bound=None)
        torch.cuda.synchronize()
        _check(case, d, st0, cs0, out, lower_bound=None)


@pytest.mark.parametrize("state_dtype,cluster", [(torch.float32, 0), (torch.bfloat16, 1)])
def test_packed_fused_null_checkpoints_and_bad_accepted_counts(state_dtype, cluster):
    """Skipped, null and out-of-range checkpoint slots; with a bf16 state and
    one CTA per unit the checkpoints leave by TMA stores."""
    case = synth.packed_fused_case(4, 3, H=3, seed=32, lengths=[3, 3, 2, 3], accepted=[1, 2, 4, 0],
                                   state_dtype=state_dtype)
    case["state_indices"][0, 1] = -1   # checkpoint 1 of sequence 0 not kept
    case["state_indices"][1, 1] = 0    # sequence 1 starts from the null slot
    case["state_indices"][0, 2] = 10 ** 6  # out of range: skipped
    d, st0, cs0 = _setup(case)
    out = torch.full((case["x"].shape[0], 3, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    binding.kda_set_split_override(cluster)
    try:
        _run(d, out=out)
        torch.cuda.synchronize()
    finally:
        binding.kda_set_split_override(0)
    _check(case, d, st0, cs0, out)


def _review(fx, seed, H=12):
    n = len(fx["state_indices"])
    lens = np.diff(fx["query_start_loc"]).tolist()
    case = synth.packed_fused_case(n, 1, H=H, seed=seed, lengths=lens,
                                   pad_rows=fx["num_token_rows"] - fx["query_start_loc"][-1], num_slots=8,
                                   accepted=fx["num_accepted_tokens"])
    case["state_indices"] = torch.tensor(fx["state_indices"], dtype=torch.int32)
    return case


def test_packed_fused_review_case_a_golden():
    with open(os.path.join(GOLDEN, "packed_fused_review_cases.json")) as f:
        fx = json.load(f)["case_a"]
    case = _review(fx, 50)
    d, st0, cs0 = _setup(case)
    out = torch.full((fx["num_token_rows"], 12, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(d, out=out)
    torch.cuda.synchronize()
    assert [s for s in range(8) if not torch.equal(st0[s], d["state"][s])] == fx["expected_mutated_slots"]
    assert [s for s in range(8) if not torch.equal(cs0[s], d["conv_state"][s])] == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert torch.count_nonzero(out[r]) == 0
    _check(case, d, st0, cs0, out)


def test_packed_fused_graph_replay_with_dynamic_metadata():
    """Captured with every sequence active; replayed with an empty middle
    sequence (the review's case B): row 1 then belongs to sequence 2."""
    with open(os.path.join(GOLDEN, "packed_fused_review_cases.json")) as f:
        fx = json.load(f)["case_b"]
    case = _review(fx, 51)
    d, st0, cs0 = _setup(case)
    d["query_start_loc"].copy_(torch.tensor([0, 1, 2, 3], dtype=torch.int32))
    out = torch.zeros(3, 12, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(d, out=out)
    d["state"].copy_(st0)
    d["conv_state"].copy_(cs0)
    d["query_start_loc"].copy_(torch.tensor(fx["query_start_loc"], dtype=torch.int32))
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    assert [s for s in range(8) if not torch.equal(st0[s], d["state"][s])] == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert torch.count_nonzero(out[r]) == 0
    _check(case, d, st0, cs0, out)


def test_packed_fused_equals_token_by_token_fused_calls():
    """One T-token call equals T single-token kda_fused_decode calls on the
    start slot, each followed by a copy of both caches to the checkpoint slot."""
    N, T, H = 6, 4, 12
    case = synth.packed_fused_case(N, T, H=H, seed=33, lengths=[4, 4, 2, 3, 1, 4], accepted=1)
    d, _, _ = _setup(case)
    out = _run(d)
    d2 = P.to_device(case)
    idx, qsl = case["state_indices"], case["query_start_loc"]
    out_seq = torch.zeros_like(out)
    for n in range(N):
        s0 = int(idx[n, 0])
        for j, t in enumerate(range(int(qsl[n]), int(qsl[n + 1]))):
            o = binding.kda_fused_decode(d2["x"][t:t + 1], d2["conv_weight"], d2["conv_state"],
                                         d2["raw_gate"][t:t + 1], d2["raw_beta"][t:t + 1], d2["A_log"],
                                         d2["dt_bias"], torch.tensor([s0], dtype=torch.int32, device="cuda"),
                                         d2["state"], d2["output_gate"][t:t + 1], d2["norm_weight"])
            out_seq[t] = o[0, 0]
            sj = int(idx[n, j])
            if sj != s0:
                d2["state"][sj].copy_(d2["state"][s0])
                d2["conv_state"][sj].copy_(d2["conv_state"][s0])
        # the start slot now holds the caches after the sequence's last token
    torch.cuda.synchronize()
    P.assert_out_close_or_ulp(out, out_seq.double().cpu().numpy())
    for n in range(N):
        L = int(qsl[n + 1]) - int(qsl[n])
        last = int(idx[n, L - 1])
        assert (d["state"][last] - d2["state"][int(idx[n, 0])]).abs().max().item() <= P.F32_STATE_ATOL


@pytest.mark.parametrize("H,state_dtype", [(12, torch.float32), (12, torch.bfloat16), (24, torch.float32)])
def test_packed_fused_full_size_every_sequence(H, state_dtype):
    """The timed configuration: 128 sequences of 5 tokens, one accepted token,
    a checkpoint per token; every token row, state checkpoint and conv
    checkpoint against the oracle."""
    N, T = 128, 5
    case = synth.packed_fused_case(N, T, H=H, seed=80 + H, lengths=[T] * N, accepted=1, state_dtype=state_dtype)
    d, st0, cs0 = _setup(case)
    out = torch.full((N * T, H, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    _run(d, out=out)
    torch.cuda.synchronize()
    assert not torch.isnan(out).any()  # every token row written
    _check(case, d, st0, cs0, out)


def test_packed_fused_no_sequences_all_rows_padding():
    """N = 0 with token rows present: every row is padding, no cache touched."""
    case = synth.packed_fused_case(1, 1, H=2, seed=97, lengths=[0], pad_rows=3)
    case["state_indices"] = case["state_indices"][:0]
    case["num_accepted_tokens"] = case["num_accepted_tokens"][:0]
    case["query_start_loc"] = torch.zeros(1, dtype=torch.int32)
    d, st0, cs0 = _setup(case)
    out = torch.full((3, 2, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert torch.equal(st0, d["state"]) and torch.equal(cs0, d["conv_state"])


def test_packed_fused_every_start_slot_null():
    case = synth.packed_fused_case(6, 3, H=4, seed=98)
    case["state_indices"][:] = -1
    d, st0, cs0 = _setup(case)
    out = torch.full((case["x"].shape[0], 4, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert torch.equal(st0, d["state"]) and torch.equal(cs0, d["conv_state"])


@pytest.mark.parametrize("cluster", [2, 4, 8])
def test_packed_fused_cluster_start_slot_is_first_checkpoint_repeated(cluster):
    """With one accepted token the start slot is also the first checkpoint
    slot, so each CTA of a cluster must read the slot's conv history before
    any peer overwrites it with its slab's checkpoint.  Fifty repeated calls
    from the same caches must give the oracle's result bit for bit every
    time."""
    binding.kda_set_split_override(cluster)
    try:
        case = synth.packed_fused_case(6, 5, H=3, seed=90 + cluster, lengths=[5, 3, 5, 1, 4, 5], accepted=1)
        d, st0, cs0 = _setup(case)
        out = _run(d)
        torch.cuda.synchronize()
        _check(case, d, st0, cs0, out)
        first = (out.clone(), d["state"].clone(), d["conv_state"].clone())
        for _ in range(50):
            d["state"].copy_(st0)
            d["conv_state"].copy_(cs0)
            out.fill_(0.0)
            _run(d, out=out)
            torch.cuda.synchronize()
            assert torch.equal(out, first[0])
            assert torch.equal(d["state"], first[1])
            assert torch.equal(d["conv_state"], first[2])
    finally:
        binding.kda_set_split_override(0)
