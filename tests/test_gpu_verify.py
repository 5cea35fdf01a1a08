"""GPU parity of kda_spec_verify_decode (speculative verify): outputs of the
ragged speculative rows from a read-only state, and the slot-indexed
correction and key/gate caches a later commit replays.
"""

import numpy as np
import pytest
import torch

from oracle import kda_oracle as ko
from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P

pytestmark = pytest.mark.gpu
CORR_ATOL = 1e-4  # float32 corrections u = beta (v - S_d^T k_hat), |u| of order 1


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    yield binding.library()
    binding.kda_set_split_override(0)


def _caches(M, H, t_cap):
    corr = torch.full((M, H, t_cap, 128), float("nan"), dtype=torch.float32, device="cuda")
    kg = torch.full((M, H, t_cap, 256), float("nan"), dtype=torch.float32, device="cuda")
    return corr, kg


def _run(d, t_max, corr, kg, out=None, beta_is_logit=True):
    return binding.kda_spec_verify_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                          d["state_indices"], d["state"], t_max, out=out, correction_cache=corr,
                                          kg_cache=kg, beta_is_logit=beta_is_logit)


def _written(case, t_cap):
    """{slot: cached token count} for the live, non-empty rows."""
    idx, cu = case["state_indices"], case["cu_seqlens"]
    M, R = case["state"].shape[0], case["q"].shape[0]
    w = {}
    for n in range(idx.shape[0]):
        s = int(idx[n])
        t0, t1 = max(int(cu[n]), 0), min(int(cu[n + 1]), R)
        if 0 < s < M and t1 > t0:
            w[s] = min(t1 - t0, t_cap)
    return w


def _check(case, d, before, out, corr, kg, t_cap, beta_is_logit=True):
    assert torch.equal(before, d["state"]), "verify mode wrote the state"
    ref_tok, ref_corr, ref_kg = P.oracle_verify(case, t_cap, beta_is_logit=beta_is_logit)
    if ref_tok:
        toks = sorted(ref_tok)
        P.assert_out_close(out[toks], np.stack([ref_tok[t] for t in toks]))
    written = _written(case, t_cap)
    corr_c, kg_c = corr.double().cpu().numpy(), kg.double().cpu().numpy()
    for s, a in written.items():
        if corr is not None:
            err = np.abs(corr_c[s, :, :a] - ref_corr[s][:, :a]).max()
            assert err <= CORR_ATOL, f"slot {s}: correction error {err:.3e}"
        if kg is not None:
            assert np.array_equal(kg_c[s, :, :a], ref_kg[s][:, :a]), f"slot {s}: key/gate cache differs"
    # every entry outside the written prefixes keeps its sentinel
    mask = np.ones(corr_c.shape[:3], dtype=bool)
    for s, a in written.items():
        mask[s, :, :a] = False
    assert np.isnan(corr_c[mask]).all() and np.isnan(kg_c[mask]).all(), "a cache entry outside the rows changed"


@pytest.mark.parametrize("N", [1, 16])
@pytest.mark.parametrize("t_max", [1, 4, 6])
def test_verify_config_sweep(N, t_max):
    case = synth.spec_case(N, t_max, seed=N * 7 + t_max, null_count=N // 8)
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(case["state"].shape[0], 16, t_max)
    out = torch.full(case["q"].shape, 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, t_max, corr, kg, out=out)
    torch.cuda.synchronize()
    _check(case, d, before, out, corr, kg, t_max)


@pytest.mark.parametrize("split", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_verify_every_split(split, state_dtype):
    binding.kda_set_split_override(split)
    case = synth.spec_case(9, 5, seed=split + 40, H=4, null_count=1, pad_rows=3, state_dtype=state_dtype)
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(case["state"].shape[0], 4, 5)
    out = torch.full(case["q"].shape, 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, 5, corr, kg, out=out)
    torch.cuda.synchronize()
    binding.kda_set_split_override(0)
    _check(case, d, before, out, corr, kg, 5)


def test_verify_long_rows_past_the_cache_capacity():
    """Rows of up to 16 tokens with a capacity of 6: all decoded, six cached."""
    case = synth.spec_case(4, 16, seed=11, H=2, lengths=[16, 9, 0, 13])
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(case["state"].shape[0], 2, 6)
    out = _run(d, 16, corr, kg)
    torch.cuda.synchronize()
    _check(case, d, before, out, corr, kg, 6)


def test_verify_outputs_equal_spec_decode():
    """Verify mode's outputs are spec decode's; spec decode then advances the state."""
    case = synth.spec_case(12, 6, seed=13, H=8, null_count=1)
    d = P.to_device(case)
    corr, kg = _caches(case["state"].shape[0], 8, 6)
    out_v = _run(d, 6, corr, kg)
    out_s = binding.kda_spec_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                    d["state_indices"], d["state"], 6)
    torch.cuda.synchronize()
    assert (out_v.float() - out_s.float()).abs().max().item() <= P.OUT_ATOL


def test_verify_graph_replay_with_dynamic_cu_seqlens():
    """Captured with every row active; replayed with new tokens and an empty
    middle row: the outputs and caches follow the new metadata."""
    H, t_cap = 6, 4
    case = synth.spec_case(3, 2, seed=15, H=H, lengths=[2, 2, 2], num_slots=8)
    case["state_indices"] = torch.tensor([1, 2, 3], dtype=torch.int32)
    d = P.to_device(case)
    corr, kg = _caches(8, H, t_cap)
    out = torch.zeros(6, H, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        _run(d, 2, corr, kg, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _run(d, 2, corr, kg, out=out)
    c2 = synth.spec_case(3, 2, seed=16, H=H, lengths=[2, 2, 2], num_slots=8)
    c2["state"] = case["state"]
    c2["state_indices"] = case["state_indices"]
    c2["cu_seqlens"] = torch.tensor([0, 2, 2, 4], dtype=torch.int32)
    for key in ("q", "k", "v", "g", "beta", "cu_seqlens"):
        d[key].copy_(c2[key].cuda())
    corr.fill_(float("nan"))
    kg.fill_(float("nan"))
    out.fill_(3.0)
    before = d["state"].clone()
    g.replay()
    torch.cuda.synchronize()
    _check(c2, d, before, out, corr, kg, t_cap)
    assert torch.count_nonzero(out[4:]) == 0  # token rows past cu_seqlens[N] are padding


def test_verify_without_caches():
    case = synth.spec_case(5, 3, seed=14, H=3)
    d = P.to_device(case)
    before = d["state"].clone()
    out = binding.kda_spec_verify_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"],
                                         d["state_indices"], d["state"], 3)
    torch.cuda.synchronize()
    assert torch.equal(before, d["state"])
    ref_tok, _, _ = P.oracle_verify(case, 3)
    toks = sorted(ref_tok)
    P.assert_out_close(out[toks], np.stack([ref_tok[t] for t in toks]))


def test_verify_precomputed_beta():
    case = synth.spec_case(6, 3, seed=15, H=3)
    case["beta"] = torch.rand(case["beta"].shape, generator=torch.Generator().manual_seed(2))
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(case["state"].shape[0], 3, 3)
    out = _run(d, 3, corr, kg, beta_is_logit=False)
    torch.cuda.synchronize()
    _check(case, d, before, out, corr, kg, 3, beta_is_logit=False)


@pytest.mark.parametrize("state_dtype", [torch.float32, torch.bfloat16])
def test_commit_from_device_caches(state_dtype):
    """Replaying the first `a` cached tokens of a row on the committed state
    gives the state that decoding those `a` tokens gives."""
    N, T, H = 6, 5, 4
    case = synth.spec_case(N, T, seed=16, H=H, lengths=[5, 3, 5, 1, 4, 2], state_dtype=state_dtype)
    d = P.to_device(case)
    corr, kg = _caches(case["state"].shape[0], H, T)
    _run(d, T, corr, kg)
    torch.cuda.synchronize()
    corr_c, kg_c = corr.double().cpu().numpy(), kg.double().cpu().numpy()
    accepted = [2, 3, 5, 0, 1, 2]
    # the oracle's state after the accepted prefix of each row
    pre = dict(case)
    cu = [0]
    sel = []
    for n, a in enumerate(accepted):
        t0 = int(case["cu_seqlens"][n])
        sel += list(range(t0, t0 + a))
        cu.append(cu[-1] + a)
    s_idx = torch.tensor(sel, dtype=torch.long)
    for key in ("q", "k", "v", "g", "beta"):
        pre[key] = case[key][s_idx]
    pre["cu_seqlens"] = torch.tensor(cu, dtype=torch.int32)
    _, ref_state = P.oracle_spec(pre)
    for n, a in enumerate(accepted):
        s = int(case["state_indices"][n])
        S0 = P.f64(case["state"][s])
        for h in range(H):
            got = ko.commit_from_cache(S0[h], kg_c[s, h, :a], corr_c[s, h, :a])
            want = ref_state[s][h] if a > 0 else S0[h]
            err = np.abs(got - want).max()
            assert err <= P.F32_STATE_ATOL, f"row {n} head {h}: commit error {err:.3e}"


def test_verify_argument_errors():
    case = synth.spec_case(2, 3, seed=17, H=2)
    d = P.to_device(case)
    M = case["state"].shape[0]
    with pytest.raises(binding.KdaError, match="16 tokens"):
        _run(d, 17, None, None)
    corr, _ = _caches(M, 2, 3)
    _, kg = _caches(M, 2, 4)
    with pytest.raises(binding.KdaError, match="token capacity"):
        _run(d, 3, corr, kg)
    bad = torch.zeros(M + 1, 2, 3, 128, dtype=torch.float32, device="cuda")
    with pytest.raises(binding.KdaError):
        _run(d, 3, bad, None)
    with pytest.raises(binding.KdaError):
        _run(d, 3, d["state"].view(M, 2, 128, 128)[:, :, :3, :], None)


def test_verify_no_rows_all_token_rows_padding():
    case = synth.spec_case(1, 1, seed=18, H=2, lengths=[0], pad_rows=3, num_slots=4)
    case["state_indices"] = case["state_indices"][:0]
    case["cu_seqlens"] = torch.zeros(1, dtype=torch.int32)
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(4, 2, 2)
    out = torch.full((3, 2, 128), 5.0, dtype=torch.bfloat16, device="cuda")
    _run(d, 1, corr, kg, out=out)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0
    assert torch.equal(before, d["state"])
    assert torch.isnan(corr).all() and torch.isnan(kg).all()


@pytest.mark.parametrize("state_dtype,schedule", [(torch.float32, binding.SCHED_AUTO),
                                                  (torch.bfloat16, binding.SCHED_AUTO),
                                                  (torch.bfloat16, binding.SCHED_SPLIT)])
def test_verify_full_size(state_dtype, schedule):
    """N=128 rows of up to 16 tokens (H=16) from a read-only pool of either
    dtype; with a bf16 pool the dispatcher's choice at t_max=16 (the
    tensor-core form) and the per-token kernel."""
    case = synth.spec_case(128, 16, seed=22, null_count=8, state_dtype=state_dtype)
    d = P.to_device(case)
    before = d["state"].clone()
    corr, kg = _caches(case["state"].shape[0], 16, 16)
    binding.kda_set_schedule_override(schedule)
    try:
        out = _run(d, 16, corr, kg)
        torch.cuda.synchronize()
    finally:
        binding.kda_set_schedule_override(binding.SCHED_AUTO)
    _check(case, d, before, out, corr, kg, 16)
    assert binding.kda_device_error() == 0
