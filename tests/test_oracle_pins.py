"""Pins of the float64 oracle to facts outside itself (CPU only).

Each test checks the oracle against something the pages or the mathematics
fix: library routines for the special cases that reduce to them (softplus,
sigmoid, L2 normalisation, depthwise causal conv1d, RMSNorm, matrix-vector
products), closed forms (decay-only, no-write, unit-key write, the
Householder form of the delta rule), invariants (null rows, untouched slots,
T sequential steps = one T-token call) and the values the pages print
(contract constants, the trailing-empty-rows repro).
"""

import json
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import kda_oracle as ko
from linear_attention_decode_02_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rng(seed=0):
    return np.random.default_rng(seed)


# --- constants and elementwise pieces ---------------------------------------------

def test_contract_constants_match_pages():
    with open(os.path.join(GOLDEN, "contract_constants.json")) as f:
        c = json.load(f)
    assert ko.D == c["head_dim"]
    assert ko.PACKED_HEADS == c["packed_heads"]
    assert 3 * ko.PACKED_HEADS * ko.D == c["packed_qkv_width"]
    assert ko.PACKED_HEADS * ko.D == c["packed_gate_width"]
    assert ko.SCALE == pytest.approx(c["scale"], rel=1e-15)
    assert ko.L2_EPS == c["l2_eps"]
    assert ko.PACKED_LOWER_BOUND == c["packed_lower_bound"]
    assert ko.FUSED_NORM_EPS == c["fused_norm_eps"]
    assert ko.CONV_WIDTH == c["conv_width"]


def test_softplus_matches_logaddexp():
    x = np.concatenate([np.linspace(-60, 60, 2001), [-700.0, 700.0, 0.0]])
    np.testing.assert_allclose(ko.softplus(x), np.logaddexp(0.0, x), rtol=1e-14, atol=1e-300)


def test_sigmoid_and_silu_match_scipy():
    x = np.concatenate([np.linspace(-50, 50, 2001), [-800.0, 800.0]])
    np.testing.assert_allclose(ko.sigmoid(x), scipy.special.expit(x), rtol=1e-14, atol=1e-300)
    np.testing.assert_allclose(ko.silu(x), x * scipy.special.expit(x), rtol=1e-14, atol=1e-300)


def test_l2_normalize_matches_torch_normalize():
    x = _rng(1).standard_normal((64, 128))
    ref = torch.nn.functional.normalize(torch.from_numpy(x), dim=-1).numpy()
    # (sum + 1e-6)^-1/2 vs 1/||x||: relative gap 5e-7 / sum(x^2) < 1e-8 here
    np.testing.assert_allclose(ko.l2_normalize(x), ref, rtol=1e-8)


def test_softplus_gate_identities():
    rng = _rng(2)
    H = 3
    raw = rng.standard_normal((H, 128))
    dt = 0.1 * rng.standard_normal((H, 128))
    A_log = np.array([-2.0, -0.5, 0.0])
    g = ko.gate_softplus(raw, dt, A_log)
    assert np.all(g < 0)
    # at raw + dt = 0 the gate is -exp(A_log) * ln 2 (dt_bias shifts the raw gate)
    g0 = ko.gate_softplus(-dt, dt, A_log)
    np.testing.assert_allclose(g0, -np.exp(A_log)[:, None] * np.log(2.0) * np.ones((H, 128)),
                               rtol=1e-15)
    # A_log -> -inf switches the decay off
    assert np.all(np.abs(ko.gate_softplus(raw, dt, np.full(H, -60.0))) < 1e-24)
    # per-head scaling: head h is exp(A_log[h]) times the unit-rate gate
    unit = ko.gate_softplus(raw, dt, np.zeros(H))
    np.testing.assert_allclose(g, np.exp(A_log)[:, None] * unit, rtol=1e-14)


def test_lower_bound_gate_identities():
    rng = _rng(3)
    lb = -5.0
    H = 2
    A_log = np.array([-1.0, 0.3])
    raw = 3 * rng.standard_normal((H, 128))
    dt = np.zeros((H, 128))
    g = ko.gate_lower_bound(raw, dt, A_log, lb)
    assert np.all(g < 0) and np.all(g > lb)
    g0 = ko.gate_lower_bound(np.zeros((H, 128)), dt, A_log, lb)
    np.testing.assert_array_equal(g0, np.full((H, 128), lb / 2))
    shift = 0.3 * rng.standard_normal((H, 128))
    np.testing.assert_allclose(ko.gate_lower_bound(-shift, shift, A_log, lb), lb / 2, rtol=1e-15)
    # large positive argument saturates at the bound, large negative at zero
    np.testing.assert_allclose(ko.gate_lower_bound(np.full((H, 128), 80.0), dt, A_log, lb),
                               lb, rtol=1e-12)
    assert np.all(np.abs(ko.gate_lower_bound(np.full((H, 128), -80.0), dt, A_log, lb)) < 1e-12)
    # monotone decreasing in the raw gate
    xs = np.linspace(-4, 4, 9)[None, :].repeat(H, 0)
    gs = ko.gate_lower_bound(xs, np.zeros_like(xs), A_log, lb)
    assert np.all(np.diff(gs, axis=1) < 0)
    # dispatch: None selects the softplus form
    np.testing.assert_array_equal(ko.gate(raw, dt, A_log, None), ko.gate_softplus(raw, dt, A_log))


def test_lower_bound_gate_per_head_rate():
    # exp(A_log[h]) is a per-head rate on the pre-activation: head h's gate at
    # x equals the unit-rate gate (A_log = 0) at exp(A_log[h]) * x
    rng = _rng(31)
    lb = -5.0
    A_log = np.array([-2.0, -0.7, 0.0, 0.9])
    H = A_log.size
    raw = 2 * rng.standard_normal((H, 128))
    dt = 0.1 * rng.standard_normal((H, 128))
    g = ko.gate_lower_bound(raw, dt, A_log, lb)
    x = raw + dt
    unit = ko.gate_lower_bound(np.exp(A_log)[:, None] * x, np.zeros_like(x), np.zeros(H), lb)
    np.testing.assert_allclose(g, unit, rtol=1e-13, atol=1e-15)
    # heads with different rates differ away from the midpoint
    assert np.abs(g[0] - ko.gate_lower_bound(raw[:1], dt[:1], A_log[1:2], lb)[0]).max() > 1e-3
    # slope at the midpoint: d/dx lb * sigmoid(a x) at x = 0 is lb * a / 4
    h = 1e-5
    xs = np.array([[h], [-h]])
    for hh in range(H):
        gp, gm = ko.gate_lower_bound(xs, np.zeros_like(xs), np.full(2, A_log[hh]), lb)[:, 0]
        slope = (gp - gm) / (2 * h)
        np.testing.assert_allclose(slope, lb * np.exp(A_log[hh]) / 4, rtol=1e-8)


def test_bf16_ulp_matches_torch_spacing():
    x = torch.tensor([1.0, 1.5, 3.0, 0.01, -7.25, 1e-3, 100.0], dtype=torch.bfloat16)
    nxt = (x.view(torch.int16) + 1).view(torch.bfloat16)
    spacing = (nxt.double() - x.double()).abs().numpy()
    np.testing.assert_array_equal(ko.bf16_ulp(x.double().numpy()), spacing)


# --- the recurrent step --------------------------------------------------------------

def _unit(seed=4):
    rng = _rng(seed)
    S = 0.1 * rng.standard_normal((128, 128))
    q, k, v = rng.standard_normal((3, 128))
    g = -rng.uniform(0, 3, 128)
    return S, q, k, v, g


def test_no_write_no_decay_leaves_state_and_reads_it():
    S, q, k, v, _ = _unit()
    S2, o = ko.kda_step(S, q, k, v, np.zeros(128), 0.0)
    np.testing.assert_array_equal(S2, S)
    ref = ko.SCALE * np.dot(S.T, q) / np.linalg.norm(q)
    np.testing.assert_allclose(o, ref, rtol=1e-7, atol=1e-12)


def test_decay_only_is_diagonal_scaling():
    S, q, k, v, g = _unit(5)
    S2, o = ko.kda_step(S, q, k, v, g, 0.0)
    np.testing.assert_array_equal(S2, np.diag(np.exp(g)) @ S)
    np.testing.assert_allclose(o, ko.SCALE * (np.diag(np.exp(g)) @ S).T @ (q / np.linalg.norm(q)),
                               rtol=1e-7, atol=1e-12)


def test_unit_key_write_recovers_value():
    S, q, k, v, _ = _unit(6)
    S2, _ = ko.kda_step(S, q, k, v, np.zeros(128), 1.0)
    kn = k / np.linalg.norm(k)
    # S'^T k_hat = v ||k_hat||^2 + (1 - ||k_hat||^2) S^T k_hat with ||k_hat||^2 = 1 - O(1e-8)
    np.testing.assert_allclose(S2.T @ kn, v, atol=1e-6)


def test_householder_form_and_column_closed_form():
    S, q, k, v, g = _unit(7)
    beta = 0.37
    S2, o = ko.kda_step(S, q, k, v, g, beta)
    kn = k / np.sqrt(k @ k + 1e-6)
    qn = q / np.sqrt(q @ q + 1e-6)
    Sd = np.diag(np.exp(g)) @ S
    house = (np.eye(128) - beta * np.outer(kn, kn)) @ Sd + beta * np.outer(kn, v)
    np.testing.assert_allclose(S2, house, rtol=1e-12, atol=1e-14)
    # per value column: o_v = scale * (q.Sd[:, v] + (q.k) u_v), u_v = beta (v_v - k.Sd[:, v])
    o_col = np.empty(128)
    qk = float(qn @ kn)
    for c in range(128):
        u = beta * (v[c] - float(kn @ Sd[:, c]))
        o_col[c] = ko.SCALE * (float(qn @ Sd[:, c]) + qk * u)
    np.testing.assert_allclose(o, o_col, rtol=1e-12, atol=1e-15)


def test_state_orientation_key_rows():
    # the write lands in the key row: a one-hot key touches exactly that row of S
    S = np.zeros((128, 128))
    k = np.zeros(128)
    k[5] = 1.0
    v = np.arange(128, dtype=np.float64)
    S2, _ = ko.kda_step(S, np.ones(128), k, v, np.zeros(128), 1.0)
    nz_rows = np.nonzero(np.abs(S2).sum(axis=1))[0]
    assert list(nz_rows) == [5]
    np.testing.assert_allclose(S2[5], v / np.sqrt(1 + 1e-6), rtol=1e-15)


# --- entry points --------------------------------------------------------------------

def _np(case):
    out = {}
    for key, t in case.items():
        if isinstance(t, torch.Tensor):
            out[key] = t.numpy() if t.dtype == torch.int32 else synth.to_f64(t)
        else:
            out[key] = t
    return out


def test_recurrent_null_rows_and_untouched_slots():
    c = _np(synth.tiny_recurrent_case())
    out, st = ko.recurrent_decode(c["q"], c["k"], c["v"], c["raw_gate"], c["raw_beta"],
                                  c["A_log"], c["dt_bias"], c["state_indices"], c["state"])
    assert np.all(out[2] == 0.0)
    for s in (0, 2, 4, 5, 7):
        np.testing.assert_array_equal(st[s], c["state"][s])
    for s in (1, 3, 6):
        assert np.abs(st[s] - c["state"][s]).max() > 1e-3
    assert np.all(np.abs(out[[0, 1, 3]]).sum(axis=-1) > 0)


def test_out_of_range_slot_is_null():
    c = _np(synth.recurrent_case(2, 2, 4, in_dtype=torch.float32, state_indices=[4, 7]))
    out, st = ko.recurrent_decode(c["q"], c["k"], c["v"], c["raw_gate"], c["raw_beta"],
                                  c["A_log"], c["dt_bias"], c["state_indices"], c["state"])
    assert np.all(out == 0.0)
    np.testing.assert_array_equal(st, c["state"])


def test_packed_is_recurrent_on_split_views_with_bound_minus_5():
    case = synth.packed_case(3, num_slots=6, null_frac=0.34)
    c = _np(case)
    out, st = ko.packed_decode(c["mixed_qkv"], c["raw_gate"], c["raw_beta"], c["A_log"],
                               c["dt_bias"], c["state_indices"], c["state"])
    # split with torch views: [B, 3, 12, 128]
    qkv = case["mixed_qkv"].view(3, 3, 12, 128).double().numpy()
    rg = case["raw_gate"].view(3, 12, 128).double().numpy()
    out2, st2 = ko.recurrent_decode(qkv[:, 0], qkv[:, 1], qkv[:, 2], rg, c["raw_beta"],
                                    c["A_log"], c["dt_bias"], c["state_indices"], c["state"],
                                    lower_bound=-5.0)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(st, st2)


def test_conv_update_matches_torch_causal_conv1d():
    rng = _rng(8)
    C, steps = 3 * 2 * 128, 5
    weight = 0.5 * rng.standard_normal((3, 4, C // 3))
    xs = rng.standard_normal((steps, C))
    cache = np.zeros((C, 3))
    got = []
    for t in range(steps):
        a, cache = ko.conv_update(xs[t], weight, cache)
        got.append(a)
    got = np.stack(got)  # [steps, C]
    # depthwise causal conv: channel ch = sec * (C/3) + c uses weight[sec, :, c]
    w = torch.from_numpy(weight).permute(0, 2, 1).reshape(C, 1, 4)
    seq = torch.from_numpy(xs.T).unsqueeze(0)  # [1, C, steps]
    y = torch.nn.functional.conv1d(seq, w, padding=3, groups=C)[..., :steps]
    ref = torch.nn.functional.silu(y)[0].T.numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)
    np.testing.assert_array_equal(cache, xs[-3:].T)


def test_gated_rmsnorm_matches_torch_rms_norm():
    rng = _rng(9)
    o = 0.05 * rng.standard_normal((4, 6, 128))
    gate = rng.standard_normal((4, 6, 128))
    w = 1 + 0.1 * rng.standard_normal(128)
    got = ko.gated_rmsnorm(o, gate, w, 1e-5)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (128,), torch.from_numpy(w), 1e-5)
    ref = (ref * torch.sigmoid(torch.from_numpy(gate))).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-15)


@pytest.mark.parametrize("lower_bound", [-5.0, None])
def test_fused_is_conv_then_recurrent_then_norm(lower_bound):
    H, rows = 2, 5
    case = synth.fused_case(H, rows, seed=3, null_frac=0.4)
    c = _np(case)
    out, st, cs = ko.fused_decode(c["x"], c["conv_weight"], c["conv_state"], c["raw_gate"][0],
                                  c["raw_beta"][0], c["A_log"], c["dt_bias"], c["state_indices"],
                                  c["state"], c["output_gate"][0], c["norm_weight"],
                                  lower_bound=lower_bound)
    HD = H * 128
    N = c["state"].shape[0]
    idx = c["state_indices"]
    live = (idx > 0) & (idx < N)
    # conv through torch conv1d on [cache, x] windows of the live rows
    w = torch.from_numpy(c["conv_weight"]).permute(0, 2, 1).reshape(3 * HD, 1, 4)
    q = np.zeros((rows, H, 128)); k = np.zeros_like(q); v = np.zeros_like(q)
    for r in range(rows):
        if not live[r]:
            continue
        win = np.concatenate([c["conv_state"][idx[r]], c["x"][r][:, None]], axis=1)
        y = torch.nn.functional.conv1d(torch.from_numpy(win)[None], w, groups=3 * HD)
        a = torch.nn.functional.silu(y)[0, :, 0].numpy()
        q[r], k[r], v[r] = a[:HD].reshape(H, 128), a[HD:2 * HD].reshape(H, 128), a[2 * HD:].reshape(H, 128)
    o, st2 = ko.recurrent_decode(q, k, v, c["raw_gate"][0], c["raw_beta"][0], c["A_log"],
                                 c["dt_bias"], idx, c["state"], lower_bound=lower_bound)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(o), (128,),
                                       torch.from_numpy(c["norm_weight"]), 1e-5)
    ref = (ref * torch.sigmoid(torch.from_numpy(c["output_gate"][0]))).numpy()
    ref[~live] = 0.0
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(st, st2, rtol=1e-13, atol=1e-15)
    # conv cache: live slots shifted with the raw x appended, others untouched
    for s in range(N):
        rows_s = [r for r in range(rows) if live[r] and idx[r] == s]
        if rows_s:
            r = rows_s[0]
            np.testing.assert_array_equal(cs[s][:, :2], c["conv_state"][s][:, 1:])
            np.testing.assert_array_equal(cs[s][:, 2], c["x"][r])
        else:
            np.testing.assert_array_equal(cs[s], c["conv_state"][s])
            np.testing.assert_array_equal(st[s], c["state"][s])
    assert np.all(out[~live] == 0.0)


def test_spec_equals_repeated_single_token_calls():
    case = synth.spec_case(5, 4, seed=1, H=2, lengths=[4, 0, 3, 1, 2], null_count=0)
    c = _np(case)
    out, st = ko.spec_decode(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                             c["state_indices"], c["state"])
    # replay: call t processes the t-th token of every row long enough
    st_r = c["state"].copy()
    out_r = np.zeros_like(out)
    lens = c["lengths"]
    cu = c["cu_seqlens"]
    for t in range(4):
        rows = [n for n in range(5) if lens[n] > t]
        tok = [int(cu[n]) + t for n in rows]
        cu1 = np.arange(len(rows) + 1)
        o1, st_r = ko.spec_decode(c["q"][tok], c["k"][tok], c["v"][tok], c["g"][tok],
                                  c["beta"][tok], cu1, c["state_indices"][rows], st_r)
        out_r[tok] = o1
    np.testing.assert_array_equal(out, out_r)
    np.testing.assert_array_equal(st, st_r)


def test_spec_single_token_matches_recurrent_with_given_gate():
    # T=1 spec with g = the softplus gate equals the recurrent T=1 path
    case = synth.recurrent_case(3, 2, 6, in_dtype=torch.float32, seed=2)
    c = _np(case)
    g = ko.gate_softplus(c["raw_gate"], c["dt_bias"].reshape(2, 128), c["A_log"])
    out_s, st_s = ko.spec_decode(c["q"], c["k"], c["v"], g, c["raw_beta"], np.arange(4),
                                 c["state_indices"], c["state"])
    out_r, st_r = ko.recurrent_decode(c["q"], c["k"], c["v"], c["raw_gate"], c["raw_beta"],
                                      c["A_log"], c["dt_bias"], c["state_indices"], c["state"])
    np.testing.assert_allclose(out_s, out_r, rtol=1e-14, atol=1e-17)
    np.testing.assert_allclose(st_s, st_r, rtol=1e-14, atol=1e-17)


def test_spec_trailing_empty_rows_from_review_repro():
    with open(os.path.join(GOLDEN, "spec_trailing_empty.json")) as f:
        fx = json.load(f)
    R = fx["num_token_rows"]
    n = len(fx["state_indices"])
    case = synth.spec_case(n, 2, seed=4, H=2, lengths=[1, 1, 0, 0], pad_rows=R - 2,
                           num_slots=8)
    case["state_indices"] = torch.tensor(fx["state_indices"], dtype=torch.int32)
    assert case["cu_seqlens"].tolist() == fx["cu_seqlens"]
    c = _np(case)
    out, st = ko.spec_decode(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                             c["state_indices"], c["state"])
    mutated = [s for s in range(8) if not np.array_equal(st[s], c["state"][s])]
    assert mutated == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert np.all(out[r] == 0.0)
    assert np.all(np.abs(out[:2]).sum(-1) > 0)


def test_spec_precomputed_beta_flag():
    case = synth.spec_case(2, 2, seed=5, H=1, lengths=[2, 1])
    c = _np(case)
    rate = scipy.special.expit(c["beta"])
    o1, s1 = ko.spec_decode(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                            c["state_indices"], c["state"], beta_is_logit=True)
    o2, s2 = ko.spec_decode(c["q"], c["k"], c["v"], c["g"], rate, c["cu_seqlens"],
                            c["state_indices"], c["state"], beta_is_logit=False)
    # expit and the oracle's sigmoid may differ in the last bit of beta
    np.testing.assert_allclose(o1, o2, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(s1, s2, rtol=1e-12, atol=1e-15)


def test_verify_outputs_match_spec_and_leave_state():
    case = synth.spec_case(6, 5, seed=11, H=2)
    c = _np(case)
    out_s, _ = ko.spec_decode(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                              c["state_indices"], c["state"])
    before = c["state"].copy()
    out_v, corr, kg = ko.spec_verify(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                                     c["state_indices"], c["state"], t_cap=5)
    np.testing.assert_array_equal(out_v, out_s)
    np.testing.assert_array_equal(c["state"], before)


def test_commit_from_cached_tokens_rebuilds_the_state():
    """Replaying (k, g, u) of the first a tokens equals the spec state after a tokens."""
    case = synth.spec_case(5, 6, seed=12, H=2, lengths=[6, 4, 0, 5, 2])
    c = _np(case)
    _, corr, kg = ko.spec_verify(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                                 c["state_indices"], c["state"], t_cap=6)
    lens, cu, idx = c["lengths"], c["cu_seqlens"], c["state_indices"]
    rng = np.random.default_rng(0)
    for n in range(5):
        if lens[n] == 0:
            continue
        acc = int(rng.integers(0, lens[n] + 1))
        # spec decode of only the accepted tokens of this row
        cu1 = np.array([0, acc])
        tok = list(range(int(cu[n]), int(cu[n]) + acc))
        _, st = ko.spec_decode(c["q"][tok], c["k"][tok], c["v"][tok], c["g"][tok], c["beta"][tok], cu1,
                               idx[n:n + 1], c["state"])
        s = int(idx[n])
        for h in range(2):
            rebuilt = ko.commit_from_cache(c["state"][s, h], kg[s, h, :acc], corr[s, h, :acc])
            np.testing.assert_allclose(rebuilt, st[s, h], rtol=1e-12, atol=1e-14)


def test_verify_cache_capacity_and_null_rows():
    case = synth.spec_case(4, 6, seed=13, H=1, lengths=[6, 3, 2, 4], null_count=1)
    c = _np(case)
    _, corr, kg = ko.spec_verify(c["q"], c["k"], c["v"], c["g"], c["beta"], c["cu_seqlens"],
                                 c["state_indices"], c["state"], t_cap=3)
    idx = c["state_indices"]
    M = c["state"].shape[0]
    for n in range(4):
        s = int(idx[n])
        if not (0 < s < M):
            continue
        L = min(int(c["lengths"][n]), 3)
        t0 = int(c["cu_seqlens"][n])
        for t in range(L):
            np.testing.assert_array_equal(kg[s, 0, t, :128], c["k"][t0 + t, 0])
            np.testing.assert_array_equal(kg[s, 0, t, 128:], c["g"][t0 + t, 0])
    live = {int(s) for s in idx if 0 < int(s) < M}
    for s in range(M):
        if s not in live:
            assert not corr[s].any() and not kg[s].any()


# --- packed fused speculative decode with per-token checkpoints -------------------

def _pf(case):
    c = _np(case)
    return c, ko.packed_fused_decode(c["x"], c["conv_weight"], c["conv_state"], c["raw_gate"], c["raw_beta"],
                                     c["A_log"], c["dt_bias"], c["state_indices"], c["query_start_loc"],
                                     c["num_accepted_tokens"], c["state"], c["output_gate"], c["norm_weight"])


def test_packed_fused_one_token_rows_are_fused_decode():
    """query_start_loc = arange, one column, one accepted token: fused_decode on column 0."""
    case = synth.packed_fused_case(5, 1, H=2, seed=21, lengths=[1] * 5, null_count=1)
    c, (out, st, cs) = _pf(case)
    o2, st2, cs2 = ko.fused_decode(c["x"], c["conv_weight"], c["conv_state"], c["raw_gate"], c["raw_beta"],
                                   c["A_log"], c["dt_bias"], c["state_indices"][:, 0], c["state"],
                                   c["output_gate"], c["norm_weight"])
    np.testing.assert_allclose(out, o2, rtol=1e-14, atol=1e-16)
    np.testing.assert_allclose(st, st2, rtol=1e-14, atol=1e-16)
    np.testing.assert_array_equal(cs, cs2)


def test_packed_fused_checkpoints_are_a_chain_of_fused_calls():
    """Token j of a sequence and checkpoint j equal j+1 single-token fused
    calls on a scratch slot holding the caches of the start slot."""
    N, T, H = 4, 4, 2
    case = synth.packed_fused_case(N, T, H=H, seed=22, lengths=[4, 2, 3, 1])
    c, (out, st, cs) = _pf(case)
    idx, acc, qsl = c["state_indices"], c["num_accepted_tokens"], c["query_start_loc"]
    assert len(set(acc.tolist())) > 1  # several start columns exercised
    for n in range(N):
        s0 = int(idx[n, int(acc[n]) - 1])
        pool = np.stack([np.zeros_like(c["state"][0]), c["state"][s0]])
        conv = np.stack([np.zeros_like(c["conv_state"][0]), c["conv_state"][s0]])
        for j, t in enumerate(range(int(qsl[n]), int(qsl[n + 1]))):
            o1, pool, conv = ko.fused_decode(c["x"][t:t + 1], c["conv_weight"], conv, c["raw_gate"][t:t + 1],
                                             c["raw_beta"][t:t + 1], c["A_log"], c["dt_bias"], np.array([1]),
                                             pool, c["output_gate"][t:t + 1], c["norm_weight"])
            np.testing.assert_allclose(out[t], o1[0], rtol=1e-13, atol=1e-15)
            np.testing.assert_allclose(st[int(idx[n, j])], pool[1], rtol=1e-13, atol=1e-15)
            np.testing.assert_array_equal(cs[int(idx[n, j])], conv[1])
    # every slot no sequence checkpoints to is untouched
    written = {int(idx[n, j]) for n in range(N) for j in range(int(c["lengths"][n]))}
    for s in range(c["state"].shape[0]):
        if s not in written:
            np.testing.assert_array_equal(st[s], c["state"][s])
            np.testing.assert_array_equal(cs[s], c["conv_state"][s])


def test_packed_fused_conv_checkpoint_holds_the_last_three_raw_samples():
    case = synth.packed_fused_case(1, 4, H=1, seed=23, lengths=[4], accepted=[2])
    c, (_, _, cs) = _pf(case)
    idx = c["state_indices"][0]
    hist = np.concatenate([c["conv_state"][int(idx[1])], c["x"].T], axis=1)  # [C, 3 + 4] oldest first
    for j in range(4):
        np.testing.assert_array_equal(cs[int(idx[j])], hist[:, j + 1:j + 4])


def _review_case(fx, seed):
    n = len(fx["state_indices"])
    lens = np.diff(fx["query_start_loc"]).tolist()
    case = synth.packed_fused_case(n, 1, H=2, seed=seed, lengths=lens,
                                   pad_rows=fx["num_token_rows"] - fx["query_start_loc"][-1], num_slots=8,
                                   accepted=fx["num_accepted_tokens"])
    case["state_indices"] = torch.tensor(fx["state_indices"], dtype=torch.int32)
    return case


def test_packed_fused_review_case_a_trailing_padding():
    with open(os.path.join(GOLDEN, "packed_fused_review_cases.json")) as f:
        fx = json.load(f)["case_a"]
    c, (out, st, cs) = _pf(_review_case(fx, 24))
    assert [s for s in range(8) if not np.array_equal(st[s], c["state"][s])] == fx["expected_mutated_slots"]
    assert [s for s in range(8) if not np.array_equal(cs[s], c["conv_state"][s])] == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert np.all(out[r] == 0.0)
    assert np.all(np.abs(out[:2]).sum(-1) > 0)


def test_packed_fused_review_case_b_empty_middle_sequence():
    with open(os.path.join(GOLDEN, "packed_fused_review_cases.json")) as f:
        fx = json.load(f)["case_b"]
    c, (out, st, cs) = _pf(_review_case(fx, 25))
    assert [s for s in range(8) if not np.array_equal(st[s], c["state"][s])] == fx["expected_mutated_slots"]
    for r in fx["expected_zero_rows"]:
        assert np.all(out[r] == 0.0)
    # each live token row is the one-row fused decode on the slot the fixture names
    for r, s in enumerate(fx["expected_row_slots"]):
        o1, st1, _ = ko.fused_decode(c["x"][r:r + 1], c["conv_weight"], c["conv_state"], c["raw_gate"][r:r + 1],
                                     c["raw_beta"][r:r + 1], c["A_log"], c["dt_bias"], np.array([s]), c["state"],
                                     c["output_gate"][r:r + 1], c["norm_weight"])
        np.testing.assert_allclose(out[r], o1[0], rtol=1e-14, atol=1e-16)
        np.testing.assert_allclose(st[s], st1[s], rtol=1e-14, atol=1e-16)


def test_packed_fused_null_start_and_null_checkpoint_columns():
    case = synth.packed_fused_case(3, 3, H=1, seed=26, lengths=[3, 3, 2], accepted=[1, 2, 4])
    case["state_indices"][0, 1] = -1  # checkpoint 1 of sequence 0 is not kept
    case["state_indices"][1, 1] = 0   # sequence 1 starts from the null slot
    c, (out, st, cs) = _pf(case)
    idx, qsl = c["state_indices"], c["query_start_loc"]
    # sequence 0: all three tokens decode, checkpoints 0 and 2 written, slot of column 1 is null
    assert np.all(np.abs(out[0:3]).sum(-1) > 0)
    assert not np.array_equal(st[int(idx[0, 0])], c["state"][int(idx[0, 0])])
    assert not np.array_equal(st[int(idx[0, 2])], c["state"][int(idx[0, 2])])
    # sequence 1 (null start) and sequence 2 (accepted 4 > 3 columns) are null
    assert np.all(out[int(qsl[1]):] == 0.0)
    for n in (1, 2):
        for s in idx[n]:
            if 0 < int(s) < c["state"].shape[0]:
                np.testing.assert_array_equal(st[int(s)], c["state"][int(s)])
                np.testing.assert_array_equal(cs[int(s)], c["conv_state"][int(s)])
