"""Helpers for the GPU parity tests: device copies of seeded cases, the
float64 oracle on all or on a sample of rows, and the comparisons.

Rows are independent (each live row owns a unique slot), so the oracle can
run on any subset of rows over a compact pool holding only their slots; its
results for those rows are the ones of the full call.
"""

from __future__ import annotations

import os

import numpy as np
import torch

from oracle import kda_oracle as ko
from linear_attention_decode_02_gb300 import synth

OUT_ATOL = 2e-3        # bf16 outputs, max abs error
F32_STATE_ATOL = 1e-4  # float32 state, max abs error
# bf16 state: one bf16 ulp of the oracle value, floored at the float32
# arithmetic error of the update itself (128-term dots of terms ~0.1-1 carry
# ~128 * 2^-24 absolute error), which matters only where S' nearly cancels.
BF16_STATE_FLOOR = 1e-6


def dev(t):
    """Copy to cuda:0 keeping the strides of a dense permuted view."""
    return t.to("cuda")


def to_device(case):
    return {k: (dev(v) if isinstance(v, torch.Tensor) else v) for k, v in case.items()}


def f64(t):
    return synth.to_f64(t)


def _compact(idx, num_slots, rows):
    """Slots used by `rows` remapped to 1..n (0 stays the null slot)."""
    live = [r for r in rows if 0 < int(idx[r]) < num_slots]
    slots = sorted({int(idx[r]) for r in live})
    remap = {s: i + 1 for i, s in enumerate(slots)}
    sub_idx = np.array([remap.get(int(idx[r]), -1) if r in set(live) else -1 for r in rows])
    return slots, remap, sub_idx


def _pool(state_cpu, slots):
    H = state_cpu.shape[1]
    pool = np.zeros((len(slots) + 1, H, 128, 128))
    if slots:
        pool[1:] = f64(state_cpu[torch.tensor(slots, dtype=torch.long)])
    return pool


def oracle_recurrent(case, rows=None, lower_bound=None, scale=ko.SCALE):
    """Oracle out for `rows` and the new state of their slots: (out, {slot: S})."""
    idx = case["state_indices"].numpy()
    B = idx.shape[0]
    rows = list(range(B)) if rows is None else list(rows)
    slots, remap, sub_idx = _compact(idx, case["state"].shape[0], rows)
    r = torch.tensor(rows, dtype=torch.long)
    out, st = ko.recurrent_decode(f64(case["q"][r]), f64(case["k"][r]), f64(case["v"][r]),
                                  f64(case["raw_gate"][r]), f64(case["raw_beta"][r]), f64(case["A_log"]),
                                  f64(case["dt_bias"]), sub_idx, _pool(case["state"], slots),
                                  lower_bound=lower_bound, scale=scale)
    return out, {s: st[remap[s]] for s in slots}


def oracle_packed(case, rows=None):
    idx = case["state_indices"].numpy()
    B = idx.shape[0]
    rows = list(range(B)) if rows is None else list(rows)
    slots, remap, sub_idx = _compact(idx, case["state"].shape[0], rows)
    r = torch.tensor(rows, dtype=torch.long)
    out, st = ko.packed_decode(f64(case["mixed_qkv"][r]), f64(case["raw_gate"][r]), f64(case["raw_beta"][r]),
                               f64(case["A_log"]), f64(case["dt_bias"]), sub_idx, _pool(case["state"], slots))
    return out, {s: st[remap[s]] for s in slots}


def oracle_fused(case, rows=None, lower_bound=-5.0, norm_eps=1e-5):
    """(out, {slot: S}, {slot: conv cache [C, 3]}) for `rows`."""
    idx = case["state_indices"].numpy()
    n_rows = idx.shape[0]
    rows = list(range(n_rows)) if rows is None else list(rows)
    slots, remap, sub_idx = _compact(idx, case["state"].shape[0], rows)
    r = torch.tensor(rows, dtype=torch.long)
    cs = case["conv_state"]
    conv = np.zeros((len(slots) + 1, cs.shape[1], 3))
    if slots:
        conv[1:] = f64(cs[torch.tensor(slots, dtype=torch.long)])
    rg = case["raw_gate"].reshape(n_rows, *case["raw_gate"].shape[-2:])
    rb = case["raw_beta"].reshape(n_rows, case["raw_beta"].shape[-1])
    og = case["output_gate"].reshape(n_rows, *case["output_gate"].shape[-2:])
    out, st, cst = ko.fused_decode(f64(case["x"][r]), f64(case["conv_weight"]), conv, f64(rg[r]), f64(rb[r]),
                                   f64(case["A_log"]), f64(case["dt_bias"]), sub_idx,
                                   _pool(case["state"], slots), f64(og[r]), f64(case["norm_weight"]),
                                   lower_bound=lower_bound, norm_eps=norm_eps)
    return out, {s: st[remap[s]] for s in slots}, {s: cst[remap[s]] for s in slots}


def oracle_spec(case, rows=None, beta_is_logit=True, scale=ko.SCALE):
    """Oracle over the sequences `rows`: ({token_row: out [H,128]}, {slot: S})."""
    idx = case["state_indices"].numpy()
    cu = case["cu_seqlens"].numpy()
    N = idx.shape[0]
    rows = list(range(N)) if rows is None else list(rows)
    slots, remap, sub_idx = _compact(idx, case["state"].shape[0], rows)
    R = case["q"].shape[0]
    tok, sub_cu = [], [0]
    for n in rows:
        t0, t1 = max(int(cu[n]), 0), min(int(cu[n + 1]), R)
        ts = list(range(t0, t1)) if t1 > t0 else []
        tok += ts
        sub_cu.append(sub_cu[-1] + len(ts))
    t = torch.tensor(tok, dtype=torch.long)
    out, st = ko.spec_decode(f64(case["q"][t]), f64(case["k"][t]), f64(case["v"][t]), f64(case["g"][t]),
                             f64(case["beta"][t]), np.array(sub_cu), sub_idx, _pool(case["state"], slots),
                             beta_is_logit=beta_is_logit, scale=scale)
    return {tr: out[i] for i, tr in enumerate(tok)}, {s: st[remap[s]] for s in slots}


# ---- comparisons ----------------------------------------------------------------

def assert_out_close(gpu_out, ref, atol=OUT_ATOL, what="out"):
    got = gpu_out.detach().double().cpu().numpy()
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max(initial=0.0) <= atol, f"{what}: max abs error {err.max():.3e} > {atol:.1e}"
    return float(err.max(initial=0.0))


# Per test: elements that passed the gated-output check only through the
# one-ulp branch (error above 2e-3 but within one bf16 ulp of the oracle),
# out of all elements checked, and the worst error in half-ulps.  The test
# session prints these in its summary.
ULP_BRANCH = {}
# Drift curves of the chained-step diagnostics: {name: [(step, out err, state err)]}.
DRIFT = {}


def assert_out_close_or_ulp(gpu_out, ref, atol=OUT_ATOL, what="out"):
    """Each element within atol or within one bf16 ulp of the oracle."""
    got = gpu_out.detach().double().cpu().numpy()
    err = np.abs(got - ref)
    ulp = ko.bf16_ulp(ref)
    ok = (err <= atol) | (err <= ulp)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert ok.all(), f"{what}: {int((~ok).sum())} elements beyond max(2e-3, 1 bf16 ulp); worst {err.max():.3e}"
    test = os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]
    n_ulp, n_all, worst = ULP_BRANCH.get(test, (0, 0, 0.0))
    branch = err > atol
    ULP_BRANCH[test] = (n_ulp + int(branch.sum()), n_all + err.size,
                        max(worst, float((2 * err[branch] / ulp[branch]).max(initial=0.0))))
    return float(err.max(initial=0.0))


def assert_state_close(gpu_slot, ref):
    """fp32 state: max abs <= 1e-4; bf16 state: within one bf16 ulp of the oracle."""
    got = gpu_slot.detach().double().cpu().numpy()
    err = np.abs(got - ref)
    if gpu_slot.dtype == torch.float32:
        assert err.max() <= F32_STATE_ATOL, f"fp32 state max abs error {err.max():.3e}"
    else:
        ulp = np.maximum(ko.bf16_ulp(ref), BF16_STATE_FLOOR)
        bad = err > ulp
        assert not bad.any(), f"bf16 state: {int(bad.sum())} elements beyond 1 ulp; worst {err.max():.3e}"
    return float(err.max())


def assert_untouched(before, after, touched_slots):
    """Every slot not in `touched_slots` is bit-identical (whole-pool compare on device)."""
    mask = torch.ones(before.shape[0], dtype=torch.bool, device=before.device)
    if touched_slots:
        mask[torch.tensor(sorted(touched_slots), dtype=torch.long, device=before.device)] = False
    assert torch.equal(before[mask], after[mask]), "an untouched slot changed"


def live_slots(idx, num_slots):
    return sorted({int(s) for s in idx.tolist() if 0 < int(s) < num_slots})


def oracle_verify(case, t_cap, rows=None, beta_is_logit=True, scale=ko.SCALE):
    """Oracle verify mode over the sequences `rows`:
    ({token_row: out [H,128]}, {slot: corr [H,t_cap,128]}, {slot: kg [H,t_cap,256]})."""
    idx = case["state_indices"].numpy()
    cu = case["cu_seqlens"].numpy()
    N = idx.shape[0]
    rows = list(range(N)) if rows is None else list(rows)
    slots, remap, sub_idx = _compact(idx, case["state"].shape[0], rows)
    R = case["q"].shape[0]
    tok, sub_cu = [], [0]
    for n in rows:
        t0, t1 = max(int(cu[n]), 0), min(int(cu[n + 1]), R)
        ts = list(range(t0, t1)) if t1 > t0 else []
        tok += ts
        sub_cu.append(sub_cu[-1] + len(ts))
    t = torch.tensor(tok, dtype=torch.long)
    out, corr, kg = ko.spec_verify(f64(case["q"][t]), f64(case["k"][t]), f64(case["v"][t]), f64(case["g"][t]),
                                   f64(case["beta"][t]), np.array(sub_cu), sub_idx, _pool(case["state"], slots),
                                   t_cap, beta_is_logit=beta_is_logit, scale=scale)
    return ({tr: out[i] for i, tr in enumerate(tok)}, {s: corr[remap[s]] for s in slots},
            {s: kg[remap[s]] for s in slots})


def oracle_packed_fused(case, seqs=None, lower_bound=-5.0, norm_eps=1e-5):
    """Oracle over the sequences `seqs` on a compact pool of their slots:
    ({token_row: out [H,128]}, {slot: S}, {slot: conv [C,3]}) for every slot
    the oracle wrote."""
    idx = case["state_indices"].numpy()
    qsl = case["query_start_loc"].numpy()
    acc = case["num_accepted_tokens"].numpy()
    M = case["state"].shape[0]
    N, cols = idx.shape
    seqs = list(range(N)) if seqs is None else list(seqs)
    slots = sorted({int(s) for n in seqs for s in idx[n] if 0 < int(s) < M})
    remap = {s: i + 1 for i, s in enumerate(slots)}
    sub_idx = np.array([[remap.get(int(s), -1) for s in idx[n]] for n in seqs]).reshape(len(seqs), cols)
    R = case["x"].shape[0]
    tok, sub_qsl = [], [0]
    for n in seqs:
        t0, t1 = max(int(qsl[n]), 0), min(int(qsl[n + 1]), R)
        ts = list(range(t0, t1)) if t1 > t0 else []
        tok += ts
        sub_qsl.append(sub_qsl[-1] + len(ts))
    t = torch.tensor(tok, dtype=torch.long)
    sl = torch.tensor(slots, dtype=torch.long)
    pool = _pool(case["state"], slots)
    conv = np.zeros((len(slots) + 1,) + tuple(case["conv_state"].shape[1:]))
    if slots:
        conv[1:] = f64(case["conv_state"][sl])
    out, st, cs = ko.packed_fused_decode(f64(case["x"][t]), f64(case["conv_weight"]), conv, f64(case["raw_gate"][t]),
                                         f64(case["raw_beta"][t]), f64(case["A_log"]), f64(case["dt_bias"]),
                                         sub_idx, np.array(sub_qsl), acc[seqs], pool, f64(case["output_gate"][t]),
                                         f64(case["norm_weight"]), lower_bound=lower_bound, norm_eps=norm_eps)
    written = {}
    for s in slots:
        i = remap[s]
        if not (np.array_equal(st[i], pool[i]) and np.array_equal(cs[i], conv[i])):
            written[s] = i
    return ({tr: out[i] for i, tr in enumerate(tok)}, {s: st[i] for s, i in written.items()},
            {s: cs[i] for s, i in written.items()})


def packed_fused_written_slots(case):
    """Slots the call must write: checkpoint columns j < len of live sequences."""
    idx = case["state_indices"].numpy()
    qsl = case["query_start_loc"].numpy()
    acc = case["num_accepted_tokens"].numpy()
    M, R = case["state"].shape[0], case["x"].shape[0]
    N, cols = idx.shape
    out = set()
    for n in range(N):
        t0, t1 = max(int(qsl[n]), 0), min(int(qsl[n + 1]), R)
        a = int(acc[n])
        if t1 <= t0 or not 1 <= a <= cols or not 0 < int(idx[n, a - 1]) < M:
            continue
        out |= {int(s) for s in idx[n, :min(t1 - t0, cols)] if 0 < int(s) < M}
    return out
