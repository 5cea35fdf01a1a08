"""The oracle pins catch plausible mistakes (CPU only).

Each case plants one mistake in the oracle (a transposed operand, a dropped
term, a wrong sign or axis) by patching one of its functions, runs every pin
of test_oracle_pins, and requires at least one pin to fail.  Nothing here
touches the CUDA path.
"""

import contextlib

import numpy as np
import pytest

from oracle import kda_oracle as ko
from tests import test_oracle_pins as pins

ORIG_STEP = ko.kda_step
ORIG_GATE_SP = ko.gate_softplus
ORIG_GATE_LB = ko.gate_lower_bound
ORIG_L2 = ko.l2_normalize
ORIG_CONV_TAPS = ko.conv_weight_taps
ORIG_RMS = ko.gated_rmsnorm


def _step_variant(kind):
    def step(S, q, k, v, g, beta, scale=ko.SCALE):
        S = np.asarray(S, np.float64)
        qh, kh = ko.l2_normalize(q), ko.l2_normalize(k)
        e = np.exp(np.asarray(g, np.float64))
        Sd = S * e[None, :] if kind == "decay_columns" else e[:, None] * S
        read = Sd @ kh if kind == "transposed_read" else Sd.T @ kh
        b = 1.0 if kind == "dropped_beta" else float(beta)
        sign = 1.0 if kind == "delta_sign" else -1.0
        u = b * (np.asarray(v, np.float64) + sign * read)
        S_new = Sd + (np.outer(u, kh) if kind == "transposed_write" else np.outer(kh, u))
        src = Sd if kind == "output_before_write" else S_new
        o = scale * (src.T @ (np.asarray(q, np.float64) if kind == "unnormalised_q" else qh))
        if kind == "output_transposed":
            o = scale * (src @ qh)
        return S_new, o
    return step


MUTATIONS = {
    "transposed_read": ("kda_step", _step_variant("transposed_read")),
    "transposed_write": ("kda_step", _step_variant("transposed_write")),
    "decay_columns": ("kda_step", _step_variant("decay_columns")),
    "dropped_beta": ("kda_step", _step_variant("dropped_beta")),
    "delta_sign": ("kda_step", _step_variant("delta_sign")),
    "output_before_write": ("kda_step", _step_variant("output_before_write")),
    "unnormalised_q": ("kda_step", _step_variant("unnormalised_q")),
    "output_transposed": ("kda_step", _step_variant("output_transposed")),
    "softplus_gate_sign": ("gate_softplus", lambda r, d, a: -ORIG_GATE_SP(r, d, a)),
    "softplus_gate_no_bias": ("gate_softplus", lambda r, d, a: ORIG_GATE_SP(r, np.zeros_like(d), a)),
    "bounded_gate_flipped": ("gate_lower_bound",
                             lambda r, d, a, lb: float(lb) - ORIG_GATE_LB(r, d, a, lb)),
    "bounded_gate_no_A": ("gate_lower_bound", lambda r, d, a, lb: ORIG_GATE_LB(r, d, np.zeros_like(a), lb)),
    "bounded_gate_A_not_exp": ("gate_lower_bound",
                               lambda r, d, a, lb: float(lb) * ko.sigmoid(
                                   np.asarray(a, np.float64)[..., :, None] *
                                   (np.asarray(r, np.float64) + np.asarray(d, np.float64)))),
    "l2_eps_outside": ("l2_normalize",
                       lambda x, eps=ko.L2_EPS: np.asarray(x, np.float64) /
                       (np.sqrt(np.sum(np.asarray(x, np.float64) ** 2, -1, keepdims=True)) + 1e-2)),
    "conv_taps_reversed": ("conv_weight_taps", lambda w: ORIG_CONV_TAPS(w)[:, ::-1]),
    "start_from_column_zero": ("start_slot", lambda row, acc: int(row[0])),
    "start_from_accepted_column": ("start_slot", lambda row, acc: int(row[min(int(acc), len(row) - 1)])),
    "rmsnorm_without_gate": ("gated_rmsnorm",
                             lambda o, g, w, eps=ko.FUSED_NORM_EPS: ORIG_RMS(o, np.full_like(g, 50.0), w, eps)),
}


@contextlib.contextmanager
def planted(name):
    attr, fn = MUTATIONS[name]
    saved = getattr(ko, attr)
    setattr(ko, attr, fn)
    try:
        yield
    finally:
        setattr(ko, attr, saved)


def _pins():
    out = []
    for name in dir(pins):
        if not name.startswith("test_"):
            continue
        fn = getattr(pins, name)
        if name == "test_fused_is_conv_then_recurrent_then_norm":
            out += [(name + "[-5]", lambda fn=fn: fn(-5.0)), (name + "[None]", lambda fn=fn: fn(None))]
        else:
            out.append((name, fn))
    return out


def test_unmutated_oracle_passes_every_pin():
    for _, fn in _pins():
        fn()


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_each_planted_mistake_fails_a_pin(mutation):
    caught = []
    with planted(mutation):
        for name, fn in _pins():
            try:
                fn()
            except (AssertionError, ValueError, IndexError):
                caught.append(name)
    assert caught, f"no pin catches the planted mistake {mutation!r}"
