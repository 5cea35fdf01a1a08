"""Failure detection without a GPU fault: the bounded waits give up.

The streaming kernels bound every mbarrier wait in time and report a
timeout in a device error word instead of spinning.  The self-test launches
one warp that waits on a barrier nothing completes; after ~2 s it must set
bit 2 of the error word and return, leaving the context usable.
"""

import time

import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return binding.library()


def test_bounded_wait_times_out_and_reports():
    binding.kda_device_error(clear=True)
    t0 = time.time()
    binding.kda_selftest_wait_timeout()
    flags = binding.kda_device_error(clear=True)
    elapsed = time.time() - t0
    assert flags & 4, f"self-test bit not set (flags={flags})"
    assert 1.5 < elapsed < 30.0
    # the context still runs a decode, and the word is clean afterwards
    case = synth.tiny_recurrent_case()
    d = P.to_device(case)
    out = binding.kda_recurrent_decode(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["A_log"],
                                       d["dt_bias"], d["state_indices"], d["state"])
    torch.cuda.synchronize()
    ref_out, _ = P.oracle_recurrent(case)
    P.assert_out_close(out, ref_out)
    assert binding.kda_device_error() == 0
