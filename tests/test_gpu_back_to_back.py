"""Dependent calls back to back on one stream, with nothing between them.

Every entry point launches with programmatic stream serialization, so a call
may begin while the previous one drains; each kernel waits for the previous
kernel before its first global-memory access.  Here each call reads the
state the previous call wrote (the same slots, or the checkpoint it wrote
last), as direct launches and replayed from a CUDA graph.  The kernels are
deterministic, so the results must equal, bit for bit, the same calls with
the host waiting for each one to finish before launching the next (which
leaves nothing to overlap).
"""

import pytest
import torch

from linear_attention_decode_02_gb300 import binding, build, synth
from tests import parity as P
from tests import test_gpu_fused as TF
from tests import test_gpu_recurrent as TR
from tests import test_gpu_spec as TS

pytestmark = pytest.mark.gpu
REPEATS = 4


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    yield binding.library()
    binding.kda_set_schedule_override(binding.SCHED_AUTO)


def _back_to_back(calls, graph):
    """calls[k]() for every k, back to back: direct launches or one CUDA graph."""
    if not graph:
        for c in calls:
            c()
        return
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for c in calls:
                c()
    torch.cuda.current_stream().wait_stream(s)
    g.replay()


def _serialised(calls):
    for c in calls:
        c()
        torch.cuda.synchronize()


def _compare(run, tensors, graph):
    """Runs the calls serialised and back to back from the same initial
    tensors; every tensor must come out identical."""
    init = [t.clone() for t in tensors]
    calls = run()
    if graph:  # one warm-up call outside the capture, then the initial values again
        calls[0]()
        torch.cuda.synchronize()
        for t, t0 in zip(tensors, init):
            t.copy_(t0)
    _serialised(calls)
    ref = [t.clone() for t in tensors]
    for t, t0 in zip(tensors, init):
        t.copy_(t0)
    torch.cuda.synchronize()
    _back_to_back(calls, graph)
    torch.cuda.synchronize()
    for t, r in zip(tensors, ref):
        assert torch.equal(t, r), "back-to-back calls differ from serialised calls"


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("schedule,state_dtype", [(binding.SCHED_SPLIT, torch.float32),
                                                  (binding.SCHED_STREAM, torch.bfloat16)])
def test_recurrent_back_to_back(graph, schedule, state_dtype):
    case = synth.recurrent_case(6, 4, 16, seed=501, state_dtype=state_dtype, null_count=1)
    d = P.to_device(case)
    outs = [torch.empty(6, 4, 128, dtype=torch.bfloat16, device="cuda") for _ in range(REPEATS)]
    binding.kda_set_schedule_override(schedule)
    try:
        _compare(lambda: [lambda o=o: TR._run_recurrent(d, out=o) for o in outs], [d["state"]] + outs, graph)
    finally:
        binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("schedule", [binding.SCHED_SPLIT, binding.SCHED_STREAM])
def test_fused_back_to_back(graph, schedule):
    case = synth.fused_case(8, 5, seed=502, null_frac=0.2)
    d = TF._device_case(case)
    outs = [torch.empty(1, 5, 8, 128, dtype=torch.bfloat16, device="cuda") for _ in range(REPEATS)]
    binding.kda_set_schedule_override(schedule)
    try:
        _compare(lambda: [lambda o=o: TF._run(d, out=o) for o in outs], [d["state"], d["conv_state"]] + outs,
                 graph)
    finally:
        binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("schedule", [binding.SCHED_SPLIT, binding.SCHED_MMA])
def test_spec_back_to_back(graph, schedule):
    case = synth.spec_case(5, 4, seed=503, H=4, lengths=[4, 2, 0, 3, 4], state_dtype=torch.bfloat16)
    d = P.to_device(case)
    outs = [torch.empty(case["q"].shape, dtype=torch.bfloat16, device="cuda") for _ in range(REPEATS)]
    binding.kda_set_schedule_override(schedule)
    try:
        _compare(lambda: [lambda o=o: TS._run(d, 4, out=o) for o in outs], [d["state"]] + outs, graph)
    finally:
        binding.kda_set_schedule_override(binding.SCHED_AUTO)


@pytest.mark.parametrize("graph", [False, True])
@pytest.mark.parametrize("cluster", [0, 2])
def test_packed_fused_back_to_back(graph, cluster):
    """Each call starts from the checkpoint the previous call wrote last: one
    accepted token, two checkpoint columns, swapped between calls."""
    N, T = 3, 2
    case = synth.packed_fused_case(N, T, H=2, seed=504, lengths=[T] * N, accepted=1, cols=T)
    d = P.to_device(case)
    idx_a = d["state_indices"].clone()
    idx_b = idx_a[:, [1, 0]].contiguous()
    seq = [idx_a, idx_b, idx_a, idx_b]
    outs = [torch.empty(N * T, 2, 128, dtype=torch.bfloat16, device="cuda") for _ in range(REPEATS)]

    def call(k):
        return binding.kda_packed_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"],
                                               d["raw_beta"], d["A_log"], d["dt_bias"], seq[k],
                                               d["query_start_loc"], d["num_accepted_tokens"], d["state"],
                                               d["output_gate"], d["norm_weight"], out=outs[k])
    binding.kda_set_split_override(cluster)
    try:
        _compare(lambda: [lambda k=k: call(k) for k in range(REPEATS)], [d["state"], d["conv_state"]] + outs,
                 graph)
    finally:
        binding.kda_set_split_override(0)


def test_concurrent_host_threads_on_their_own_streams():
    """Two host threads drive the library at once, each on its own stream with
    its own state pool (chains of dependent recurrent and speculative calls):
    both end exactly where the same calls run one after another end."""
    import threading

    def make(seed):
        rc = synth.recurrent_case(8, 4, 32, seed=seed, state_dtype=torch.bfloat16)
        sc = synth.spec_case(6, 4, seed=seed + 1, H=4, state_dtype=torch.bfloat16)
        return P.to_device(rc), P.to_device(sc)

    def chain(dr, ds, reps):
        for _ in range(reps):
            TR._run_recurrent(dr)
            TS._run(ds, 4)

    cases = [make(601), make(611)]
    init = [(dr["state"].clone(), ds["state"].clone()) for dr, ds in cases]
    for dr, ds in cases:
        chain(dr, ds, 20)
    torch.cuda.synchronize()
    ref = [(dr["state"].clone(), ds["state"].clone()) for dr, ds in cases]
    for (dr, ds), (s_r, s_s) in zip(cases, init):
        dr["state"].copy_(s_r)
        ds["state"].copy_(s_s)
    torch.cuda.synchronize()
    errors = []

    def worker(i):
        try:
            st = torch.cuda.Stream()
            with torch.cuda.stream(st):
                chain(*cases[i], 20)
            st.synchronize()
        except Exception as e:  # noqa: BLE001 - reported below
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for (dr, ds), (r_r, r_s) in zip(cases, ref):
        assert torch.equal(dr["state"], r_r) and torch.equal(ds["state"], r_s)
