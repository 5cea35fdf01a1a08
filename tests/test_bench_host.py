"""Host-side pieces of bench.py (CPU): the byte models and the validity check
of the recorded ncu traffic against each kernel's sources."""

import json
import os

import bench

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_source_closure_follows_local_includes():
    t1 = bench.source_closure("kda_t1.cu")
    assert t1[0] != "" and "kda_t1.cu" in t1 and "kda_kernels.cuh" in t1 and "kda_device.cuh" in t1
    assert "kda_stream.cu" not in t1 and "kda_api.cu" not in t1
    st = bench.source_closure("kda_stream.cu")
    assert {"kda_stream_common.cuh", "kda_async.cuh", "kda_kernels.cuh"} <= set(st)
    assert bench.source_closure("") == [] and bench.source_closure("no_such_file.cu") == []


def test_kernel_hashes_differ_per_translation_unit():
    hashes = {f: bench.kernel_source_hash(f) for f in ("kda_t1.cu", "kda_stream.cu", "kda_spec.cu", "kda_fused.cu")}
    assert len(set(hashes.values())) == 4
    assert all(len(h) == 16 for h in hashes.values())


def test_recorded_traffic_is_well_formed():
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    with open(path) as f:
        rec = json.load(f)
    for kind, e in rec["kernels"].items():
        assert e["source"].endswith(".cu") and os.path.isfile(os.path.join(bench.CSRC, e["source"])), kind
        assert e["dram_bytes_per_launch"] == e["dram_read_per_launch"] + e["dram_write_per_launch"]
        assert "--clock-control none" in e["command"]
        got = bench.ncu_traffic(kind)
        assert got is None or got == e["dram_bytes_per_launch"]
    assert bench.ncu_traffic("no_such_workload") is None


def test_byte_models():
    # fp32 state, bf16 activations: 2*64 KiB state + 4*256 B vectors + 2 B beta + 256 B out per unit
    assert bench.bytes_t1(1, 0, 1, 4) - bench.bytes_t1(0, 0, 1, 4) == 2 * 128 * 128 * 4 + 4 * 256 + 2 + 256 + 4  # + the slot index


def test_packed_fused_byte_model():
    # one sequence of two tokens, one checkpoint column, H=1, fp32: state and conv
    # cache read once and written once, two tokens' activations, no padding
    unit = 128 * 128 * 4 + 3 * 3 * 128 * 2
    per_tok = 3 * 128 * 2 + 128 * 2 + 2 + 128 * 2 + 128 * 2
    params = 3 * 4 * 128 * 4 + 4 + 128 * 4 + 128 * 4
    meta = 2 * 4 + 4 + 4
    assert bench.bytes_packed_fused([2], 1, 1, 4, 2) == 2 * unit + 2 * per_tok + params + meta
    # an empty sequence adds only its metadata and padding rows add zero output
    assert bench.bytes_packed_fused([2, 0], 1, 1, 4, 3) == 2 * unit + 2 * per_tok + 128 * 2 + params + 3 * 4 + 8 + 8


def test_oracle_baseline_runs_on_several_single_threaded_processes():
    (g1, r1, e1), per_step, procs = bench.oracle_rates(0.4, H=2, workers=2, steps=2)
    assert procs == 2 and len(per_step) == 2
    assert g1 > 0 and r1 >= 8 and e1 >= 0.2
    for g, r, e in per_step:
        assert g > 0 and r >= 16 and e >= 0.2


def test_source_hash_ignores_comments_but_not_code():
    src = 'int f(int x) {  // doubles\n  /* see\n below */ return 2 * x; }\nconst char* s = "// kept";\n'
    assert bench.code_only(src) == bench.code_only(src.replace("// doubles", "// twice").replace("see", "look"))
    assert bench.code_only(src) != bench.code_only(src.replace("2 * x", "3 * x"))
    assert '"// kept"' in bench.code_only(src)
