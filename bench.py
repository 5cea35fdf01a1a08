"""Benchmark of the KDA decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Headline workload: Kimi-Linear equal-head T=1 recurrent decode, H=32,
K=V=128, float32 state pool [1024, 32, 128, 128], B=512 rows on distinct
slots, bf16 activations, softplus gate.  A step is one kda_recurrent_decode
call; two disjoint slot sets alternate between steps and every step moves
1.07 GB of state, far more than the 129 MB L2, so no flush is needed there.

Metric: achieved HBM GB/s of the algorithmic bytes (live state read + write
plus the activations and parameters read and the output written) per call;
ms_per_step is the time per call.  The line also carries the same metric end
to end (pinned host inputs copied in and the output copied out each step),
the roofline of the kernel against the measured copy bandwidth, the SM clocks
seen during the timed region, per-path / per-batch measurements of the four
entry points, and the float64 oracle timed on the host cores.

Multi-GPU: every rank runs its own replica (the decode units are independent
and need no exchange); value sums the bytes of all ranks over the slowest
rank's time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_decode_02_gb300 import binding, synth  # noqa: E402

D = 128
METRIC = "KDA decode µs/call and achieved HBM GB/s (state R+W) vs GB300 peak, 1 GPU"
HEADLINE = dict(workload="kimi_linear_t1_recurrent", H=32, B=512, num_slots=1024, state="float32",
                activations="bfloat16", gate="softplus")
FALLBACK_HBM_GBS = 6800.0


# ---- byte model (algorithmic bytes per call) -------------------------------------

def bytes_t1(live, null, H, state_esize, act_esize=2):
    """Live units: state R+W + q, k, v, raw gate + beta + bf16 out; null rows: index + zero out."""
    per_live = 2 * D * D * state_esize + 4 * D * act_esize + act_esize + 2 * D
    params = H * 4 + H * D * 4
    return live * H * per_live + null * H * 2 * D + (live + null) * 4 + params


def bytes_fused(live, null, H, state_esize):
    """Live units add the conv input (3x128 bf16), the conv cache R+W and the output gate."""
    per_live = 2 * D * D * state_esize + 3 * D * 2 + 2 * (3 * 3 * D * 2) + D * 2 + 2 + D * 2 + D * 2
    params = H * 4 + H * D * 4 + 3 * 4 * H * D * 4 + D * 4
    return live * H * per_live + null * H * 2 * D + (live + null) * 4 + params


def bytes_spec(tokens_live, rows_live, rows, R, H, state_esize):
    """Per live row: state R+W once; per live token: q, k, v (bf16), g (fp32), beta, out."""
    per_tok = 3 * D * 2 + D * 4 + 2 + 2 * D
    zero_tok = R - tokens_live
    return (rows_live * H * 2 * D * D * state_esize + tokens_live * H * per_tok + zero_tok * H * 2 * D
            + (rows + 1) * 4 + rows * 4)


# ---- environment -------------------------------------------------------------------

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


def kernel_source_hash():
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "linear_attention_decode_02_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kind):
    """DRAM bytes per launch from the committed ncu summary, if the kernels are unchanged since."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_hash") != kernel_source_hash():
        return None
    entry = rec.get("kernels", {}).get(kind)
    if not entry:
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index=0):
        self.samples = []
        self.proc = None
        self.gpu = self._physical_id(device_index)

    @staticmethod
    def _physical_id(i):
        try:
            uuid = str(torch.cuda.get_device_properties(i).uuid)
            return uuid if uuid.startswith("GPU-") else "GPU-" + uuid
        except Exception:
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            return vis.split(",")[i] if vis else str(i)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0, t1):
        rows = [p for (t, p) in self.samples if t0 <= t <= t1] or [p for (_, p) in self.samples]
        if not rows:
            return None
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        sm = [float(p[0]) for p in rows if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in rows if p[1].replace(".", "").isdigit()]
        reasons = sorted({names[i] for p in rows for i in range(4) if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ---- timing helpers ------------------------------------------------------------------

def time_direct(fn, steps, warmup, stream, barrier):
    """Average ms per call over `steps` back-to-back launches on `stream`."""
    for i in range(warmup):
        fn(i)
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    e0.record(stream)
    for i in range(steps):
        fn(i)
    e1.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    barrier()
    return e0.elapsed_time(e1) / steps, (wall0, wall1)


def time_graph(calls, reps, flush):
    """Per-call ms of a CUDA graph of `calls` launches, L2 flushed before each replay."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for fn in calls:
            fn()
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        for fn in calls:
            fn()
    times = []
    for r in range(reps + 2):
        flush.fill_(r)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if r >= 2:
            times.append(e0.elapsed_time(e1) / len(calls))
    return statistics.median(times)


# ---- workloads -------------------------------------------------------------------------

def recurrent_device_case(B, H, num_slots, seed, state_dtype=torch.float32, null_count=0, n_sets=2):
    """Device inputs with `n_sets` disjoint slot sets (alternated between steps)."""
    g = torch.Generator().manual_seed(seed)
    case = synth.recurrent_case(B, H, 2, seed=seed, state_dtype=state_dtype, state_indices=[1] * B)
    d = {k: v.cuda() for k, v in case.items() if k not in ("state", "state_indices")}
    perm = (torch.randperm(num_slots - 1, generator=g) + 1).to(torch.int32)
    sets = []
    for i in range(n_sets):
        idx = perm[i * B:(i + 1) * B].clone()
        if null_count:
            idx = synth.with_nulls(g, idx, null_count)
        sets.append(idx.cuda())
    gen = torch.Generator(device="cuda").manual_seed(seed)
    state = torch.empty(num_slots, H, D, D, dtype=torch.float32, device="cuda")
    state.normal_(0.0, 0.1, generator=gen)
    d["state"] = state.to(state_dtype) if state_dtype != torch.float32 else state
    d["sets"] = sets
    return d


def run_recurrent(d, i, out):
    binding.kda_recurrent_decode(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["A_log"], d["dt_bias"],
                                 d["sets"][i % len(d["sets"])], d["state"], out=out)


def headline(args, rank, world, barrier, peaks):
    H, B, N = HEADLINE["H"], HEADLINE["B"], HEADLINE["num_slots"]
    d = recurrent_device_case(B, H, N, seed=rank)
    out = torch.empty(B, H, D, dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    ms, (w0, w1) = time_direct(lambda i: run_recurrent(d, i, out), args.steps, args.warmup, stream, barrier)
    clocks.stop()
    nbytes = bytes_t1(B, 0, H, 4)
    return ms, nbytes, clocks.summary(w0, w1), d, out


def e2e_recurrent(d, steps, warmup, barrier):
    """Same call with pinned-host activations copied in and the output copied out every step."""
    host = {k: d[k].cpu().pin_memory() for k in ("q", "k", "v", "raw_gate", "raw_beta")}
    host["sets"] = [s.cpu().pin_memory() for s in d["sets"]]
    out = torch.empty(d["q"].shape, dtype=torch.bfloat16, device="cuda")
    out_h = torch.empty(out.shape, dtype=torch.bfloat16).pin_memory()
    idx = torch.empty_like(d["sets"][0])

    def step(i):
        for k in ("q", "k", "v", "raw_gate", "raw_beta"):
            d[k].copy_(host[k], non_blocking=True)
        idx.copy_(host["sets"][i % len(host["sets"])], non_blocking=True)
        binding.kda_recurrent_decode(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["A_log"],
                                     d["dt_bias"], idx, d["state"], out=out)
        out_h.copy_(out, non_blocking=True)

    ms, _ = time_direct(step, steps, warmup, torch.cuda.current_stream(), barrier)
    h2d = sum(host[k].numel() * host[k].element_size() for k in ("q", "k", "v", "raw_gate", "raw_beta"))
    h2d += host["sets"][0].numel() * 4
    d2h = out_h.numel() * out_h.element_size()
    return ms, h2d, d2h


def path_measurements(flush, peak):
    """Per-path and per-batch CUDA-graph timings (L2 flushed before each replay)."""
    res = {}

    def rec(name, ms, nbytes, extra=None):
        gbs = nbytes / (ms * 1e-3) / 1e9
        res[name] = dict(us=round(ms * 1e3, 3), gbs=round(gbs, 1), frac=round(gbs / peak, 4), **(extra or {}))

    # Kimi-Linear recurrent, batch sweep (20 calls per graph on disjoint slot sets)
    for B in (1, 8, 32, 128, 512):
        n_sets = max(1, min(20, 1023 // B))
        d = recurrent_device_case(B, 32, 1024, seed=B, n_sets=n_sets)
        out = torch.empty(B, 32, D, dtype=torch.bfloat16, device="cuda")
        calls = [(lambda i=i: run_recurrent(d, i, out)) for i in range(n_sets if B < 512 else 2)]
        rec(f"recurrent_h32_f32_b{B}", time_graph(calls, 10, flush), bytes_t1(B, 0, 32, 4))
        del d
    # packed Kimi K3 (bf16 state, 10% padding rows), B sweep
    for B in (1, 8, 32, 128, 512):
        nn = int(math.floor(0.1 * B))
        n_sets = max(1, min(20, 2047 // B))
        g = torch.Generator().manual_seed(B)
        c = synth.packed_case(B, num_slots=2, seed=B, null_frac=0.0)
        c["state_indices"] = torch.ones(B, dtype=torch.int32)
        dd = {k: v.cuda() for k, v in c.items() if k != "state"}
        perm = (torch.randperm(2047, generator=g) + 1).to(torch.int32)
        sets = [synth.with_nulls(g, perm[i * B:(i + 1) * B].clone(), nn).cuda() for i in range(n_sets)]
        gen = torch.Generator(device="cuda").manual_seed(B)
        state = torch.empty(2048, 12, D, D, dtype=torch.float32, device="cuda").normal_(0, 0.1, generator=gen)
        state = state.to(torch.bfloat16)
        out = torch.empty(B, 1, 12, D, dtype=torch.bfloat16, device="cuda")

        def pk(i, dd=dd, sets=sets, state=state, out=out):
            binding.kda_packed_decode(dd["mixed_qkv"], dd["raw_gate"], dd["raw_beta"], dd["A_log"], dd["dt_bias"],
                                      sets[i], state, out=out)
        calls = [(lambda i=i: pk(i)) for i in range(n_sets)]
        rec(f"packed_k3_bf16_b{B}", time_graph(calls, 10, flush), bytes_t1(B - nn, nn, 12, 2))
        del state
    # fused conv + KDA + gated RMSNorm, fp32 state, 10% null rows
    for H, rows in ((8, 256), (32, 256), (96, 256), (32, 32)):
        c = synth.fused_case(H, rows, seed=H, num_slots=2 * rows + 1)
        nn = int((c["state_indices"] <= 0).sum())
        dd = {k: v.cuda() for k, v in c.items() if k != "conv_state"}
        dd["conv_state"] = c["conv_state"].permute(0, 2, 1).contiguous().cuda().permute(0, 2, 1)
        out = torch.empty(1, rows, H, D, dtype=torch.bfloat16, device="cuda")

        def fz(dd=dd, out=out):
            binding.kda_fused_decode(dd["x"], dd["conv_weight"], dd["conv_state"], dd["raw_gate"], dd["raw_beta"],
                                     dd["A_log"], dd["dt_bias"], dd["state_indices"], dd["state"],
                                     dd["output_gate"], dd["norm_weight"], out=out)
        rec(f"fused_h{H}_rows{rows}_f32", time_graph([fz], 10, flush), bytes_fused(rows - nn, nn, H, 4))
        del dd
    # speculative ragged rows, H=16, fp32 pool [4N]
    for N, T in ((128, 2), (128, 6), (16, 6)):
        c = synth.spec_case(N, T, seed=N + T)
        dd = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in c.items()}
        out = torch.empty(c["q"].shape, dtype=torch.bfloat16, device="cuda")
        lens = c["lengths"]
        live_rows = int((lens > 0).sum())

        def sp(dd=dd, out=out, T=T):
            binding.kda_spec_decode(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["cu_seqlens"],
                                    dd["state_indices"], dd["state"], T, out=out)
        R = c["q"].shape[0]
        rec(f"spec_h16_n{N}_t{T}_f32", time_graph([sp], 10, flush),
            bytes_spec(R, live_rows, N, R, 16, 4), {"tokens": R})
        del dd
    return res


# ---- CPU oracle -------------------------------------------------------------------------

def oracle_sample_rate(budget_s, H=32, B=512):
    """The float64 oracle on a bounded sample of the headline workload: (GB/s, rows, seconds)."""
    from oracle import kda_oracle as ko
    case = synth.recurrent_case(8, H, 9, seed=0)
    f = synth.to_f64
    args = [f(case[k]) for k in ("q", "k", "v", "raw_gate", "raw_beta", "A_log", "dt_bias")]
    idx = case["state_indices"].numpy()
    pool = f(case["state"])
    rows = 0
    t0 = time.perf_counter()
    while True:
        ko.recurrent_decode(*args, idx, pool)
        rows += 8
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    gbs = bytes_t1(rows, 0, H, 4) / el / 1e9
    return gbs, rows, el


def run_reference(args, rank, world):
    if rank != 0:
        return
    H, B = HEADLINE["H"], HEADLINE["B"]
    per_step = []
    rows_total = 0
    for i in range(args.warmup + args.steps):
        gbs, rows, el = oracle_sample_rate(1.0, H, B)
        if i >= args.warmup:
            per_step.append((gbs, el))
            rows_total += rows
    gbs = statistics.median(g for g, _ in per_step)
    us_call = bytes_t1(B, 0, H, 4) / (gbs * 1e9) * 1e6
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_call / 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(HEADLINE, sample="8 rows x 32 heads per oracle call, repeated for ~1 s per step",
                       note="float64 numpy oracle on the host cores, one thread"),
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": f"{rows_total} rows x 32 heads over {args.steps} steps"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---- main -------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-paths", action="store_true", help="skip the per-path / per-batch measurements")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU baseline budget")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    def barrier():
        if dist is not None:
            dist.barrier()

    from linear_attention_decode_02_gb300 import build
    if rank == 0:
        build.build()
    barrier()
    binding.library()

    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else FALLBACK_HBM_GBS
    peak_src = "measured" if peaks and peaks.get("hbm_gbs") else "fallback"

    ms, nbytes, clocks, d, out = headline(args, rank, world, barrier, peaks)
    t = torch.tensor([ms], dtype=torch.float64, device="cuda")
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    ms_max = float(t.item())
    value = world * nbytes / (ms_max * 1e-3) / 1e9
    achieved = nbytes / (ms * 1e-3) / 1e9

    e2e_ms, h2d, d2h = e2e_recurrent(d, max(20, args.steps // 4), 3, barrier)
    t = torch.tensor([e2e_ms], dtype=torch.float64, device="cuda")
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    e2e_value = world * nbytes / (float(t.item()) * 1e-3) / 1e9
    del d, out
    torch.cuda.empty_cache()

    paths = None
    if not args.no_paths and rank == 0:
        flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
        paths = path_measurements(flush, peak)
        del flush

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        gbs, rows, el = oracle_sample_rate(args.cpu_seconds)
        cpu = {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
               "sample": f"{rows} rows x 32 heads of the headline workload in {el:.1f} s, float64 numpy, one thread"}

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "us_per_call": round(ms_max * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": dict(HEADLINE, bytes_per_call=nbytes,
                           l2="inputs larger than L2: 1.07 GB of state per step, two disjoint slot sets alternate",
                           parallelism=f"replicas x{world}"),
            "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": ncu_traffic("recurrent_h32_f32_b512"),
                         "peak_source": f"{peak_src} copy bandwidth (burst)"},
            "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h},
            "clocks": clocks,
            "cpu_baseline": cpu,
            "paths": paths,
            "kernel_source_hash": kernel_source_hash(),
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
