"""Benchmark of the KDA decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload recurrent|packed|fused|spec] [--batch B] [--heads H]
                    [--slots S] [--t-max T] [--no-paths] [--no-e2e] [--cpu-seconds X]

Default (headline) workload: Kimi-Linear equal-head T=1 recurrent decode,
H=32, K=V=128, float32 state pool [1024, 32, 128, 128], B=512 rows on
distinct slots, bf16 activations, softplus gate.  A step is one
kda_recurrent_decode call; two random slot sets alternate between steps and
every step moves 1.07 GB of state, far more than the 129 MB L2.

Metric: achieved HBM GB/s of the algorithmic bytes (live state read + write
plus the activations and parameters read and the output written) per call;
ms_per_step is the time per call.  The line also carries the same metric end
to end (pinned host inputs copied in and the output copied out each step),
the roofline of the kernel against the measured copy bandwidth, the SM clocks
seen during the timed region, per-path / per-batch CUDA-graph measurements of
the decode entry points (L2 flushed between replays), and the float64 oracle
timed on the host cores.

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
import re
import statistics
import subprocess
import sys
import threading
import time

os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")
os.environ.setdefault("OMP_NUM_THREADS", "1")
os.environ.setdefault("MKL_NUM_THREADS", "1")

import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_decode_02_gb300 import binding, synth  # noqa: E402

D = 128
METRIC = "KDA decode µs/call and achieved HBM GB/s (state R+W) vs GB300 peak, 1 GPU"
FALLBACK_HBM_GBS = 6800.0
L2_BYTES = 129 * 1024 * 1024


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


def bytes_packed_fused(seq_lens, cols, H, state_esize, R):
    """Per live sequence and head: the state and conv cache read once, and
    written once per checkpoint (min(len, cols) of them); per token: x, raw
    gate, beta, output gate and out; padding rows: zero out; params once."""
    conv = 3 * 3 * D * 2
    unit = D * D * state_esize + conv
    live_tokens = sum(seq_lens)
    per_tok = 3 * D * 2 + D * 2 + 2 + D * 2 + D * 2
    ckpts = sum(min(L, cols) for L in seq_lens if L > 0)
    live = sum(1 for L in seq_lens if L > 0)
    params = 3 * 4 * H * D * 4 + H * 4 + H * D * 4 + D * 4
    n = len(seq_lens)
    meta = (n + 1) * 4 + n * 4 + n * cols * 4
    return (live + ckpts) * H * unit + live_tokens * H * per_tok + (R - live_tokens) * H * D * 2 + params + meta


# ---- workloads ---------------------------------------------------------------------

def _device_pool(num_slots, H, dtype, seed):
    gen = torch.Generator(device="cuda").manual_seed(seed)
    pool = torch.empty(num_slots, H, D, D, dtype=torch.float32, device="cuda").normal_(0.0, 0.1, generator=gen)
    return pool if dtype == torch.float32 else pool.to(dtype)


def _slot_sets(n_sets, count, num_slots, null_count, seed, null_values=(-1,)):
    g = torch.Generator().manual_seed(seed + 7)
    sets = []
    for _ in range(n_sets):
        s = synth.with_nulls(g, synth.distinct_slots(g, count, num_slots), null_count, null_values)
        sets.append(s)
    return sets


SPLIT_SOURCE = {0: "kda_t1.cu", 1: "kda_t1.cu", 2: "kda_fused.cu", 3: "kda_spec.cu"}


def kernel_source(op, units, state_dtype, t_max=1):
    """Translation unit of the kernel the library's dispatch picks for this call shape."""
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    code = 0 if state_dtype == torch.float32 else 1
    sched = binding.kda_plan_schedule(op, units, code, t_max, sms)
    if sched == binding.SCHED_STREAM:
        return "kda_stream.cu"
    if sched == binding.SCHED_MMA:
        return "kda_spec_mma.cu"
    return SPLIT_SOURCE[op]


class Workload:
    """One decode path at one size: device inputs, a call per step, its byte model."""

    name = ""

    def call(self, idx):
        raise NotImplementedError

    def step(self, i):
        self.call(self.sets[i % len(self.sets)])


class Recurrent(Workload):
    def __init__(self, B=512, H=32, slots=1024, state_dtype=torch.float32, n_sets=2, null_count=0, seed=0,
                 lower_bound=None):
        self.name = f"recurrent_h{H}_{'f32' if state_dtype == torch.float32 else 'bf16'}_b{B}"
        c = synth.recurrent_case(B, H, slots, seed=seed, make_state=False)
        self.d = {k: v.cuda() for k, v in c.items() if k not in ("state", "state_indices")}
        self.d["state"] = _device_pool(slots, H, state_dtype, seed)
        self.sets = [s.cuda() for s in _slot_sets(n_sets, B, slots, null_count, seed)]
        self.out = torch.empty(B, H, D, dtype=torch.bfloat16, device="cuda")
        self.lower_bound = lower_bound
        esz = 4 if state_dtype == torch.float32 else 2
        self.nbytes = bytes_t1(B - null_count, null_count, H, esz)
        self.config = dict(workload="kimi_linear_t1_recurrent", H=H, B=B, num_slots=slots,
                           state="float32" if esz == 4 else "bfloat16", activations="bfloat16",
                           gate="softplus" if lower_bound is None else f"lower_bound {lower_bound}")
        self.e2e_keys = ("q", "k", "v", "raw_gate", "raw_beta")
        self.source = kernel_source(0, B * H, state_dtype)

    def call(self, idx):
        d = self.d
        binding.kda_recurrent_decode(d["q"], d["k"], d["v"], d["raw_gate"], d["raw_beta"], d["A_log"], d["dt_bias"],
                                     idx, d["state"], out=self.out, lower_bound=self.lower_bound)


class Packed(Workload):
    def __init__(self, B=512, slots=2048, n_sets=2, null_frac=0.1, seed=0):
        self.name = f"packed_k3_bf16_b{B}"
        nn = int(math.floor(null_frac * B))
        c = synth.packed_case(B, num_slots=slots, seed=seed, null_frac=0.0, make_state=False)
        self.d = {k: v.cuda() for k, v in c.items() if k not in ("state", "state_indices")}
        self.d["state"] = _device_pool(slots, 12, torch.bfloat16, seed)
        self.sets = [s.cuda() for s in _slot_sets(n_sets, B, slots, nn, seed)]
        self.out = torch.empty(B, 1, 12, D, dtype=torch.bfloat16, device="cuda")
        self.nbytes = bytes_t1(B - nn, nn, 12, 2)
        self.config = dict(workload="packed_kimi_k3_t1", H=12, B=B, num_slots=slots, state="bfloat16",
                           padding_rows=nn, gate="lower_bound -5")
        self.e2e_keys = ("mixed_qkv", "raw_gate", "raw_beta")
        self.source = kernel_source(1, B * 12, torch.bfloat16)

    def call(self, idx):
        d = self.d
        binding.kda_packed_decode(d["mixed_qkv"], d["raw_gate"], d["raw_beta"], d["A_log"], d["dt_bias"], idx,
                                  d["state"], out=self.out)


class Fused(Workload):
    def __init__(self, H=32, rows=256, slots=None, state_dtype=torch.float32, n_sets=2, null_frac=0.1, seed=0,
                 lower_bound=-5.0):
        slots = slots or 2 * rows + 1
        self.name = f"fused_h{H}_rows{rows}_{'f32' if state_dtype == torch.float32 else 'bf16'}"
        nn = int(math.floor(null_frac * rows))
        c = synth.fused_case(H, rows, seed=seed, num_slots=slots, null_frac=0.0, make_state=False)
        self.d = {k: v.cuda() for k, v in c.items() if k not in ("state", "state_indices", "conv_state")}
        self.d["state"] = _device_pool(slots, H, state_dtype, seed)
        gen = torch.Generator(device="cuda").manual_seed(seed + 1)
        phys = torch.empty(slots, 3, 3 * H * D, dtype=torch.float32, device="cuda").normal_(generator=gen)
        self.d["conv_state"] = phys.to(torch.bfloat16).permute(0, 2, 1)
        self.sets = [s.cuda() for s in _slot_sets(n_sets, rows, slots, nn, seed, (0, -1))]
        self.out = torch.empty(1, rows, H, D, dtype=torch.bfloat16, device="cuda")
        self.lower_bound = lower_bound
        self.nbytes = bytes_fused(rows - nn, nn, H, 4 if state_dtype == torch.float32 else 2)
        self.config = dict(workload="fused_conv_kda_gated_rmsnorm_t1", H=H, rows=rows, num_slots=slots,
                           state="float32" if state_dtype == torch.float32 else "bfloat16", null_rows=nn,
                           gate=f"lower_bound {lower_bound}" if lower_bound is not None else "softplus")
        self.e2e_keys = ("x", "raw_gate", "raw_beta", "output_gate")
        self.source = kernel_source(2, rows * H, state_dtype)

    def call(self, idx):
        d = self.d
        binding.kda_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"], d["raw_beta"], d["A_log"],
                                 d["dt_bias"], idx, d["state"], d["output_gate"], d["norm_weight"],
                                 lower_bound=self.lower_bound, out=self.out)


class Spec(Workload):
    """Ragged speculative rows (lengths 1..t_max, some empty), or with
    `fixed` every row exactly t_max tokens long."""

    def __init__(self, N=128, t_max=6, H=16, slots=None, state_dtype=torch.float32, n_sets=2, seed=0, fixed=False):
        slots = slots or 4 * N
        self.name = (f"spec_h{H}_n{N}_t{t_max}{'_fixed' if fixed else ''}_"
                     f"{'f32' if state_dtype == torch.float32 else 'bf16'}")
        c = synth.spec_case(N, t_max, seed=seed, H=H, num_slots=slots, make_state=False,
                            lengths=[t_max] * N if fixed else None)
        self.t_max = t_max
        self.d = {k: v.cuda() for k, v in c.items() if isinstance(v, torch.Tensor) and k not in ("state",
                                                                                                   "state_indices")}
        self.d["state"] = _device_pool(slots, H, state_dtype, seed)
        self.sets = [s.cuda() for s in _slot_sets(n_sets, N, slots, 0, seed)]
        R = c["q"].shape[0]
        self.out = torch.empty(R, H, D, dtype=torch.bfloat16, device="cuda")
        lens = c["lengths"]
        live_rows = int((lens > 0).sum())
        self.nbytes = bytes_spec(R, live_rows, N, R, H, 4 if state_dtype == torch.float32 else 2)
        self.config = dict(workload="packed_speculative_" + ("fixed" if fixed else "ragged"), H=H, rows=N,
                           t_max=t_max, tokens=R,
                           empty_rows=N - live_rows, num_slots=slots,
                           state="float32" if state_dtype == torch.float32 else "bfloat16",
                           gates="precomputed fp32 log decay in [-5, 0]")
        self.source = kernel_source(3, N * H, state_dtype, t_max)
        self.e2e_keys = ("q", "k", "v", "g", "beta", "cu_seqlens")

    def call(self, idx):
        d = self.d
        binding.kda_spec_decode(d["q"], d["k"], d["v"], d["g"], d["beta"], d["cu_seqlens"], idx, d["state"],
                                self.t_max, out=self.out)


class PackedFused(Workload):
    """Packed fused speculative decode: N sequences of T tokens, one accepted
    token (start column 0), a checkpoint after every token."""

    def __init__(self, N=128, T=5, H=12, state_dtype=torch.float32, n_sets=2, seed=0):
        cols = T
        slots = n_sets * N * cols + 1
        tag = "f32" if state_dtype == torch.float32 else "bf16"
        self.name = f"packed_fused_h{H}_n{N}_t{T}_{tag}"
        c = synth.packed_fused_case(N, T, H=H, seed=seed, lengths=[T] * N, accepted=1, num_slots=slots,
                                    make_state=False)
        self.d = {k: v.cuda() for k, v in c.items()
                  if isinstance(v, torch.Tensor) and k not in ("state_indices", "lengths")}
        self.d["state"] = _device_pool(slots, H, state_dtype, seed)
        gen = torch.Generator(device="cuda").manual_seed(seed + 1)
        phys = torch.empty(slots, 3, 3 * H * D, dtype=torch.float32, device="cuda").normal_(generator=gen)
        self.d["conv_state"] = phys.to(torch.bfloat16).permute(0, 2, 1)
        g = torch.Generator().manual_seed(seed + 7)
        perm = (torch.randperm(slots - 1, generator=g) + 1).to(torch.int32)
        self.sets = [perm[i * N * cols:(i + 1) * N * cols].view(N, cols).cuda() for i in range(n_sets)]
        R = N * T
        self.out = torch.empty(R, H, D, dtype=torch.bfloat16, device="cuda")
        self.nbytes = bytes_packed_fused([T] * N, cols, H, 4 if state_dtype == torch.float32 else 2, R)
        self.config = dict(workload="packed_fused_spec_checkpoints", H=H, sequences=N, tokens_per_sequence=T,
                           num_accepted_tokens=1, checkpoint_columns=cols, num_slots=slots, state=
                           "float32" if state_dtype == torch.float32 else "bfloat16", gate="lower_bound -5")
        self.e2e_keys = ("x", "raw_gate", "raw_beta", "output_gate")
        self.source = "kda_packed_fused.cu"

    def call(self, idx):
        d = self.d
        binding.kda_packed_fused_decode(d["x"], d["conv_weight"], d["conv_state"], d["raw_gate"], d["raw_beta"],
                                        d["A_log"], d["dt_bias"], idx, d["query_start_loc"],
                                        d["num_accepted_tokens"], d["state"], d["output_gate"], d["norm_weight"],
                                        out=self.out)


def make_workload(args, seed):
    state_dtype = torch.bfloat16 if args.bf16_state else torch.float32
    if args.workload == "recurrent":
        return Recurrent(B=args.batch or 512, H=args.heads or 32, slots=args.slots or 1024, state_dtype=state_dtype,
                         seed=seed)
    if args.workload == "packed":
        return Packed(B=args.batch or 512, slots=args.slots or 2048, seed=seed)
    if args.workload == "fused":
        return Fused(H=args.heads or 32, rows=args.batch or 256, slots=args.slots or None, state_dtype=state_dtype,
                     seed=seed)
    if args.workload == "packed_fused":
        return PackedFused(N=args.batch or 128, T=args.t_max or 5, H=args.heads or 12, state_dtype=state_dtype,
                           seed=seed)
    return Spec(N=args.batch or 128, t_max=args.t_max or 6, H=args.heads or 16, slots=args.slots, seed=seed,
                state_dtype=state_dtype, fixed=args.fixed)


# ---- environment -------------------------------------------------------------------

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f)
    except (OSError, ValueError):
        return None


CSRC = os.path.join(ROOT, "linear_attention_decode_02_gb300", "csrc")


def source_closure(name):
    """`name` and every csrc file it includes, transitively (quoted includes only)."""
    seen, todo = [], [name]
    while todo:
        f = todo.pop()
        if not f or f in seen or not os.path.isfile(os.path.join(CSRC, f)):
            continue
        seen.append(f)
        with open(os.path.join(CSRC, f)) as fh:
            todo += re.findall(r'^#include\s+"([^"/]+)"', fh.read(), re.M)
    return sorted(seen)


_COMMENT = re.compile(r'//[^\n]*|/\*.*?\*/|"(?:\\.|[^"\\])*"', re.S)


def code_only(text):
    """C++ source without its comments and with whitespace runs collapsed
    (string literals kept), so that editing a comment leaves the hash alone."""
    text = _COMMENT.sub(lambda m: m.group(0) if m.group(0).startswith('"') else " ", text)
    return " ".join(text.split())


def kernel_source_hash(name="kda_t1.cu"):
    """Hash of one kernel translation unit and the csrc headers it includes,
    comments and whitespace ignored."""
    h = hashlib.sha256()
    for f in source_closure(name):
        with open(os.path.join(CSRC, f)) as fh:
            h.update(f.encode() + b"\0" + code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def ncu_traffic(kind):
    """DRAM bytes per launch from the committed ncu summary, if that kernel's sources are unchanged since."""
    try:
        with open(os.path.join(ROOT, "profiles", "ncu_traffic.json")) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    entry = rec.get("kernels", {}).get(kind)
    if not entry or entry.get("source_hash") != kernel_source_hash(entry.get("source", "")):
        return None
    return entry.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi SM clocks and throttle reasons sampled every 100 ms while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

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
        threading.Thread(target=self._read, daemon=True).start()
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
        inside = [p for (t, p) in self.samples if t0 <= t <= t1]
        rows = inside or [p for (_, p) in self.samples]
        if not rows:
            return None

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [v for v in (num(p[0]) for p in rows) if v is not None]
        mx = [v for v in (num(p[1]) for p in rows) if v is not None]
        reasons = sorted({self.REASONS[i] for p in rows for i in range(4) if p[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside)}


class NvmlSampler:
    """SM clock and clock-event reasons polled through NVML (read-only queries)
    every `period` seconds from a thread, so that even a timed region of a few
    milliseconds holds samples.  Same summary as ClockSampler."""

    REASONS = (("hw_slowdown", 0x8), ("hw_thermal_slowdown", 0x40), ("sw_thermal_slowdown", 0x20),
               ("sw_power_cap", 0x4))

    def __init__(self, device_index=0, period=0.002):
        import ctypes
        self.ct = ctypes
        self.samples = []
        self.period = period
        self.stop_ev = threading.Event()
        self.thread = None
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.lib = lib
        self.dev = ctypes.c_void_p()
        uuid = ClockSampler._physical_id(device_index).encode()
        if lib.nvmlDeviceGetHandleByUUID(ctypes.c_char_p(uuid), ctypes.byref(self.dev)) != 0:
            raise OSError("no NVML handle for " + uuid.decode())
        self.reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        mx = ctypes.c_uint()
        self.max_mhz = float(mx.value) if lib.nvmlDeviceGetMaxClockInfo(self.dev, 1, ctypes.byref(mx)) == 0 else None

    def _poll(self):
        ct = self.ct
        clk, rs = ct.c_uint(), ct.c_ulonglong()
        while not self.stop_ev.is_set():
            ok = self.lib.nvmlDeviceGetClockInfo(self.dev, 1, ct.byref(clk)) == 0
            ok = ok and self.reasons_fn(self.dev, ct.byref(rs)) == 0
            if ok:
                self.samples.append((time.time(), float(clk.value), int(rs.value)))
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._poll, daemon=True)
        self.thread.start()
        time.sleep(0.05)

    def stop(self):
        self.stop_ev.set()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0, t1):
        inside = [x for x in self.samples if t0 <= x[0] <= t1]
        rows = inside or self.samples
        if not rows:
            return None
        reasons = sorted({n for (_, _, r) in rows for n, bit in self.REASONS if r & bit})
        return {"sm_mhz": statistics.median(c for (_, c, _) in rows), "sm_max_mhz": self.max_mhz,
                "reasons": reasons, "samples": len(rows), "samples_in_timed_region": len(inside),
                "source": "nvml, every %.0f ms" % (self.period * 1e3)}


def clock_sampler(device_index):
    """NVML poller when the library loads, else nvidia-smi at 100 ms."""
    try:
        return NvmlSampler(device_index)
    except (OSError, AttributeError):
        return ClockSampler(device_index)


# ---- rank aggregation ------------------------------------------------------------------

def reduce_max(x, dist=None, device="cpu"):
    """Max of a per-rank float over the process group (identity without one)."""
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    if dist is not None:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_gbs(bytes_per_rank, world, ms_max):
    """Whole-job GB/s: every rank's bytes over the slowest rank's time per step."""
    return world * bytes_per_rank / (ms_max * 1e-3) / 1e9


# ---- timing helpers ------------------------------------------------------------------

def time_direct(fn, steps, warmup, barrier):
    """Average ms per step over `steps` back-to-back steps on the current stream."""
    stream = torch.cuda.current_stream()
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


class L2Flush:
    """Cold-L2 preparation before a timed replay: write a buffer larger than
    L2, then read a second one, so the written lines are back in DRAM before
    the timed region starts (otherwise the kernel pays the flush's own
    write-backs) and L2 holds none of the kernel's data."""

    def __init__(self):
        self.w = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")
        self.r = torch.zeros(2 * L2_BYTES // 4, dtype=torch.float32, device="cuda")

    def __call__(self, value):
        self.w.fill_(value)
        return self.r.sum()


def time_graph(wl, n_calls, reps, flush):
    """Per-call ms of a CUDA graph of `n_calls` launches on rotating slot sets, L2 flushed before each replay."""
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for i in range(n_calls):
            wl.step(i)
    torch.cuda.current_stream().wait_stream(s)
    with torch.cuda.graph(g):
        for i in range(n_calls):
            wl.step(i)
    times = []
    for r in range(reps + 2):
        flush(float(r))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if r >= 2:
            times.append(e0.elapsed_time(e1) / n_calls)
    return statistics.median(times)


def _staging(wl):
    """Pinned host staging of a step's inputs: each input and the slot indices
    at 256-byte aligned offsets of one buffer (one buffer per slot set), and a
    function giving the typed views of such a buffer."""
    keys = list(wl.e2e_keys)
    fields, off = [], 0
    for k in keys + ["__idx__"]:
        t = wl.sets[0] if k == "__idx__" else wl.d[k]
        nbytes = t.numel() * t.element_size()
        fields.append((k, off, nbytes, t.dtype, tuple(t.shape)))
        off += (nbytes + 255) // 256 * 256
    total = off

    def views(buf):
        return {k: buf[o:o + n].view(dt).view(shape) for k, o, n, dt, shape in fields}

    host = []
    for idx in wl.sets:
        hb = torch.empty(total, dtype=torch.uint8).pin_memory()
        hv = views(hb)
        for k in keys:
            hv[k].copy_(wl.d[k].cpu())
        hv["__idx__"].copy_(idx.cpu())
        host.append(hb)
    return keys, fields, total, views, host


def e2e(wl, steps, warmup, barrier):
    """The same call end to end: every step copies its activations and slot
    indices from pinned host memory to the device and its output back.

    The steps are pipelined the way a serving loop would run them: a step's
    inputs sit in one pinned staging buffer and cross in one host-to-device
    copy (the entry point then takes views into the device copy); inputs and
    outputs are double-buffered on the device, host-to-device copies run on
    one side stream and device-to-host copies on another, and events keep
    step i's copies ordered with its kernel; the state pool is updated in
    place on the compute stream, so kernels stay in order.
    """
    keys, fields, total, views, host = _staging(wl)
    nb = 2
    dev = [torch.empty(total, dtype=torch.uint8, device="cuda") for _ in range(nb)]
    dv = [views(d) for d in dev]
    outs = [torch.empty_like(wl.out) for _ in range(nb)]
    out_h = [torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory() for _ in range(nb)]
    comp = torch.cuda.current_stream()
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in range(nb)]
    ev_k = [torch.cuda.Event() for _ in range(nb)]
    ev_out = [torch.cuda.Event() for _ in range(nb)]
    base = dict(wl.d)
    dmaps = [{**base, **{k: dv[b][k] for k in keys}} for b in range(nb)]

    def step(i):
        b = i % nb
        s_in.wait_event(ev_k[b])  # the kernel two steps back has read this input buffer
        with torch.cuda.stream(s_in):
            dev[b].copy_(host[i % len(host)], non_blocking=True)
        ev_in[b].record(s_in)
        comp.wait_event(ev_in[b])
        comp.wait_event(ev_out[b])  # the output buffer has been copied out
        wl.d = dmaps[b]
        wl.out = outs[b]
        wl.call(dv[b]["__idx__"])
        ev_k[b].record(comp)
        s_out.wait_event(ev_k[b])
        with torch.cuda.stream(s_out):
            out_h[b].copy_(outs[b], non_blocking=True)
        ev_out[b].record(s_out)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    for i in range(warmup, warmup + steps):
        step(i)
    for b in range(nb):
        comp.wait_event(ev_out[b])  # the timed region ends with the last outputs on the host
    e1.record(comp)
    torch.cuda.synchronize()
    barrier()
    wl.d = base
    h2d = sum(n for _, _, n, _, _ in fields)
    d2h = out_h[0].numel() * out_h[0].element_size()
    return e0.elapsed_time(e1) / steps, h2d, d2h
def path_measurements(flush, peak):
    """CUDA-graph timings of the decode entry points over their configured sizes."""
    res = {}

    def run(wl, n_sets, schedule=None):
        if schedule is not None:
            binding.kda_set_schedule_override(schedule)
        try:
            ms = time_graph(wl, n_sets, 10, flush)
        finally:
            binding.kda_set_schedule_override(binding.SCHED_AUTO)
        gbs = wl.nbytes / (ms * 1e-3) / 1e9
        name = wl.name + ("_mma" if schedule == binding.SCHED_MMA else "")
        res[name] = dict(us=round(ms * 1e3, 3), gbs=round(gbs, 1), frac=round(gbs / peak, 4))

    for B in (1, 8, 32, 128, 512):
        n = max(1, min(16, 1023 // B))
        run(Recurrent(B=B, H=32, slots=1024, n_sets=n, seed=B), n)
    for B in (1, 8, 16, 31, 32, 64, 128, 256, 512):
        n = max(1, min(16, 2047 // B))
        run(Packed(B=B, slots=2048, n_sets=n, seed=B), n)
    # Small batches replay up to 16 calls per graph on distinct slot sets, as
    # the T=1 paths above do, so that the graph's own launch is spread over
    # the calls it holds.
    for H, rows in ((8, 1), (8, 32), (8, 256), (12, 256), (32, 32), (32, 256), (96, 256)):
        n = min(16, max(2, 1024 // rows))
        run(Fused(H=H, rows=rows, slots=n * rows + 1, n_sets=n, seed=H + rows), n)
    for N, T in ((1, 6), (16, 6), (128, 2), (128, 4), (128, 6)):
        n = 16 if N <= 16 else 2
        run(Spec(N=N, t_max=T, H=16, slots=max(4 * N, n * N + 1), n_sets=n, seed=N + T), n)
    # bf16 state: the per-token kernel (the policy's choice) and the tensor-core
    # chunked form, on ragged rows and on rows of exactly T tokens
    for N, T, fixed in ((128, 6, False), (128, 6, True), (128, 8, True), (128, 16, True)):
        for sched in (None, binding.SCHED_MMA):
            run(Spec(N=N, t_max=T, H=16, state_dtype=torch.bfloat16, n_sets=2, seed=N + T, fixed=fixed), 2, sched)
    for H, N in ((12, 1), (12, 8), (12, 32), (12, 128), (24, 8), (24, 128)):
        n = 16 if N <= 8 else 2
        for dt in (torch.float32, torch.bfloat16):
            run(PackedFused(N=N, T=5, H=H, state_dtype=dt, n_sets=n, seed=H + N), n)
    torch.cuda.empty_cache()
    return res


def e2e_serial(wl, steps, warmup):
    """End to end on one stream, one step after another, driven from Python
    (no CUDA graph): the step's inputs in one copy from pinned host memory,
    the entry point (descriptor marshalling, validation, launch), the output
    copied back to pinned memory.  Returns ms per step and the bytes each way."""
    keys, fields, total, views, host = _staging(wl)
    dev = torch.empty(total, dtype=torch.uint8, device="cuda")
    dv = views(dev)
    base = dict(wl.d)
    wl.d = {**base, **{k: dv[k] for k in keys}}
    out_h = torch.empty(wl.out.shape, dtype=wl.out.dtype).pin_memory()

    def step(i):
        dev.copy_(host[i % len(host)], non_blocking=True)
        wl.call(dv["__idx__"])
        out_h.copy_(wl.out, non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(warmup, warmup + steps):
        step(i)
    e1.record()
    torch.cuda.synchronize()
    wl.d = base
    return e0.elapsed_time(e1) / steps, sum(n for _, _, n, _, _ in fields), out_h.numel() * out_h.element_size()


def small_e2e():
    """End to end at small batches (`e2e_serial`).  At these sizes the host
    work, not the kernel, sets the pace; `paths` times the same kernels from
    a CUDA graph."""
    res = {}
    makers = (lambda: Recurrent(B=1, H=32, slots=64, n_sets=2, seed=1),
              lambda: Recurrent(B=8, H=32, slots=64, n_sets=2, seed=8),
              lambda: Packed(B=1, slots=64, n_sets=2, seed=1),
              lambda: Fused(H=8, rows=1, n_sets=2, seed=9),
              lambda: Spec(N=1, t_max=6, H=16, n_sets=2, seed=7),
              lambda: PackedFused(N=1, T=5, H=12, state_dtype=torch.bfloat16, n_sets=2, seed=13))
    for make in makers:
        wl = make()
        ms, h2d, d2h = e2e_serial(wl, 300, 30)
        res[wl.name] = {"us": round(ms * 1e3, 2), "h2d_bytes": h2d, "d2h_bytes": d2h}
        del wl
    torch.cuda.empty_cache()
    return res


# ---- CPU oracle -------------------------------------------------------------------------

THREAD_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _oracle_worker(job):
    """One host process running the float64 oracle on its own sample of the
    headline workload for `budget_s` seconds: (rows, seconds)."""
    budget_s, H, seed = job
    from oracle import kda_oracle as ko
    case = synth.recurrent_case(8, H, 9, seed=seed)
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
    return rows, el


def oracle_rates(budget_s, H=32, workers=0, steps=1):
    """The oracle on the host cores, each process single-threaded (spawned, so
    no GPU context is inherited).  Returns ((GB/s, rows, s) on one core,
    [(GB/s, rows, s) per step on all processes], processes); each step gives
    every process budget_s / 2 seconds."""
    import multiprocessing
    ctx = multiprocessing.get_context("spawn")
    n = workers or os.cpu_count() or 1
    saved = {k: os.environ.get(k) for k in THREAD_VARS}
    os.environ.update({k: "1" for k in THREAD_VARS})
    try:
        with ctx.Pool(1) as p:
            r1, e1 = p.apply(_oracle_worker, ((budget_s / 2, H, 0),))
        per_step = []
        with ctx.Pool(n) as p:
            for step in range(steps):
                res = p.map(_oracle_worker, [(budget_s / 2, H, step * n + i) for i in range(n)])
                rn, en = sum(r for r, _ in res), max(e for _, e in res)
                per_step.append((bytes_t1(rn, 0, H, 4) / en / 1e9, rn, en))
    finally:
        for k, v in saved.items():
            if v is None:
                os.environ.pop(k, None)
            else:
                os.environ[k] = v
    return (bytes_t1(r1, 0, H, 4) / e1 / 1e9, r1, e1), per_step, n


def run_reference(args, rank, world):
    """The float64 oracle as the reference arm, timed on the host cores (rank 0 only).
    Each step is a bounded sample, sized so the whole run takes about two minutes."""
    if rank != 0:
        return
    H, B = 32, 512
    budget = max(0.05, min(1.0, 120.0 / max(1, args.warmup + args.steps)))
    (g1, _, _), per_step, procs = oracle_rates(budget, H, steps=args.warmup + args.steps)
    timed = per_step[args.warmup:]
    gbs = statistics.median(g for g, _, _ in timed)
    rows_total = sum(r for _, r, _ in timed)
    us_call = bytes_t1(B, 0, H, 4) / (gbs * 1e9) * 1e6
    cfg = dict(workload="kimi_linear_t1_recurrent", H=H, B=B, num_slots=1024, state="float32",
               activations="bfloat16", gate="softplus",
               sample=f"8 rows x 32 heads per oracle call, repeated for {budget / 2:.3f} s per step in each of "
                      f"{procs} single-threaded processes")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(us_call / 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg,
        "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": procs, "kind": "oracle",
                         "value_one_core": round(g1, 4),
                         "sample": f"{rows_total} rows x 32 heads over {args.steps} steps, float64 numpy"},
        "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


# ---- main -------------------------------------------------------------------------------

def main():
    ap = argparse.ArgumentParser(description="KDA decode benchmark (GB300)")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=("recurrent", "packed", "fused", "spec", "packed_fused"),
                    default="recurrent")
    ap.add_argument("--bf16-state", action="store_true", help="recurrent, fused, packed_fused, spec: bfloat16 state pool (packed always has one)")
    ap.add_argument("--fixed", action="store_true", help="spec: every row exactly --t-max tokens")
    ap.add_argument("--schedule", choices=("auto", "split", "stream", "mma"), default="auto",
                    help="force a kernel schedule (mma: the tensor-core speculative form, bf16 state)")
    ap.add_argument("--batch", type=int, default=0, help="rows (B / rows / N); 0 = the workload's default")
    ap.add_argument("--heads", type=int, default=0)
    ap.add_argument("--slots", type=int, default=0)
    ap.add_argument("--t-max", type=int, default=0)
    ap.add_argument("--no-paths", action="store_true", help="skip the per-path / per-batch measurements")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end measurement")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU baseline budget (0 = skip)")
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

    def max_over_ranks(x):
        return reduce_max(x, dist, "cuda")

    from linear_attention_decode_02_gb300 import build
    if rank == 0:
        build.build()
    barrier()
    binding.library()

    peaks = measured_peaks()
    peak = float(peaks["hbm_gbs"]) if peaks and peaks.get("hbm_gbs") else FALLBACK_HBM_GBS
    peak_src = "measured" if peaks and peaks.get("hbm_gbs") else "fallback"

    binding.kda_set_schedule_override({"auto": binding.SCHED_AUTO, "split": binding.SCHED_SPLIT,
                                       "stream": binding.SCHED_STREAM, "mma": binding.SCHED_MMA}[args.schedule])
    wl = make_workload(args, seed=rank)
    clocks = clock_sampler(torch.cuda.current_device())
    clocks.start()
    ms, (w0, w1) = time_direct(wl.step, args.steps, args.warmup, barrier)
    # Clock window: the same loop repeated for at least half a second, so
    # that the clock record spans many samples as well; its time per step is
    # reported beside the timed one (time x median clock can be compared).
    reps = max(args.steps, int(math.ceil(0.5 / max(ms * 1e-3, 1e-6))))
    ms_win, (v0, v1) = time_direct(wl.step, reps, 0, barrier)
    clocks.stop()
    clock_rec = clocks.summary(w0, w1)
    if clock_rec is not None:
        win = clocks.summary(v0, v1)
        clock_rec["window"] = {"steps": reps, "ms_per_step": round(ms_win, 5),
                               "sm_mhz": win and win["sm_mhz"], "samples": win and win["samples_in_timed_region"],
                               "reasons": win and win["reasons"]}
    ms_max = max_over_ranks(ms)
    value = job_gbs(wl.nbytes, world, ms_max)
    achieved = wl.nbytes / (ms * 1e-3) / 1e9

    e2e_obj = None
    if not args.no_e2e:
        e_ms, h2d, d2h = e2e(wl, max(20, args.steps // 4), 3, barrier)
        e_max = max_over_ranks(e_ms)
        e2e_obj = {"value": round(job_gbs(wl.nbytes, world, e_max), 1), "unit": "GB/s",
                   "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(e_max, 5)}
    name, cfg, nbytes, source = wl.name, dict(wl.config), wl.nbytes, wl.source
    if args.schedule != "auto":
        cfg["schedule"] = args.schedule
        name += "_" + args.schedule
    binding.kda_set_schedule_override(binding.SCHED_AUTO)
    del wl
    torch.cuda.empty_cache()

    paths = small = None
    if not args.no_paths and rank == 0:
        flush = L2Flush()
        paths = path_measurements(flush, peak)
        del flush
        small = small_e2e()

    cpu = None
    if rank == 0 and world == 1 and args.cpu_seconds > 0:
        (g1, r1, e1), ((gn, rn, en),), procs = oracle_rates(args.cpu_seconds)
        cpu = {"value": round(gn, 4), "unit": "GB/s", "cores": procs, "kind": "oracle",
               "value_one_core": round(g1, 4),
               "sample": f"{rn} rows x 32 heads of the headline workload in {en:.1f} s over {procs} "
                         f"single-threaded processes ({r1} rows in {e1:.1f} s on one), float64 numpy"}

    if rank == 0:
        cfg.update(bytes_per_call=nbytes, parallelism=f"replicas x{world}",
                   l2=("inputs larger than L2" if nbytes > L2_BYTES else "state smaller than L2: slot sets rotate")
                   + "; slot sets alternate between steps")
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(ms_max, 5), "us_per_call": round(ms_max * 1e3, 2),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic", "config": cfg, "gpu_launches": args.steps,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": ncu_traffic(name), "kernel": name,
                         "peak_source": f"{peak_src} copy bandwidth (burst)"},
            "e2e": e2e_obj, "clocks": clock_rec, "cpu_baseline": cpu, "paths": paths, "e2e_small": small,
            "kernel_source": source, "kernel_source_hash": kernel_source_hash(source),
        }
        print(json.dumps(line))
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
