"""Thin Python binding of libkda (ctypes): argument marshalling only.

Each function has the name of its C entry point, turns torch tensors into
``kda_tensor`` descriptors, passes the current CUDA stream, and raises
``KdaError`` on any non-OK status.  All arithmetic runs in the library's
CUDA kernels; there is no fallback path: if ``libkda.so`` is missing the
first call raises.
"""

from __future__ import annotations

import contextlib
import ctypes
import math
import os
import threading

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkda.so")
_lock = threading.Lock()
_lib = None

KDA_OK = 0
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED", 3: "KDA_ERR_ALIAS",
                4: "KDA_ERR_CUDA"}
OP_RECURRENT, OP_PACKED, OP_FUSED, OP_SPEC = 0, 1, 2, 3
KDA_F32, KDA_BF16, KDA_I32 = 0, 1, 2
_DTYPES = {torch.float32: KDA_F32, torch.bfloat16: KDA_BF16, torch.int32: KDA_I32}
DEFAULT_SCALE = 1.0 / math.sqrt(128.0)

# Every symbol include/kda.h declares.
EXPORTS = ("kda_recurrent_decode", "kda_packed_decode", "kda_fused_decode", "kda_spec_decode",
           "kda_packed_fused_decode",
           "kda_spec_verify_decode",
           "kda_plan_split", "kda_set_split_override", "kda_plan_schedule", "kda_set_schedule_override",
           "kda_device_error", "kda_selftest_wait_timeout", "kda_status_string", "kda_last_error_message",
           "kda_version")
SCHED_AUTO, SCHED_SPLIT, SCHED_STREAM, SCHED_MMA = 0, 1, 2, 3


class KdaError(RuntimeError):
    """A non-OK status returned by libkda."""

    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class KdaTensor(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 4), ("stride", ctypes.c_int64 * 4)]


def _declare(lib):
    T = ctypes.POINTER(KdaTensor)
    i32, f32, vp = ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    sigs = {
        "kda_recurrent_decode": [T, T, T, T, T, T, T, T, T, T, i32, f32, f32, vp],
        "kda_packed_decode": [T, T, T, T, T, T, T, T, vp],
        "kda_fused_decode": [T, T, T, T, T, T, T, T, T, T, T, i32, f32, f32, T, vp],
        "kda_packed_fused_decode": [T, T, T, T, T, T, T, T, T, T, T, T, T, i32, f32, f32, T, vp],
        "kda_spec_decode": [T, T, T, T, T, i32, T, i32, T, T, T, f32, vp],
        "kda_spec_verify_decode": [T, T, T, T, T, i32, T, i32, T, T, T, T, T, f32, vp],
    }
    for name, args in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.kda_plan_split.argtypes = [i32, ctypes.c_int64, i32, i32, i32]
    lib.kda_plan_split.restype = i32
    lib.kda_set_split_override.argtypes = [i32]
    lib.kda_set_split_override.restype = ctypes.c_int
    lib.kda_plan_schedule.argtypes = [i32, ctypes.c_int64, i32, i32, i32]
    lib.kda_plan_schedule.restype = i32
    lib.kda_set_schedule_override.argtypes = [i32]
    lib.kda_set_schedule_override.restype = ctypes.c_int
    lib.kda_device_error.argtypes = [ctypes.POINTER(ctypes.c_uint32), i32]
    lib.kda_device_error.restype = ctypes.c_int
    lib.kda_selftest_wait_timeout.argtypes = [vp]
    lib.kda_selftest_wait_timeout.restype = ctypes.c_int
    lib.kda_status_string.argtypes = [ctypes.c_int]
    lib.kda_status_string.restype = ctypes.c_char_p
    lib.kda_last_error_message.argtypes = []
    lib.kda_last_error_message.restype = ctypes.c_char_p
    lib.kda_version.argtypes = []
    lib.kda_version.restype = ctypes.c_char_p
    return lib


def library(path=None):
    """Load (once) and return the ctypes handle of libkda.so."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    with _lock:
        if _lib is None:
            p = path or _LIB_PATH
            if not os.path.exists(p):
                raise RuntimeError(f"libkda.so is not built ({p}); run "
                                   "`python -m linear_attention_decode_02_gb300.build`")
            _lib = _declare(ctypes.CDLL(p))
        return _lib


def desc(t):
    """kda_tensor descriptor of a torch tensor (shape and strides in elements)."""
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}")
    if t.dim() < 1 or t.dim() > 4:
        raise ValueError(f"rank {t.dim()} not in 1..4")
    d = KdaTensor()
    d.data = t.data_ptr() if t.numel() > 0 else None
    d.dtype = _DTYPES[t.dtype]
    d.ndim = t.dim()
    for i, (s, st) in enumerate(zip(t.shape, t.stride())):
        d.shape[i] = s
        d.stride[i] = st
    return d


# A descriptor depends only on the tensor's address, dtype, shape and
# strides, and the library only reads it, so the per-call marshalling reuses
# descriptors cached on exactly those (bounded; cleared when full).
_DESC_CACHE = {}
_DESC_CACHE_MAX = 1024


def _ref(t):
    key = (t.data_ptr(), t.dtype, t.shape, t.stride())
    r = _DESC_CACHE.get(key)
    if r is None:
        r = ctypes.byref(desc(t))  # holds the descriptor alive
        if len(_DESC_CACHE) >= _DESC_CACHE_MAX:
            _DESC_CACHE.clear()
        _DESC_CACHE[key] = r
    return r


# The current stream's raw handle without building a torch.cuda.Stream
# object (2.2 -> 0.1 us a call on the Grace host); the public query where
# the raw one is absent.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(t):
    if _raw_stream is not None and t.device.type == "cuda":
        return ctypes.c_void_p(_raw_stream(t.device.index))
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


_SAME_DEVICE = contextlib.nullcontext()


def _on(dev):
    """Device guard for the call, entered only when `dev` is not already current."""
    if dev.type == "cuda" and dev.index == torch.cuda.current_device():
        return _SAME_DEVICE
    return torch.cuda.device(dev)


def _check(lib, status):
    if status != KDA_OK:
        raise KdaError(status, lib.kda_last_error_message().decode())


def kda_recurrent_decode(q, k, v, raw_gate, raw_beta, A_log, dt_bias, state_indices, state,
                         out=None, lower_bound=None, scale=DEFAULT_SCALE):
    """T=1 recurrent decode; updates `state` in place, returns bf16 out [B, H, 128]."""
    lib = library()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    with _on(q.device):
        st = lib.kda_recurrent_decode(_ref(q), _ref(k), _ref(v), _ref(raw_gate), _ref(raw_beta),
                                      _ref(A_log), _ref(dt_bias), _ref(state_indices), _ref(state),
                                      _ref(out), int(lower_bound is not None),
                                      float(lower_bound if lower_bound is not None else 0.0),
                                      float(scale), _stream(q))
    _check(lib, st)
    return out


def kda_packed_decode(mixed_qkv, raw_gate, raw_beta, A_log, dt_bias, state_indices, state, out=None):
    """Packed Kimi K3 T=1 decode; updates `state` in place, returns out [B, 1, 12, 128]."""
    lib = library()
    if out is None:
        out = torch.empty((mixed_qkv.shape[0], 1, 12, 128), dtype=torch.bfloat16, device=mixed_qkv.device)
    with _on(mixed_qkv.device):
        st = lib.kda_packed_decode(_ref(mixed_qkv), _ref(raw_gate), _ref(raw_beta), _ref(A_log),
                                   _ref(dt_bias), _ref(state_indices), _ref(state), _ref(out),
                                   _stream(mixed_qkv))
    _check(lib, st)
    return out


def kda_fused_decode(x, conv_weight, conv_state, raw_gate, raw_beta, A_log, dt_bias, state_indices,
                     state, output_gate, norm_weight, lower_bound=-5.0, norm_eps=1e-5, out=None):
    """Fused conv + KDA + gated RMSNorm; updates both caches, returns out [1, rows, H, 128]."""
    lib = library()
    if out is None:
        H = state.shape[1]
        out = torch.empty((1, x.shape[0], H, 128), dtype=torch.bfloat16, device=x.device)
    with _on(x.device):
        st = lib.kda_fused_decode(_ref(x), _ref(conv_weight), _ref(conv_state), _ref(raw_gate),
                                  _ref(raw_beta), _ref(A_log), _ref(dt_bias), _ref(state_indices),
                                  _ref(state), _ref(output_gate), _ref(norm_weight),
                                  int(lower_bound is not None),
                                  float(lower_bound if lower_bound is not None else 0.0),
                                  float(norm_eps), _ref(out), _stream(x))
    _check(lib, st)
    return out


def kda_packed_fused_decode(x, conv_weight, conv_state, raw_gate, raw_beta, A_log, dt_bias, state_indices,
                            query_start_loc, num_accepted_tokens, state, output_gate, norm_weight,
                            lower_bound=-5.0, norm_eps=1e-5, out=None):
    """Packed fused speculative decode; writes per-token checkpoints of both caches, returns out [R, H, 128]."""
    lib = library()
    if out is None:
        out = torch.empty((x.shape[0], state.shape[1], 128), dtype=torch.bfloat16, device=x.device)
    with _on(x.device):
        st = lib.kda_packed_fused_decode(_ref(x), _ref(conv_weight), _ref(conv_state), _ref(raw_gate),
                                         _ref(raw_beta), _ref(A_log), _ref(dt_bias), _ref(state_indices),
                                         _ref(query_start_loc), _ref(num_accepted_tokens), _ref(state),
                                         _ref(output_gate), _ref(norm_weight), int(lower_bound is not None),
                                         float(lower_bound if lower_bound is not None else 0.0),
                                         float(norm_eps), _ref(out), _stream(x))
    _check(lib, st)
    return out


def kda_spec_decode(q, k, v, g, beta, cu_seqlens, state_indices, state, t_max, out=None,
                    beta_is_logit=True, scale=DEFAULT_SCALE):
    """Ragged speculative decode; updates `state` in place, returns out [R, H, 128]."""
    lib = library()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    with _on(q.device):
        st = lib.kda_spec_decode(_ref(q), _ref(k), _ref(v), _ref(g), _ref(beta), int(bool(beta_is_logit)),
                                 _ref(cu_seqlens), int(t_max), _ref(state_indices), _ref(state),
                                 _ref(out), float(scale), _stream(q))
    _check(lib, st)
    return out


def kda_spec_verify_decode(q, k, v, g, beta, cu_seqlens, state_indices, state, t_max, out=None,
                           correction_cache=None, kg_cache=None, beta_is_logit=True, scale=DEFAULT_SCALE):
    """Speculative verify: spec outputs from a read-only state, optional commit caches."""
    lib = library()
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    cc = _ref(correction_cache) if correction_cache is not None else None
    kg = _ref(kg_cache) if kg_cache is not None else None
    with _on(q.device):
        st = lib.kda_spec_verify_decode(_ref(q), _ref(k), _ref(v), _ref(g), _ref(beta), int(bool(beta_is_logit)),
                                        _ref(cu_seqlens), int(t_max), _ref(state_indices), _ref(state), _ref(out),
                                        cc, kg, float(scale), _stream(q))
    _check(lib, st)
    return out


def kda_plan_split(op, units, state_dtype, t_max, sm_count):
    """Split the dispatcher picks (host-only query)."""
    return int(library().kda_plan_split(int(op), int(units), int(state_dtype), int(t_max), int(sm_count)))


def kda_set_split_override(split):
    """Force every later call's split (0 restores the policy)."""
    lib = library()
    _check(lib, lib.kda_set_split_override(int(split)))


def kda_plan_schedule(op, units, state_dtype, t_max, sm_count):
    """Schedule the dispatcher picks (host-only query)."""
    return int(library().kda_plan_schedule(int(op), int(units), int(state_dtype), int(t_max), int(sm_count)))


def kda_set_schedule_override(schedule):
    """Force the schedule (SCHED_SPLIT / SCHED_STREAM for T=1, SCHED_SPLIT / SCHED_MMA for the
    speculative entry points; SCHED_AUTO restores the policy)."""
    lib = library()
    _check(lib, lib.kda_set_schedule_override(int(schedule)))


def kda_device_error(clear=True):
    """Device error word of the streaming kernels (synchronises the device)."""
    lib = library()
    flags = ctypes.c_uint32(0)
    _check(lib, lib.kda_device_error(ctypes.byref(flags), int(bool(clear))))
    return int(flags.value)


def kda_selftest_wait_timeout(device=None):
    """Launch the bounded-wait self-test on the current stream (sets device error bit 2 after ~2 s)."""
    lib = library()
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(dev):
        st = lib.kda_selftest_wait_timeout(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))
    _check(lib, st)


def kda_version():
    return library().kda_version().decode()
