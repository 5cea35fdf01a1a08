// libkda C ABI: host-side contract validation, split policy and launch.
//
// Every entry point validates its whole contract on the host before
// launching anything (no device reads, no allocation, no synchronisation),
// then launches exactly one kernel on the caller's stream.
#include <cuda_runtime.h>

#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "../../include/kda.h"
#include "kda_launch.h"
#include "kda_packed_fused.h"

namespace {

constexpr int64_t kD = 128;
constexpr int64_t kUnit = kD * kD;  // elements of one (slot, head) state block

thread_local std::string g_last_error;
std::atomic<int> g_split_override{0};
std::atomic<int> g_schedule_override{KDA_SCHED_AUTO};

kda_status fail(kda_status st, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return st;
}

#define KDA_CHECK(cond, st, ...)          \
  do {                                    \
    if (!(cond)) return fail(st, __VA_ARGS__); \
  } while (0)

#define KDA_TRY(expr)                \
  do {                               \
    kda_status s__ = (expr);         \
    if (s__ != KDA_OK) return s__;   \
  } while (0)

int64_t esize(int32_t dtype) { return dtype == KDA_BF16 ? 2 : 4; }

const char* dtname(int32_t d) {
  switch (d) {
    case KDA_F32: return "float32";
    case KDA_BF16: return "bfloat16";
    case KDA_I32: return "int32";
    default: return "unknown";
  }
}

// A tensor viewed with a fixed rank after dropping a leading/inner unit axis.
struct View {
  const char* name = nullptr;
  char* data = nullptr;
  int32_t dtype = -1;
  int ndim = 0;
  int64_t shape[4] = {0, 0, 0, 0};
  int64_t stride[4] = {0, 0, 0, 0};
  int64_t numel() const {
    int64_t n = 1;
    for (int i = 0; i < ndim; ++i) n *= shape[i];
    return n;
  }
  // Byte range [lo, hi) touched by the view (all strides are positive).
  void range(uintptr_t* lo, uintptr_t* hi) const {
    if (numel() == 0) { *lo = *hi = 0; return; }
    int64_t ext = 1;
    for (int i = 0; i < ndim; ++i) ext += (shape[i] - 1) * stride[i];
    *lo = reinterpret_cast<uintptr_t>(data);
    *hi = *lo + static_cast<uintptr_t>(ext * esize(dtype));
  }
};

kda_status raw_view(const kda_tensor* t, const char* name, View* v) {
  KDA_CHECK(t != nullptr, KDA_ERR_INVALID_ARG, "%s: null tensor descriptor", name);
  KDA_CHECK(t->ndim >= 1 && t->ndim <= 4, KDA_ERR_INVALID_ARG, "%s: ndim %d not in 1..4", name, t->ndim);
  KDA_CHECK(t->dtype == KDA_F32 || t->dtype == KDA_BF16 || t->dtype == KDA_I32, KDA_ERR_INVALID_ARG,
            "%s: unknown dtype %d", name, t->dtype);
  v->name = name;
  v->data = static_cast<char*>(t->data);
  v->dtype = t->dtype;
  v->ndim = t->ndim;
  for (int i = 0; i < t->ndim; ++i) {
    KDA_CHECK(t->shape[i] >= 0, KDA_ERR_INVALID_ARG, "%s: negative extent %lld on axis %d", name,
              (long long)t->shape[i], i);
    KDA_CHECK(t->stride[i] > 0 || t->shape[i] <= 1, KDA_ERR_INVALID_ARG,
              "%s: stride %lld on axis %d must be positive", name, (long long)t->stride[i], i);
    v->shape[i] = t->shape[i];
    v->stride[i] = t->shape[i] <= 1 && t->stride[i] <= 0 ? 1 : t->stride[i];
  }
  KDA_CHECK(v->data != nullptr || v->numel() == 0, KDA_ERR_INVALID_ARG, "%s: null data pointer", name);
  return KDA_OK;
}

// Accepts rank `want`, or rank want+1 with a unit axis at `unit_axis` (dropped).
kda_status ranked_view(const kda_tensor* t, const char* name, int want, int unit_axis, View* v) {
  KDA_TRY(raw_view(t, name, v));
  if (v->ndim == want + 1 && unit_axis >= 0 && v->shape[unit_axis] == 1) {
    for (int i = unit_axis; i < v->ndim - 1; ++i) {
      v->shape[i] = v->shape[i + 1];
      v->stride[i] = v->stride[i + 1];
    }
    v->ndim = want;
  }
  KDA_CHECK(v->ndim == want, KDA_ERR_INVALID_ARG, "%s: expected rank %d, got %d", name, want, t->ndim);
  return KDA_OK;
}

kda_status need_dtype(const View& v, int32_t a, int32_t b = -1) {
  KDA_CHECK(v.dtype == a || v.dtype == b, KDA_ERR_INVALID_ARG, "%s: dtype %s not accepted", v.name,
            dtname(v.dtype));
  return KDA_OK;
}

kda_status need_shape(const View& v, int axis, int64_t want) {
  KDA_CHECK(v.shape[axis] == want, KDA_ERR_INVALID_ARG, "%s: axis %d is %lld, expected %lld", v.name, axis,
            (long long)v.shape[axis], (long long)want);
  return KDA_OK;
}

kda_status need_contiguous(const View& v) {
  int64_t expect = 1;
  for (int i = v.ndim - 1; i >= 0; --i) {
    KDA_CHECK(v.shape[i] <= 1 || v.stride[i] == expect, KDA_ERR_INVALID_ARG, "%s: must be contiguous", v.name);
    expect *= v.shape[i];
  }
  return KDA_OK;
}

// Activation vectors [rows, heads, 128]: channel stride 1, 4-element aligned
// rows and heads so lanes can read 4 channels with one 8/16-byte load.
kda_status need_vec_layout(const View& v) {
  KDA_CHECK(v.stride[v.ndim - 1] == 1, KDA_ERR_INVALID_ARG, "%s: channel axis must have stride 1", v.name);
  for (int i = 0; i < v.ndim - 1; ++i)
    KDA_CHECK(v.shape[i] <= 1 || v.stride[i] % 4 == 0, KDA_ERR_INVALID_ARG,
              "%s: stride %lld on axis %d must be a multiple of 4 elements", v.name, (long long)v.stride[i], i);
  KDA_CHECK(reinterpret_cast<uintptr_t>(v.data) % (4 * esize(v.dtype)) == 0, KDA_ERR_INVALID_ARG,
            "%s: data must be %lld-byte aligned", v.name, (long long)(4 * esize(v.dtype)));
  return KDA_OK;
}

// State pool [num_slots, H, 128, 128]: per-slot block contiguous, slot stride
// >= H*128*128 and 16-byte aligned.
kda_status need_state_layout(const View& v, int64_t H) {
  KDA_TRY(need_dtype(v, KDA_F32, KDA_BF16));
  KDA_CHECK(v.ndim == 4, KDA_ERR_INVALID_ARG, "state: expected rank 4");
  KDA_TRY(need_shape(v, 1, H));
  KDA_TRY(need_shape(v, 2, kD));
  KDA_TRY(need_shape(v, 3, kD));
  KDA_CHECK(v.shape[0] >= 1 && v.shape[0] <= INT32_MAX, KDA_ERR_INVALID_ARG, "state: num_slots %lld out of range",
            (long long)v.shape[0]);
  KDA_CHECK(v.stride[3] == 1 && v.stride[2] == kD && (H <= 1 || v.stride[1] == kUnit), KDA_ERR_INVALID_ARG,
            "state: each slot's [H, 128, 128] block must be contiguous");
  KDA_CHECK(v.shape[0] <= 1 || v.stride[0] >= H * kUnit, KDA_ERR_INVALID_ARG,
            "state: slot stride %lld overlaps slots (needs >= %lld)", (long long)v.stride[0], (long long)(H * kUnit));
  KDA_CHECK((v.stride[0] * esize(v.dtype)) % 16 == 0 || v.shape[0] <= 1, KDA_ERR_INVALID_ARG,
            "state: slot stride must keep 16-byte alignment");
  KDA_CHECK(reinterpret_cast<uintptr_t>(v.data) % 16 == 0, KDA_ERR_INVALID_ARG, "state: data must be 16-byte aligned");
  return KDA_OK;
}

kda_status need_indices(const View& v, int64_t n) {
  KDA_TRY(need_dtype(v, KDA_I32));
  KDA_CHECK(v.ndim == 1, KDA_ERR_INVALID_ARG, "%s: expected rank 1", v.name);
  KDA_TRY(need_shape(v, 0, n));
  KDA_CHECK(v.shape[0] <= 1 || v.stride[0] == 1, KDA_ERR_INVALID_ARG, "%s: must be contiguous", v.name);
  return KDA_OK;
}

kda_status need_f32_vector(const View& v, int64_t n) {
  KDA_TRY(need_dtype(v, KDA_F32));
  KDA_CHECK(v.numel() == n, KDA_ERR_INVALID_ARG, "%s: expected %lld elements, got %lld", v.name, (long long)n,
            (long long)v.numel());
  KDA_TRY(need_contiguous(v));
  KDA_CHECK(reinterpret_cast<uintptr_t>(v.data) % 16 == 0, KDA_ERR_INVALID_ARG, "%s: data must be 16-byte aligned",
            v.name);
  return KDA_OK;
}

kda_status need_out(const View& v) {
  KDA_TRY(need_dtype(v, KDA_BF16));
  KDA_TRY(need_contiguous(v));
  KDA_CHECK(reinterpret_cast<uintptr_t>(v.data) % 16 == 0, KDA_ERR_INVALID_ARG, "%s: data must be 16-byte aligned",
            v.name);
  return KDA_OK;
}

bool overlap(const View& a, const View& b) {
  uintptr_t alo, ahi, blo, bhi;
  a.range(&alo, &ahi);
  b.range(&blo, &bhi);
  if (alo == ahi || blo == bhi) return false;
  return alo < bhi && blo < ahi;
}

// `w` is written: it must not share bytes with any other argument.
kda_status no_alias(const View& w, std::initializer_list<const View*> others) {
  for (const View* o : others)
    KDA_CHECK(!overlap(w, *o), KDA_ERR_ALIAS, "%s overlaps %s", w.name, o->name);
  return KDA_OK;
}

// ---- device properties (cached per device) ------------------------------------

struct DeviceInfo {
  int cc_major = 0, cc_minor = 0, sms = 0;
  bool valid = false;
};
std::mutex g_dev_mu;
DeviceInfo g_dev[64];

kda_status current_device(cudaStream_t stream, DeviceInfo* info) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  KDA_CHECK(e == cudaSuccess, KDA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  KDA_CHECK(dev >= 0 && dev < 64, KDA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_dev[dev].valid) {
      DeviceInfo d;
      e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
      if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
      KDA_CHECK(e == cudaSuccess, KDA_ERR_CUDA, "cudaDeviceGetAttribute: %s", cudaGetErrorString(e));
      d.valid = true;
      g_dev[dev] = d;
    }
    *info = g_dev[dev];
  }
  KDA_CHECK(info->cc_major == 10 && info->cc_minor == 3, KDA_ERR_UNSUPPORTED,
            "device %d is compute capability %d.%d; this library is built for sm_103a (GB300) only", dev,
            info->cc_major, info->cc_minor);
  // The stream's device is checked outside graph capture only: the query is
  // not permitted on a capturing stream (a capture on a stream of another
  // device fails at launch instead).
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (stream != nullptr) {
    e = cudaStreamIsCapturing(stream, &cap);
    KDA_CHECK(e == cudaSuccess, KDA_ERR_INVALID_ARG, "stream: %s", cudaGetErrorString(e));
  }
  if (stream != nullptr && cap == cudaStreamCaptureStatusNone) {
    int sdev = -1;
    e = cudaStreamGetDevice(stream, &sdev);
    KDA_CHECK(e == cudaSuccess, KDA_ERR_INVALID_ARG, "stream: %s", cudaGetErrorString(e));
    KDA_CHECK(sdev == dev, KDA_ERR_INVALID_ARG, "stream belongs to device %d, current device is %d", sdev, dev);
  }
  return KDA_OK;
}

// Schedule policy, measured on GB300 (152 SMs) with CUDA-graph timings and
// an L2 flush between replays:
//  - float32 state, T=1: the split kernel (4 value slabs per unit) reaches
//    ~95% of copy bandwidth at B >= 128 and beats the streaming kernel;
//  - bfloat16 state, T=1: the streaming kernel once the units fill five per
//    SM (packed K3 B >= 64), the split kernel below;
//  - fused: the streaming kernel from 2.5 units per SM (H=32 rows=12:
//    14.4 vs 15.8 us split, fp32; rows=256: 164.8 us, 91 % of copy
//    bandwidth), split below (rows=8: 11.3 vs 12.4 us);
//  - speculative rows: the split kernel, except a bfloat16 state with
//    t_max >= 14, which takes the tensor-core chunked form (N=128, rows of
//    exactly T tokens: T=14 102.5 vs 129.6 us, T=16 104.6 vs 142.1 us;
//    ragged rows up to T: 77.0 vs 75.0, 81.1 vs 79.1 us; at T=12 ragged rows
//    lose 5 % and at T=10 11 %, so below 14 the split kernel stays).
int plan_schedule(int op, int64_t units, int state_dtype, int t_max, int sms) {
  const int forced = g_schedule_override.load();
  if (op == KDA_OP_PACKED_FUSED) return KDA_SCHED_SPLIT;
  if (op == KDA_OP_SPEC) {
    (void)units; (void)sms;
    if (forced == KDA_SCHED_SPLIT || forced == KDA_SCHED_MMA) return forced;
    if (forced == KDA_SCHED_STREAM || g_split_override.load() != 0) return KDA_SCHED_SPLIT;
    return state_dtype == KDA_BF16 && t_max >= 14 ? KDA_SCHED_MMA : KDA_SCHED_SPLIT;
  }
  if (forced == KDA_SCHED_SPLIT || forced == KDA_SCHED_STREAM) return forced;
  if (g_split_override.load() != 0) return KDA_SCHED_SPLIT;
  if (op == KDA_OP_FUSED) return 2 * units >= 5LL * sms ? KDA_SCHED_STREAM : KDA_SCHED_SPLIT;
  if (state_dtype == KDA_F32) return KDA_SCHED_SPLIT;
  return units >= 5LL * sms ? KDA_SCHED_STREAM : KDA_SCHED_SPLIT;
}

// Every head vector of the view starts on a 16-byte boundary (bulk copies).
bool rows_aligned16(const View& v) {
  if (reinterpret_cast<uintptr_t>(v.data) % 16 != 0) return false;
  for (int i = 0; i < v.ndim - 1; ++i)
    if (v.shape[i] > 1 && (v.stride[i] * esize(v.dtype)) % 16 != 0) return false;
  return true;
}

// Packed fused speculative decode: CTAs per (sequence, head) cluster.  A
// cluster spreads a unit's conv, checkpoint stores and token updates over
// its SMs (each CTA convolves its own slab of q, k and v and shares its q
// and k activations through distributed shared memory) but repeats the
// coefficient phase, and the row forms (4 and 8 CTAs) pay a CTA barrier per
// token.  Measured on GB300 (H=12, T=5, CUDA-graph replays of 16 calls after
// an L2 flush, us at 1 / 2 / 4 / 8 CTAs): fp32 N=1 12.6 / 11.6 / 9.9 / 11.2,
// N=2 12.9 / 11.9 / 10.3 / 11.7, N=3 13.0 / 12.0 / 14.1 / 12.2, N=4
// 13.0 / 13.6 / 14.7 / 19.4; bf16 N=1 11.1 / 11.1 / 13.1 / 12.8, N=3
// 11.3 / 11.3 / 19.6 / 15.5, N=4 11.4 / 12.4 / 20.2 / 21.7.  So fp32 takes 4
// CTAs while 6 units <= SMs and 2 while 4 units <= SMs, bf16 2 while 4
// units <= SMs; otherwise one persistent CTA per unit.
int plan_cluster(int64_t units, int state_dtype, int sms) {
  if (state_dtype == KDA_F32 && 6 * units <= sms) return 4;
  return 4 * units <= sms ? 2 : 1;
}

int plan_split(int op, int64_t units, int state_dtype, int t_max, int sms) {
  (void)t_max;
  const int forced = g_split_override.load();
  // Fused split schedule: cluster of CTAs per (row, head).  Measured on
  // GB300, one CTA is never slower than 2 or 4 (H=8 N=1: 5.4 / 5.7 / 5.8 us;
  // H=32 N=4: 6.0 / 7.2 / 8.3 us): a small batch waits on the chain slot ->
  // state and conv cache -> update -> store, which a split does not shorten,
  // and the cluster barriers add to it.  Clusters only when forced.
  if (op == KDA_OP_FUSED) return forced == 0 ? 1 : (forced > 4 ? 4 : forced);
  if (forced != 0) return op == KDA_OP_PACKED_FUSED ? (forced > 8 ? 8 : forced) : forced;
  // Measured on GB300 for the split kernel: speculative rows (T tokens of
  // work per state block) 2 value slabs per unit at every size; T=1 with
  // the units at five or more per SM 4 slabs, fewer than half the SM count
  // 16 slabs, 8 in between.
  if (op == KDA_OP_SPEC) return 2;
  if (op == KDA_OP_PACKED_FUSED) return plan_cluster(units, state_dtype, sms);
  if (units >= 5LL * sms) return 4;
  return 2 * units <= sms ? 16 : 8;
}

kda_status check_launch(cudaError_t e) {
  KDA_CHECK(e == cudaSuccess, KDA_ERR_CUDA, "kernel launch: %s", cudaGetErrorString(e));
  return KDA_OK;
}

kda_status check_grid(int64_t blocks) {
  KDA_CHECK(blocks < (int64_t)INT32_MAX, KDA_ERR_UNSUPPORTED, "grid of %lld CTAs too large", (long long)blocks);
  return KDA_OK;
}

kda_status check_gate(int32_t has_lower_bound, float lower_bound) {
  KDA_CHECK(has_lower_bound == 0 || has_lower_bound == 1, KDA_ERR_INVALID_ARG, "has_lower_bound must be 0 or 1");
  KDA_CHECK(!has_lower_bound || (std::isfinite(lower_bound) && lower_bound < 0.f), KDA_ERR_INVALID_ARG,
            "lower_bound must be a finite negative number");
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_recurrent_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                const kda_tensor* raw_gate, const kda_tensor* raw_beta, const kda_tensor* A_log,
                                const kda_tensor* dt_bias, const kda_tensor* state_indices, const kda_tensor* state,
                                const kda_tensor* out, int32_t has_lower_bound, float lower_bound, float scale,
                                void* stream) {
  View Q, K, V, G, Bt, A, DT, I, S, O;
  KDA_TRY(ranked_view(q, "q", 3, 1, &Q));
  KDA_TRY(ranked_view(k, "k", 3, 1, &K));
  KDA_TRY(ranked_view(v, "v", 3, 1, &V));
  KDA_TRY(ranked_view(raw_gate, "raw_gate", 3, 1, &G));
  KDA_TRY(ranked_view(raw_beta, "raw_beta", 2, 1, &Bt));
  KDA_TRY(raw_view(A_log, "A_log", &A));
  KDA_TRY(raw_view(dt_bias, "dt_bias", &DT));
  KDA_TRY(raw_view(state_indices, "state_indices", &I));
  KDA_TRY(raw_view(state, "state", &S));
  KDA_TRY(ranked_view(out, "out", 3, 1, &O));

  const int64_t B = Q.shape[0], H = Q.shape[1];
  KDA_CHECK(H >= 1, KDA_ERR_INVALID_ARG, "q: need at least one head");
  KDA_TRY(need_dtype(Q, KDA_F32, KDA_BF16));
  KDA_TRY(need_shape(Q, 2, kD));
  for (View* t : {&K, &V}) {
    KDA_CHECK(t->dtype == Q.dtype, KDA_ERR_INVALID_ARG, "%s: dtype must match q", t->name);
    KDA_TRY(need_shape(*t, 0, B));
    KDA_TRY(need_shape(*t, 1, H));
    KDA_TRY(need_shape(*t, 2, kD));
  }
  KDA_TRY(need_dtype(G, KDA_F32, KDA_BF16));
  KDA_TRY(need_shape(G, 0, B));
  KDA_TRY(need_shape(G, 1, H));
  KDA_TRY(need_shape(G, 2, kD));
  for (View* t : {&Q, &K, &V, &G}) KDA_TRY(need_vec_layout(*t));
  KDA_TRY(need_dtype(Bt, KDA_F32, KDA_BF16));
  KDA_TRY(need_shape(Bt, 0, B));
  KDA_TRY(need_shape(Bt, 1, H));
  KDA_TRY(need_f32_vector(A, H));
  KDA_TRY(need_f32_vector(DT, H * kD));
  KDA_TRY(need_indices(I, B));
  KDA_TRY(need_state_layout(S, H));
  KDA_TRY(need_out(O));
  KDA_TRY(need_shape(O, 0, B));
  KDA_TRY(need_shape(O, 1, H));
  KDA_TRY(need_shape(O, 2, kD));
  KDA_TRY(check_gate(has_lower_bound, lower_bound));
  KDA_CHECK(std::isfinite(scale) && scale > 0.f, KDA_ERR_INVALID_ARG, "scale must be finite and positive");
  KDA_TRY(no_alias(O, {&Q, &K, &V, &G, &Bt, &A, &DT, &I, &S}));
  KDA_TRY(no_alias(S, {&Q, &K, &V, &G, &Bt, &A, &DT, &I}));
  if (B == 0) return KDA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  int sched = plan_schedule(KDA_OP_RECURRENT, B * H, S.dtype, 1, dev.sms);
  const bool stream_ok = rows_aligned16(Q) && rows_aligned16(K) && rows_aligned16(V) && rows_aligned16(G) &&
                         B * H <= INT32_MAX;
  if (sched == KDA_SCHED_STREAM && !stream_ok) {
    KDA_CHECK(g_schedule_override.load() != KDA_SCHED_STREAM, KDA_ERR_UNSUPPORTED,
              "stream schedule forced but an activation head vector is not 16-byte aligned");
    sched = KDA_SCHED_SPLIT;
  }
  const int split = sched == KDA_SCHED_STREAM ? 1 : plan_split(KDA_OP_RECURRENT, B * H, S.dtype, 1, dev.sms);
  KDA_CHECK(kda::split_supported(split), KDA_ERR_INVALID_ARG, "split %d has no kernel", split);
  KDA_TRY(check_grid(B * H * split));

  kda::T1Args a{};
  a.q = Q.data; a.k = K.data; a.v = V.data; a.gate = G.data; a.beta = Bt.data;
  a.q_rs = Q.stride[0]; a.q_hs = Q.stride[1];
  a.k_rs = K.stride[0]; a.k_hs = K.stride[1];
  a.v_rs = V.stride[0]; a.v_hs = V.stride[1];
  a.g_rs = G.stride[0]; a.g_hs = G.stride[1];
  a.b_rs = Bt.stride[0]; a.b_hs = Bt.stride[1];
  a.qkv_dtype = Q.dtype; a.gate_dtype = G.dtype; a.beta_dtype = Bt.dtype;
  a.A_log = reinterpret_cast<const float*>(A.data);
  a.dt_bias = reinterpret_cast<const float*>(DT.data);
  a.idx = reinterpret_cast<const int32_t*>(I.data);
  a.state = S.data; a.slot_stride = S.stride[0]; a.num_slots = (int32_t)S.shape[0];
  a.out = O.data; a.B = (int32_t)B; a.H = (int32_t)H;
  a.gate_mode = has_lower_bound ? kda::KDA_GATE_LOWER_BOUND : kda::KDA_GATE_SOFTPLUS;
  a.lower_bound = lower_bound; a.scale = scale;
  if (sched == KDA_SCHED_STREAM) return check_launch(kda::launch_t1_stream(a, S.dtype, dev.sms, st));
  return check_launch(kda::launch_t1(a, S.dtype, split, st));
}

kda_status kda_packed_decode(const kda_tensor* mixed_qkv, const kda_tensor* raw_gate, const kda_tensor* raw_beta,
                             const kda_tensor* A_log, const kda_tensor* dt_bias, const kda_tensor* state_indices,
                             const kda_tensor* state, const kda_tensor* out, void* stream) {
  constexpr int64_t H = 12, HD = H * kD;
  View M, G, Bt, A, DT, I, S, O;
  KDA_TRY(ranked_view(mixed_qkv, "mixed_qkv", 2, -1, &M));
  KDA_TRY(ranked_view(raw_gate, "raw_gate", 2, -1, &G));
  KDA_TRY(ranked_view(raw_beta, "raw_beta", 2, -1, &Bt));
  KDA_TRY(raw_view(A_log, "A_log", &A));
  KDA_TRY(raw_view(dt_bias, "dt_bias", &DT));
  KDA_TRY(raw_view(state_indices, "state_indices", &I));
  KDA_TRY(raw_view(state, "state", &S));
  KDA_TRY(ranked_view(out, "out", 3, 1, &O));
  const int64_t B = M.shape[0];
  KDA_TRY(need_dtype(M, KDA_BF16));
  KDA_TRY(need_shape(M, 1, 3 * HD));
  KDA_TRY(need_vec_layout(M));
  KDA_TRY(need_dtype(G, KDA_BF16));
  KDA_TRY(need_shape(G, 0, B));
  KDA_TRY(need_shape(G, 1, HD));
  KDA_TRY(need_vec_layout(G));
  KDA_TRY(need_dtype(Bt, KDA_BF16));
  KDA_TRY(need_shape(Bt, 0, B));
  KDA_TRY(need_shape(Bt, 1, H));
  KDA_TRY(need_f32_vector(A, H));
  KDA_TRY(need_f32_vector(DT, HD));
  KDA_TRY(need_indices(I, B));
  KDA_TRY(need_state_layout(S, H));
  KDA_CHECK(S.dtype == KDA_BF16, KDA_ERR_INVALID_ARG, "state: the packed contract takes a bfloat16 pool");
  KDA_TRY(need_out(O));
  KDA_TRY(need_shape(O, 0, B));
  KDA_TRY(need_shape(O, 1, H));
  KDA_TRY(need_shape(O, 2, kD));
  KDA_TRY(no_alias(O, {&M, &G, &Bt, &A, &DT, &I, &S}));
  KDA_TRY(no_alias(S, {&M, &G, &Bt, &A, &DT, &I}));
  if (B == 0) return KDA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  int sched = plan_schedule(KDA_OP_PACKED, B * H, S.dtype, 1, dev.sms);
  if (sched == KDA_SCHED_STREAM && !(rows_aligned16(M) && rows_aligned16(G))) {
    KDA_CHECK(g_schedule_override.load() != KDA_SCHED_STREAM, KDA_ERR_UNSUPPORTED,
              "stream schedule forced but a packed row is not 16-byte aligned");
    sched = KDA_SCHED_SPLIT;
  }
  const int split = sched == KDA_SCHED_STREAM ? 1 : plan_split(KDA_OP_PACKED, B * H, S.dtype, 1, dev.sms);
  KDA_CHECK(kda::split_supported(split), KDA_ERR_INVALID_ARG, "split %d has no kernel", split);
  KDA_TRY(check_grid(B * H * split));

  kda::T1Args a{};
  const char* m = M.data;  // bfloat16 elements: 2 bytes each
  a.q = m; a.k = m + 2 * HD; a.v = m + 4 * HD;
  a.q_rs = a.k_rs = a.v_rs = M.stride[0];
  a.q_hs = a.k_hs = a.v_hs = kD;
  a.gate = G.data; a.g_rs = G.stride[0]; a.g_hs = kD;
  a.beta = Bt.data; a.b_rs = Bt.stride[0]; a.b_hs = Bt.stride[1];
  a.qkv_dtype = kda::KDA_DT_BF16; a.gate_dtype = kda::KDA_DT_BF16; a.beta_dtype = kda::KDA_DT_BF16;
  a.A_log = reinterpret_cast<const float*>(A.data);
  a.dt_bias = reinterpret_cast<const float*>(DT.data);
  a.idx = reinterpret_cast<const int32_t*>(I.data);
  a.state = S.data; a.slot_stride = S.stride[0]; a.num_slots = (int32_t)S.shape[0];
  a.out = O.data; a.B = (int32_t)B; a.H = (int32_t)H;
  a.gate_mode = kda::KDA_GATE_LOWER_BOUND;
  a.lower_bound = -5.0f;
  a.scale = 0.08838834764831845f;  // 1/sqrt(128)
  if (sched == KDA_SCHED_STREAM) return check_launch(kda::launch_t1_stream(a, S.dtype, dev.sms, st));
  return check_launch(kda::launch_t1(a, S.dtype, split, st));
}

kda_status kda_fused_decode(const kda_tensor* x, const kda_tensor* conv_weight, const kda_tensor* conv_state,
                            const kda_tensor* raw_gate, const kda_tensor* raw_beta, const kda_tensor* A_log,
                            const kda_tensor* dt_bias, const kda_tensor* state_indices, const kda_tensor* state,
                            const kda_tensor* output_gate, const kda_tensor* norm_weight, int32_t has_lower_bound,
                            float lower_bound, float norm_eps, const kda_tensor* out, void* stream) {
  View X, W, C, G, Bt, A, DT, I, S, OG, NW, O;
  KDA_TRY(ranked_view(x, "x", 2, -1, &X));
  KDA_TRY(raw_view(conv_weight, "conv_weight", &W));
  KDA_TRY(ranked_view(conv_state, "conv_state", 3, -1, &C));
  KDA_TRY(ranked_view(raw_gate, "raw_gate", 3, 0, &G));
  KDA_TRY(ranked_view(raw_beta, "raw_beta", 2, 0, &Bt));
  KDA_TRY(raw_view(A_log, "A_log", &A));
  KDA_TRY(raw_view(dt_bias, "dt_bias", &DT));
  KDA_TRY(raw_view(state_indices, "state_indices", &I));
  KDA_TRY(raw_view(state, "state", &S));
  KDA_TRY(ranked_view(output_gate, "output_gate", 3, 0, &OG));
  KDA_TRY(raw_view(norm_weight, "norm_weight", &NW));
  KDA_TRY(ranked_view(out, "out", 3, 0, &O));

  KDA_CHECK(S.ndim == 4, KDA_ERR_INVALID_ARG, "state: expected rank 4");
  const int64_t H = S.shape[1], HD = H * kD, rows = X.shape[0];
  KDA_CHECK(H >= 1, KDA_ERR_INVALID_ARG, "state: need at least one head");
  KDA_TRY(need_state_layout(S, H));
  KDA_TRY(need_dtype(X, KDA_BF16));
  KDA_TRY(need_shape(X, 1, 3 * HD));
  KDA_CHECK(X.stride[1] == 1, KDA_ERR_INVALID_ARG, "x: channel axis must have stride 1");
  KDA_TRY(need_dtype(W, KDA_F32));
  KDA_CHECK(W.ndim == 3, KDA_ERR_INVALID_ARG, "conv_weight: expected rank 3");
  KDA_TRY(need_shape(W, 0, 3));
  KDA_TRY(need_shape(W, 1, 4));
  KDA_TRY(need_shape(W, 2, HD));
  KDA_TRY(need_contiguous(W));
  KDA_TRY(need_dtype(C, KDA_BF16));
  KDA_TRY(need_shape(C, 0, S.shape[0]));
  KDA_TRY(need_shape(C, 1, 3 * HD));
  KDA_TRY(need_shape(C, 2, 3));
  KDA_CHECK(C.stride[1] == 1 && C.stride[2] == 3 * HD, KDA_ERR_INVALID_ARG,
            "conv_state: strides must be [slot_stride, 1, 3*H*128]");
  KDA_CHECK(C.shape[0] <= 1 || C.stride[0] >= 9 * HD, KDA_ERR_INVALID_ARG, "conv_state: slot stride overlaps slots");
  KDA_TRY(need_dtype(G, KDA_BF16));
  KDA_TRY(need_shape(G, 0, rows));
  KDA_TRY(need_shape(G, 1, H));
  KDA_TRY(need_shape(G, 2, kD));
  KDA_CHECK(G.stride[2] == 1, KDA_ERR_INVALID_ARG, "raw_gate: channel axis must have stride 1");
  KDA_TRY(need_dtype(Bt, KDA_BF16));
  KDA_TRY(need_shape(Bt, 0, rows));
  KDA_TRY(need_shape(Bt, 1, H));
  KDA_TRY(need_f32_vector(A, H));
  KDA_TRY(need_f32_vector(DT, HD));
  KDA_TRY(need_indices(I, rows));
  KDA_TRY(need_dtype(OG, KDA_BF16));
  KDA_TRY(need_shape(OG, 0, rows));
  KDA_TRY(need_shape(OG, 1, H));
  KDA_TRY(need_shape(OG, 2, kD));
  KDA_TRY(need_vec_layout(OG));
  KDA_TRY(need_f32_vector(NW, kD));
  KDA_TRY(need_out(O));
  KDA_TRY(need_shape(O, 0, rows));
  KDA_TRY(need_shape(O, 1, H));
  KDA_TRY(need_shape(O, 2, kD));
  KDA_TRY(check_gate(has_lower_bound, lower_bound));
  KDA_CHECK(std::isfinite(norm_eps) && norm_eps >= 0.f, KDA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  KDA_TRY(no_alias(O, {&X, &W, &C, &G, &Bt, &A, &DT, &I, &S, &OG, &NW}));
  KDA_TRY(no_alias(S, {&X, &W, &C, &G, &Bt, &A, &DT, &I, &OG, &NW}));
  KDA_TRY(no_alias(C, {&X, &W, &G, &Bt, &A, &DT, &I, &OG, &NW}));
  if (rows == 0) return KDA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  KDA_TRY(check_grid(rows * H));
  int sched = plan_schedule(KDA_OP_FUSED, rows * H, S.dtype, 1, dev.sms);
  const bool stream_ok = rows_aligned16(X) && rows_aligned16(G) && rows_aligned16(OG) &&
                         reinterpret_cast<uintptr_t>(C.data) % 16 == 0 &&
                         reinterpret_cast<uintptr_t>(W.data) % 16 == 0 &&
                         (C.shape[0] <= 1 || (C.stride[0] * 2) % 16 == 0) && rows * H <= INT32_MAX;
  if (sched == KDA_SCHED_STREAM && !stream_ok) {
    KDA_CHECK(g_schedule_override.load() != KDA_SCHED_STREAM, KDA_ERR_UNSUPPORTED,
              "stream schedule forced but an activation row, a conv-cache slot or conv_weight is not 16-byte aligned");
    sched = KDA_SCHED_SPLIT;
  }

  kda::FusedArgs a{};
  a.x = X.data; a.x_rs = X.stride[0];
  a.conv_w = reinterpret_cast<const float*>(W.data);
  a.conv_state = C.data; a.cs_slot_stride = C.stride[0]; a.cs_tap_stride = C.stride[2];
  a.gate = G.data; a.g_rs = G.stride[0]; a.g_hs = G.stride[1];
  a.beta = Bt.data; a.b_rs = Bt.stride[0]; a.b_hs = Bt.stride[1];
  a.A_log = reinterpret_cast<const float*>(A.data);
  a.dt_bias = reinterpret_cast<const float*>(DT.data);
  a.idx = reinterpret_cast<const int32_t*>(I.data);
  a.state = S.data; a.slot_stride = S.stride[0]; a.num_slots = (int32_t)S.shape[0];
  a.out_gate = OG.data; a.og_rs = OG.stride[0]; a.og_hs = OG.stride[1];
  a.norm_w = reinterpret_cast<const float*>(NW.data);
  a.out = O.data; a.rows = (int32_t)rows; a.H = (int32_t)H;
  a.gate_mode = has_lower_bound ? kda::KDA_GATE_LOWER_BOUND : kda::KDA_GATE_SOFTPLUS;
  a.lower_bound = lower_bound; a.norm_eps = norm_eps;
  a.scale = 0.08838834764831845f;  // 1/sqrt(128)
  if (sched == KDA_SCHED_STREAM) return check_launch(kda::launch_fused_stream(a, S.dtype, dev.sms, st));
  const int cluster = plan_split(KDA_OP_FUSED, rows * H, S.dtype, 1, dev.sms);
  return check_launch(kda::launch_fused(a, S.dtype, cluster, st));
}

kda_status kda_packed_fused_decode(const kda_tensor* x, const kda_tensor* conv_weight, const kda_tensor* conv_state,
                                   const kda_tensor* raw_gate, const kda_tensor* raw_beta, const kda_tensor* A_log,
                                   const kda_tensor* dt_bias, const kda_tensor* state_indices,
                                   const kda_tensor* query_start_loc, const kda_tensor* num_accepted_tokens,
                                   const kda_tensor* state, const kda_tensor* output_gate,
                                   const kda_tensor* norm_weight, int32_t has_lower_bound, float lower_bound,
                                   float norm_eps, const kda_tensor* out, void* stream) {
  View X, W, C, G, Bt, A, DT, I, Q, AC, S, OG, NW, O;
  KDA_TRY(ranked_view(x, "x", 2, -1, &X));
  KDA_TRY(raw_view(conv_weight, "conv_weight", &W));
  KDA_TRY(ranked_view(conv_state, "conv_state", 3, -1, &C));
  KDA_TRY(ranked_view(raw_gate, "raw_gate", 3, 0, &G));
  KDA_TRY(ranked_view(raw_beta, "raw_beta", 2, 0, &Bt));
  KDA_TRY(raw_view(A_log, "A_log", &A));
  KDA_TRY(raw_view(dt_bias, "dt_bias", &DT));
  KDA_TRY(ranked_view(state_indices, "state_indices", 2, -1, &I));
  KDA_TRY(raw_view(query_start_loc, "query_start_loc", &Q));
  KDA_TRY(raw_view(num_accepted_tokens, "num_accepted_tokens", &AC));
  KDA_TRY(raw_view(state, "state", &S));
  KDA_TRY(ranked_view(output_gate, "output_gate", 3, 0, &OG));
  KDA_TRY(raw_view(norm_weight, "norm_weight", &NW));
  KDA_TRY(ranked_view(out, "out", 3, 0, &O));

  KDA_CHECK(S.ndim == 4, KDA_ERR_INVALID_ARG, "state: expected rank 4");
  const int64_t H = S.shape[1], HD = H * kD, R = X.shape[0];
  KDA_CHECK(H >= 1, KDA_ERR_INVALID_ARG, "state: need at least one head");
  KDA_TRY(need_state_layout(S, H));
  KDA_TRY(need_dtype(X, KDA_BF16));
  KDA_TRY(need_shape(X, 1, 3 * HD));
  KDA_CHECK(X.stride[1] == 1, KDA_ERR_INVALID_ARG, "x: channel axis must have stride 1");
  KDA_CHECK(R <= INT32_MAX, KDA_ERR_INVALID_ARG, "x: too many token rows");
  KDA_TRY(need_dtype(W, KDA_F32));
  KDA_CHECK(W.ndim == 3, KDA_ERR_INVALID_ARG, "conv_weight: expected rank 3");
  KDA_TRY(need_shape(W, 0, 3));
  KDA_TRY(need_shape(W, 1, 4));
  KDA_TRY(need_shape(W, 2, HD));
  KDA_TRY(need_contiguous(W));
  KDA_TRY(need_dtype(C, KDA_BF16));
  KDA_TRY(need_shape(C, 0, S.shape[0]));
  KDA_TRY(need_shape(C, 1, 3 * HD));
  KDA_TRY(need_shape(C, 2, 3));
  KDA_CHECK(C.stride[1] == 1 && C.stride[2] == 3 * HD, KDA_ERR_INVALID_ARG,
            "conv_state: strides must be [slot_stride, 1, 3*H*128]");
  KDA_CHECK(C.shape[0] <= 1 || C.stride[0] >= 9 * HD, KDA_ERR_INVALID_ARG, "conv_state: slot stride overlaps slots");
  KDA_TRY(need_dtype(G, KDA_BF16));
  KDA_TRY(need_shape(G, 0, R));
  KDA_TRY(need_shape(G, 1, H));
  KDA_TRY(need_shape(G, 2, kD));
  KDA_CHECK(G.stride[2] == 1, KDA_ERR_INVALID_ARG, "raw_gate: channel axis must have stride 1");
  KDA_TRY(need_dtype(Bt, KDA_BF16));
  KDA_TRY(need_shape(Bt, 0, R));
  KDA_TRY(need_shape(Bt, 1, H));
  KDA_TRY(need_f32_vector(A, H));
  KDA_TRY(need_f32_vector(DT, HD));
  KDA_TRY(need_dtype(I, KDA_I32));
  const int64_t N = I.shape[0], cols = I.shape[1];
  KDA_CHECK(cols >= 1 && cols <= INT32_MAX, KDA_ERR_INVALID_ARG, "state_indices: need at least one checkpoint column");
  KDA_CHECK(N <= INT32_MAX - 1, KDA_ERR_INVALID_ARG, "state_indices: too many sequences");
  KDA_CHECK(cols <= 1 || I.stride[1] == 1, KDA_ERR_INVALID_ARG, "state_indices: column stride must be 1");
  KDA_TRY(need_indices(Q, N + 1));
  KDA_TRY(need_indices(AC, N));
  KDA_TRY(need_dtype(OG, KDA_BF16));
  KDA_TRY(need_shape(OG, 0, R));
  KDA_TRY(need_shape(OG, 1, H));
  KDA_TRY(need_shape(OG, 2, kD));
  KDA_TRY(need_vec_layout(OG));
  KDA_TRY(need_f32_vector(NW, kD));
  KDA_TRY(need_out(O));
  KDA_TRY(need_shape(O, 0, R));
  KDA_TRY(need_shape(O, 1, H));
  KDA_TRY(need_shape(O, 2, kD));
  KDA_TRY(check_gate(has_lower_bound, lower_bound));
  KDA_CHECK(std::isfinite(norm_eps) && norm_eps >= 0.f, KDA_ERR_INVALID_ARG, "norm_eps must be finite and >= 0");
  KDA_CHECK(rows_aligned16(X) && rows_aligned16(G) && rows_aligned16(OG), KDA_ERR_UNSUPPORTED,
            "x, raw_gate and output_gate rows must start on 16-byte boundaries (base and outer strides)");
  KDA_TRY(no_alias(O, {&X, &W, &C, &G, &Bt, &A, &DT, &I, &Q, &AC, &S, &OG, &NW}));
  KDA_TRY(no_alias(S, {&X, &W, &C, &G, &Bt, &A, &DT, &I, &Q, &AC, &OG, &NW}));
  KDA_TRY(no_alias(C, {&X, &W, &G, &Bt, &A, &DT, &I, &Q, &AC, &OG, &NW}));
  if (R == 0) return KDA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  const int cluster = plan_split(KDA_OP_PACKED_FUSED, N * H, S.dtype, 1, dev.sms);
  KDA_TRY(check_grid((N + 1) * H * cluster));

  kda::PackedFusedArgs a{};
  a.x = X.data; a.x_rs = X.stride[0];
  a.conv_w = reinterpret_cast<const float*>(W.data);
  a.conv_state = C.data; a.cs_slot_stride = C.stride[0]; a.cs_tap_stride = C.stride[2];
  a.gate = G.data; a.g_rs = G.stride[0]; a.g_hs = G.stride[1];
  a.beta = Bt.data; a.b_rs = Bt.stride[0]; a.b_hs = Bt.stride[1];
  a.A_log = reinterpret_cast<const float*>(A.data);
  a.dt_bias = reinterpret_cast<const float*>(DT.data);
  a.qsl = reinterpret_cast<const int32_t*>(Q.data);
  a.idx = reinterpret_cast<const int32_t*>(I.data); a.idx_rs = I.stride[0]; a.cols = (int32_t)cols;
  a.accepted = reinterpret_cast<const int32_t*>(AC.data);
  a.state = S.data; a.slot_stride = S.stride[0]; a.num_slots = (int32_t)S.shape[0];
  a.out_gate = OG.data; a.og_rs = OG.stride[0]; a.og_hs = OG.stride[1];
  a.norm_w = reinterpret_cast<const float*>(NW.data);
  a.out = O.data; a.o_rs = H * kD;
  a.N = (int32_t)N; a.R = (int32_t)R; a.H = (int32_t)H;
  a.gate_mode = has_lower_bound ? kda::KDA_GATE_LOWER_BOUND : kda::KDA_GATE_SOFTPLUS;
  a.lower_bound = lower_bound; a.norm_eps = norm_eps;
  a.scale = 0.08838834764831845f;  // 1/sqrt(128)
  return check_launch(kda::launch_packed_fused(a, S.dtype, cluster, dev.sms, st));
}

}  // extern "C"

namespace {

// Shared by kda_spec_decode and kda_spec_verify_decode.  corr / kg are
// validated only in verify mode (either may be null there).
kda_status spec_common(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                       const kda_tensor* beta, int32_t beta_is_logit, const kda_tensor* cu_seqlens, int32_t t_max,
                       const kda_tensor* state_indices, const kda_tensor* state, const kda_tensor* out,
                       const kda_tensor* correction_cache, const kda_tensor* kg_cache, bool verify, float scale,
                       void* stream) {
  View Q, K, V, Gt, Bt, CU, I, S, O, CC, KG;
  KDA_TRY(ranked_view(q, "q", 3, -1, &Q));
  KDA_TRY(ranked_view(k, "k", 3, -1, &K));
  KDA_TRY(ranked_view(v, "v", 3, -1, &V));
  KDA_TRY(ranked_view(g, "g", 3, -1, &Gt));
  KDA_TRY(ranked_view(beta, "beta", 2, -1, &Bt));
  KDA_TRY(raw_view(cu_seqlens, "cu_seqlens", &CU));
  KDA_TRY(raw_view(state_indices, "state_indices", &I));
  KDA_TRY(raw_view(state, "state", &S));
  KDA_TRY(ranked_view(out, "out", 3, -1, &O));
  const int64_t R = Q.shape[0], H = Q.shape[1];
  KDA_CHECK(H >= 1, KDA_ERR_INVALID_ARG, "q: need at least one head");
  KDA_CHECK(R <= INT32_MAX, KDA_ERR_INVALID_ARG, "q: too many token rows");
  KDA_TRY(need_dtype(Q, KDA_F32, KDA_BF16));
  KDA_TRY(need_shape(Q, 2, kD));
  for (View* t : {&K, &V}) {
    KDA_CHECK(t->dtype == Q.dtype, KDA_ERR_INVALID_ARG, "%s: dtype must match q", t->name);
    KDA_TRY(need_shape(*t, 0, R));
    KDA_TRY(need_shape(*t, 1, H));
    KDA_TRY(need_shape(*t, 2, kD));
  }
  KDA_TRY(need_dtype(Gt, KDA_F32));
  KDA_TRY(need_shape(Gt, 0, R));
  KDA_TRY(need_shape(Gt, 1, H));
  KDA_TRY(need_shape(Gt, 2, kD));
  for (View* t : {&Q, &K, &V, &Gt}) KDA_TRY(need_vec_layout(*t));
  KDA_TRY(need_dtype(Bt, KDA_F32, KDA_BF16));
  KDA_TRY(need_shape(Bt, 0, R));
  KDA_TRY(need_shape(Bt, 1, H));
  KDA_CHECK(beta_is_logit == 0 || beta_is_logit == 1, KDA_ERR_INVALID_ARG, "beta_is_logit must be 0 or 1");
  KDA_CHECK(CU.ndim == 1 && CU.shape[0] >= 1, KDA_ERR_INVALID_ARG, "cu_seqlens: expected rank 1 with N+1 >= 1 entries");
  const int64_t N = CU.shape[0] - 1;
  KDA_TRY(need_indices(CU, N + 1));
  KDA_TRY(need_indices(I, N));
  KDA_CHECK(t_max >= 1, KDA_ERR_INVALID_ARG, "t_max must be >= 1");
  KDA_TRY(need_state_layout(S, H));
  KDA_TRY(need_out(O));
  KDA_TRY(need_shape(O, 0, R));
  KDA_TRY(need_shape(O, 1, H));
  KDA_TRY(need_shape(O, 2, kD));
  KDA_CHECK(std::isfinite(scale) && scale > 0.f, KDA_ERR_INVALID_ARG, "scale must be finite and positive");
  KDA_TRY(no_alias(O, {&Q, &K, &V, &Gt, &Bt, &CU, &I, &S}));
  int64_t t_cap = 0;
  if (verify) {
    KDA_CHECK(t_max <= 16, KDA_ERR_UNSUPPORTED, "verify mode serves up to 16 tokens per row (t_max %d)", t_max);
    for (const kda_tensor* c : {correction_cache, kg_cache}) {
      if (c == nullptr) continue;
      View* w = c == correction_cache ? &CC : &KG;
      KDA_TRY(raw_view(c, c == correction_cache ? "correction_cache" : "kg_cache", w));
      KDA_TRY(need_dtype(*w, KDA_F32));
      KDA_CHECK(w->ndim == 4, KDA_ERR_INVALID_ARG, "%s: expected rank 4", w->name);
      KDA_TRY(need_shape(*w, 0, S.shape[0]));
      KDA_TRY(need_shape(*w, 1, H));
      KDA_TRY(need_shape(*w, 3, c == correction_cache ? kD : 2 * kD));
      KDA_CHECK(w->shape[2] >= 1 && w->shape[2] <= 16, KDA_ERR_INVALID_ARG, "%s: token capacity %lld not in 1..16",
                w->name, (long long)w->shape[2]);
      KDA_CHECK(t_cap == 0 || w->shape[2] == t_cap, KDA_ERR_INVALID_ARG, "caches disagree on the token capacity");
      t_cap = w->shape[2];
      KDA_TRY(need_contiguous(*w));
      KDA_CHECK(reinterpret_cast<uintptr_t>(w->data) % 16 == 0, KDA_ERR_INVALID_ARG, "%s: data must be 16-byte aligned",
                w->name);
      KDA_TRY(no_alias(*w, {&Q, &K, &V, &Gt, &Bt, &CU, &I, &S, &O}));
    }
    if (correction_cache != nullptr && kg_cache != nullptr) KDA_TRY(no_alias(CC, {&KG}));
  } else {
    KDA_TRY(no_alias(S, {&Q, &K, &V, &Gt, &Bt, &CU, &I}));
  }
  if (R == 0) return KDA_OK;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  int sched = plan_schedule(KDA_OP_SPEC, N * H, S.dtype, t_max, dev.sms);
  if (sched == KDA_SCHED_MMA && S.dtype != KDA_BF16) {
    KDA_CHECK(g_schedule_override.load() != KDA_SCHED_MMA, KDA_ERR_UNSUPPORTED,
              "the tensor-core (MMA) schedule takes a bfloat16 state pool");
    sched = KDA_SCHED_SPLIT;
  }
  const int split = plan_split(KDA_OP_SPEC, N * H, S.dtype, t_max, dev.sms);
  KDA_CHECK(kda::split_supported(split), KDA_ERR_INVALID_ARG, "split %d has no kernel", split);
  KDA_TRY(check_grid((N + 1) * H * split));

  kda::SpecArgs a{};
  a.q = Q.data; a.k = K.data; a.v = V.data;
  a.q_rs = Q.stride[0]; a.q_hs = Q.stride[1];
  a.k_rs = K.stride[0]; a.k_hs = K.stride[1];
  a.v_rs = V.stride[0]; a.v_hs = V.stride[1];
  a.qkv_dtype = Q.dtype;
  a.g = reinterpret_cast<const float*>(Gt.data); a.g_rs = Gt.stride[0]; a.g_hs = Gt.stride[1];
  a.beta = Bt.data; a.b_rs = Bt.stride[0]; a.b_hs = Bt.stride[1];
  a.beta_dtype = Bt.dtype; a.beta_is_logit = beta_is_logit;
  a.cu = reinterpret_cast<const int32_t*>(CU.data);
  a.idx = reinterpret_cast<const int32_t*>(I.data);
  a.state = S.data; a.slot_stride = S.stride[0]; a.num_slots = (int32_t)S.shape[0];
  a.out = O.data; a.N = (int32_t)N; a.R = (int32_t)R; a.H = (int32_t)H;
  a.scale = scale;
  a.corr = verify && correction_cache != nullptr ? reinterpret_cast<float*>(CC.data) : nullptr;
  a.kg = verify && kg_cache != nullptr ? reinterpret_cast<float*>(KG.data) : nullptr;
  a.t_cap = (int32_t)t_cap;
  if (sched == KDA_SCHED_MMA) return check_launch(kda::launch_spec_mma(a, verify, dev.sms, st));
  return check_launch(kda::launch_spec(a, S.dtype, split, verify, st));
}

}  // namespace

extern "C" {

kda_status kda_spec_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v, const kda_tensor* g,
                           const kda_tensor* beta, int32_t beta_is_logit, const kda_tensor* cu_seqlens,
                           int32_t t_max, const kda_tensor* state_indices, const kda_tensor* state,
                           const kda_tensor* out, float scale, void* stream) {
  return spec_common(q, k, v, g, beta, beta_is_logit, cu_seqlens, t_max, state_indices, state, out, nullptr,
                     nullptr, false, scale, stream);
}

kda_status kda_spec_verify_decode(const kda_tensor* q, const kda_tensor* k, const kda_tensor* v,
                                  const kda_tensor* g, const kda_tensor* beta, int32_t beta_is_logit,
                                  const kda_tensor* cu_seqlens, int32_t t_max, const kda_tensor* state_indices,
                                  const kda_tensor* state, const kda_tensor* out,
                                  const kda_tensor* correction_cache, const kda_tensor* kg_cache, float scale,
                                  void* stream) {
  return spec_common(q, k, v, g, beta, beta_is_logit, cu_seqlens, t_max, state_indices, state, out,
                     correction_cache, kg_cache, true, scale, stream);
}

int32_t kda_plan_split(int32_t op, int64_t units, int32_t state_dtype, int32_t t_max, int32_t sm_count) {
  if (op < KDA_OP_RECURRENT || op > KDA_OP_PACKED_FUSED || units < 0 || sm_count < 1 || t_max < 1) return 0;
  if (state_dtype != KDA_F32 && state_dtype != KDA_BF16) return 0;
  return plan_split(op, units, state_dtype, t_max, sm_count);
}

int32_t kda_plan_schedule(int32_t op, int64_t units, int32_t state_dtype, int32_t t_max, int32_t sm_count) {
  if (op < KDA_OP_RECURRENT || op > KDA_OP_PACKED_FUSED || units < 0 || sm_count < 1 || t_max < 1) return 0;
  if (state_dtype != KDA_F32 && state_dtype != KDA_BF16) return 0;
  return plan_schedule(op, units, state_dtype, t_max, sm_count);
}

kda_status kda_set_schedule_override(int32_t schedule) {
  KDA_CHECK(schedule == KDA_SCHED_AUTO || schedule == KDA_SCHED_SPLIT || schedule == KDA_SCHED_STREAM ||
                schedule == KDA_SCHED_MMA,
            KDA_ERR_INVALID_ARG, "unknown schedule %d", schedule);
  g_schedule_override.store(schedule);
  return KDA_OK;
}

kda_status kda_device_error(uint32_t* flags, int32_t clear) {
  KDA_CHECK(flags != nullptr, KDA_ERR_INVALID_ARG, "flags: null pointer");
  unsigned int f = 0, fm = 0;
  cudaError_t e = kda::read_device_error(&f, clear != 0);
  if (e == cudaSuccess) e = kda::read_mma_error(&fm, clear != 0);
  KDA_CHECK(e == cudaSuccess, KDA_ERR_CUDA, "reading the device error word: %s", cudaGetErrorString(e));
  *flags = f | fm;
  return KDA_OK;
}

kda_status kda_selftest_wait_timeout(void* stream) {
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DeviceInfo dev;
  KDA_TRY(current_device(st, &dev));
  return check_launch(kda::launch_selftest_wait(st));
}

kda_status kda_set_split_override(int32_t split) {
  KDA_CHECK(split == 0 || kda::split_supported(split), KDA_ERR_INVALID_ARG, "split %d has no kernel", split);
  g_split_override.store(split);
  return KDA_OK;
}

const char* kda_status_string(kda_status s) {
  switch (s) {
    case KDA_OK: return "KDA_OK";
    case KDA_ERR_INVALID_ARG: return "KDA_ERR_INVALID_ARG";
    case KDA_ERR_UNSUPPORTED: return "KDA_ERR_UNSUPPORTED";
    case KDA_ERR_ALIAS: return "KDA_ERR_ALIAS";
    case KDA_ERR_CUDA: return "KDA_ERR_CUDA";
    default: return "KDA_ERR_UNKNOWN";
  }
}

const char* kda_last_error_message(void) { return g_last_error.c_str(); }

const char* kda_version(void) { return "libkda 0.1.0 (sm_103a)"; }

}  // extern "C"
