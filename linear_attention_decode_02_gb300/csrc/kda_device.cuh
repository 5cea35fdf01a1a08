// Device helpers shared by the KDA decode kernels: 16-byte state fragments,
// bf16 packing, activation loads, warp reductions and the gate transforms.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda_launch.h"

namespace kda {

constexpr int kD = 128;           // head dimension K = V = 128
constexpr float kL2Eps = 1e-6f;   // QK L2 normalisation epsilon

// ---- programmatic dependent launch ------------------------------------------------

// Returns once the previous kernel on the stream has completed and its memory
// operations are visible (immediately when the grid was launched without
// programmatic serialization).  Every kernel calls it before its first
// global-memory access; only launch and on-chip set-up overlap the previous
// kernel.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel on the stream begin its own launch and set-up.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---- bf16 <-> f32 ---------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two floats -> two bf16 (round to nearest even), low half = a.
__device__ __forceinline__ uint32_t pack_bf2(float a, float b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

// ---- state fragments: one 16-byte vector of a state row ------------------------
// Raw is the register image of the 16 bytes as stored; get() reads element j
// as float; pack() builds a Raw from VEC floats (bf16: round to nearest even).

template <typename StateT>
struct Frag;

template <>
struct Frag<float> {
  static constexpr int VEC = 4;
  using Raw = float4;
  __device__ __forceinline__ static Raw load(const float* p) {
    return __ldcs(reinterpret_cast<const float4*>(p));
  }
  __device__ __forceinline__ static void store(float* p, const Raw& r) {
    __stcs(reinterpret_cast<float4*>(p), r);
  }
  __device__ __forceinline__ static float get(const Raw& r, int j) {
    return j == 0 ? r.x : (j == 1 ? r.y : (j == 2 ? r.z : r.w));
  }
  __device__ __forceinline__ static Raw pack(const float (&s)[VEC]) {
    return make_float4(s[0], s[1], s[2], s[3]);
  }
  // Column pair p (elements 2p, 2p+1) as float2, and back.
  __device__ __forceinline__ static float2 get2(const Raw& r, int p) {
    return p == 0 ? make_float2(r.x, r.y) : make_float2(r.z, r.w);
  }
  __device__ __forceinline__ static Raw pack2(const float2 (&y)[VEC / 2]) {
    return make_float4(y[0].x, y[0].y, y[1].x, y[1].y);
  }
};

template <>
struct Frag<__nv_bfloat16> {
  static constexpr int VEC = 8;
  using Raw = uint4;
  __device__ __forceinline__ static Raw load(const __nv_bfloat16* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
  }
  __device__ __forceinline__ static void store(__nv_bfloat16* p, const Raw& r) {
    __stcs(reinterpret_cast<uint4*>(p), r);
  }
  __device__ __forceinline__ static float get(const Raw& r, int j) {
    const uint32_t w = (j >> 1) == 0 ? r.x : ((j >> 1) == 1 ? r.y : ((j >> 1) == 2 ? r.z : r.w));
    return (j & 1) ? bf_hi(w) : bf_lo(w);
  }
  __device__ __forceinline__ static Raw pack(const float (&s)[VEC]) {
    return make_uint4(pack_bf2(s[0], s[1]), pack_bf2(s[2], s[3]), pack_bf2(s[4], s[5]),
                      pack_bf2(s[6], s[7]));
  }
  __device__ __forceinline__ static float2 get2(const Raw& r, int p) {
    const uint32_t w = p == 0 ? r.x : (p == 1 ? r.y : (p == 2 ? r.z : r.w));
    return make_float2(bf_lo(w), bf_hi(w));
  }
  __device__ __forceinline__ static Raw pack2(const float2 (&y)[VEC / 2]) {
    return make_uint4(pack_bf2(y[0].x, y[0].y), pack_bf2(y[1].x, y[1].y), pack_bf2(y[2].x, y[2].y),
                      pack_bf2(y[3].x, y[3].y));
  }
};

// Paired float32 arithmetic (one instruction for two lanes' worth of
// columns); every component is rounded exactly like the scalar operation.
__device__ __forceinline__ float2 dup2(float x) { return make_float2(x, x); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }

// Geometry of one warp's column strip: CW value columns x all 128 key rows.
// Lanes walk a row segment with 16-byte vectors; a warp instruction covers
// RPI rows; each lane holds PASSES fragments (4*CW floats).
template <typename StateT, int CW>
struct Strip {
  static constexpr int VEC = Frag<StateT>::VEC;
  static constexpr int LPR = CW / VEC;      // lanes per row segment
  static constexpr int RPI = 32 / LPR;      // rows per warp instruction
  static constexpr int PASSES = kD / RPI;   // fragments per lane
  static_assert(CW % VEC == 0 && LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "bad strip width");
};

// ---- activation loads ----------------------------------------------------------

// Four consecutive elements starting at element `i` of a float32 or bfloat16
// array.  The address must be 16-byte (f32) or 8-byte (bf16) aligned.
__device__ __forceinline__ float4 load4(const void* base, int64_t i, int dtype) {
  if (dtype == KDA_DT_F32) {
    return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(base) + i));
  }
  uint2 u = __ldg(reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(base) + i));
  return make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
}

__device__ __forceinline__ float load1(const void* base, int64_t i, int dtype) {
  if (dtype == KDA_DT_F32) return __ldg(static_cast<const float*>(base) + i);
  return __bfloat162float(__ldg(static_cast<const __nv_bfloat16*>(base) + i));
}

__device__ __forceinline__ float f4get(const float4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

// ---- reductions -----------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// ---- gates ----------------------------------------------------------------------

// Log decay from the pre-gate value x = raw_gate + dt_bias and a = exp(A_log[h]).
//   gate_mode 0 (Kimi-Linear):  g = -a * softplus(x)
//   gate_mode 1 (bounded):      g = lower_bound * sigmoid(a * x)
__device__ __forceinline__ float log_decay(float x, float a, int gate_mode, float lower_bound) {
  if (gate_mode == KDA_GATE_SOFTPLUS) {
    const float sp = fmaxf(x, 0.f) + log1pf(expf(-fabsf(x)));
    return -a * sp;
  }
  return lower_bound / (1.f + expf(-a * x));
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.f / (1.f + expf(-x)); }

// Per-lane prologue of one token for one head: lane l holds channels 4l..4l+3
// of q, k and the decay d = exp(g).  Writes (d*k_hat, d*q_hat, d, k_hat) for
// those channels to coef[] and returns q_hat . k_hat (same on every lane).
__device__ __forceinline__ float token_coefficients(float4 q, float4 k, float4 d, int lane,
                                                    float4* coef) {
  float qq = q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
  float kk = k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w;
  float qk = q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w;
  qq = warp_sum(qq);
  kk = warp_sum(kk);
  qk = warp_sum(qk);
  const float rq = rsqrtf(qq + kL2Eps);
  const float rk = rsqrtf(kk + kL2Eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float kh = f4get(k, j) * rk;
    const float qh = f4get(q, j) * rq;
    const float dj = f4get(d, j);
    coef[4 * lane + j] = make_float4(dj * kh, dj * qh, dj, kh);
  }
  return qk * rq * rk;
}

}  // namespace kda
