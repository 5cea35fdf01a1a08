// Register-strip building blocks of the KDA decode kernels for sm_103a.
//
// Work decomposition.  For one (row, head) unit the value columns of the
// 128 x 128 state S[k][v] update independently:
//
//     a_v = sum_k (d_k k_k) S[k][v]          b_v = sum_k (d_k q_k) S[k][v]
//     u_v = beta (v_v - a_v)                 o_v = scale (b_v + (q.k) u_v)
//     S'[k][v] = d_k S[k][v] + k_k u_v
//
// (q, k L2-normalised, d = exp(g)).  So a CTA owns one unit and a slab of
// 128/split value columns, and each warp owns a strip of CW columns across
// all 128 key rows: the k-reduction is in-thread plus a few xor shuffles, no
// shared-memory reduction and no CTA barrier on the T=1 path.  Every state
// byte is read once into registers with 16-byte streaming loads issued
// before any arithmetic, and written once with 16-byte streaming stores.
// The per-token scalars (norms, gate, beta) are recomputed by every warp
// that needs them from the activations (a few hundred bytes, L2-resident).
#pragma once

#include "kda_device.cuh"

namespace kda {

template <int VEC>
__device__ __forceinline__ void store_out(__nv_bfloat16* p, const float (&o)[VEC]);

template <>
__device__ __forceinline__ void store_out<4>(__nv_bfloat16* p, const float (&o)[4]) {
  *reinterpret_cast<uint2*>(p) = make_uint2(pack_bf2(o[0], o[1]), pack_bf2(o[2], o[3]));
}

template <>
__device__ __forceinline__ void store_out<8>(__nv_bfloat16* p, const float (&o)[8]) {
  *reinterpret_cast<uint4*>(p) = make_uint4(pack_bf2(o[0], o[1]), pack_bf2(o[2], o[3]),
                                            pack_bf2(o[4], o[5]), pack_bf2(o[6], o[7]));
}

template <int VEC>
__device__ __forceinline__ void store_out_zero(__nv_bfloat16* p) {
  float z[VEC];
#pragma unroll
  for (int j = 0; j < VEC; ++j) z[j] = 0.f;
  store_out<VEC>(p, z);
}

// Value-column activations of one lane (VEC consecutive channels).
template <int VEC>
__device__ __forceinline__ void load_cols(const void* base, int64_t i, int dtype, float (&out)[VEC]) {
#pragma unroll
  for (int j = 0; j < VEC; j += 4) {
    const float4 t = load4(base, i + j, dtype);
    out[j] = t.x; out[j + 1] = t.y; out[j + 2] = t.z; out[j + 3] = t.w;
  }
}

// The lane's state fragments in two register forms: Raw keeps the stored
// bytes (T=1: one read, one write, bf16 stays packed); Flt keeps float32
// column pairs across the tokens of a speculative row (one rounding at the
// end).  at2(i, p) is column pair p of fragment i.
template <typename StateT, typename G>
struct RawRegs {
  typename Frag<StateT>::Raw r[G::PASSES];
  __device__ __forceinline__ float2 at2(int i, int p) const { return Frag<StateT>::get2(r[i], p); }
};

template <typename G>
struct FltRegs {
  float2 s[G::PASSES][G::VEC / 2];
  __device__ __forceinline__ float2 at2(int i, int p) const { return s[i][p]; }
};

template <typename StateT, typename G>
__device__ __forceinline__ void strip_load(const StateT* sp, int row0, int col0, RawRegs<StateT, G>& R) {
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) R.r[i] = Frag<StateT>::load(sp + (row0 + i * G::RPI) * kD + col0);
}

template <typename StateT, typename G>
__device__ __forceinline__ void strip_load(const StateT* sp, int row0, int col0, FltRegs<G>& F) {
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    const typename Frag<StateT>::Raw r = Frag<StateT>::load(sp + (row0 + i * G::RPI) * kD + col0);
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) F.s[i][p] = Frag<StateT>::get2(r, p);
  }
}

// Accumulates one fragment row into the column-pair sums:
// a += (d k)_row * S[row][cols], b += (d q)_row * S[row][cols].
template <int NP2>
__device__ __forceinline__ void accumulate_row(const float4& c, const float2* x2, float2 (&acc_a)[NP2],
                                               float2 (&acc_b)[NP2]) {
  const float2 ca = dup2(c.x), cb = dup2(c.y);
#pragma unroll
  for (int p = 0; p < NP2; ++p) {
    acc_a[p] = fma2(ca, x2[p], acc_a[p]);
    acc_b[p] = fma2(cb, x2[p], acc_b[p]);
  }
}

// Completes the column sums across the lanes that share the lane's columns
// (xor over the row-lane bits) and returns them as scalars.
template <typename G>
__device__ __forceinline__ void strip_allreduce(float2 (&acc_a)[G::VEC / 2], float2 (&acc_b)[G::VEC / 2],
                                                float (&a)[G::VEC], float (&b)[G::VEC]) {
#pragma unroll
  for (int o = G::LPR; o < 32; o <<= 1) {
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) {
      acc_a[p] = add2(acc_a[p], make_float2(__shfl_xor_sync(0xffffffffu, acc_a[p].x, o),
                                            __shfl_xor_sync(0xffffffffu, acc_a[p].y, o)));
      acc_b[p] = add2(acc_b[p], make_float2(__shfl_xor_sync(0xffffffffu, acc_b[p].x, o),
                                            __shfl_xor_sync(0xffffffffu, acc_b[p].y, o)));
    }
  }
#pragma unroll
  for (int p = 0; p < G::VEC / 2; ++p) {
    a[2 * p] = acc_a[p].x; a[2 * p + 1] = acc_a[p].y;
    b[2 * p] = acc_b[p].x; b[2 * p + 1] = acc_b[p].y;
  }
}

// k-reduction of one token over the lane's fragments: a_v = sum_k (d k)_k S[k][v],
// b_v = sum_k (d q)_k S[k][v] for the lane's VEC columns.
template <typename G, typename Regs>
__device__ __forceinline__ void strip_reduce(const Regs& S, const float4* coef, int row0, float (&acc_a)[G::VEC],
                                             float (&acc_b)[G::VEC]) {
  float2 a2[G::VEC / 2], b2[G::VEC / 2];
#pragma unroll
  for (int p = 0; p < G::VEC / 2; ++p) { a2[p] = make_float2(0.f, 0.f); b2[p] = make_float2(0.f, 0.f); }
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    float2 x2[G::VEC / 2];
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) x2[p] = S.at2(i, p);
    accumulate_row<G::VEC / 2>(coef[row0 + i * G::RPI], x2, a2, b2);
  }
  strip_allreduce<G>(a2, b2, acc_a, acc_b);
}

// Column pairs of u for the paired update.
template <int VEC>
__device__ __forceinline__ void pairs_of(const float (&u)[VEC], float2 (&u2)[VEC / 2]) {
#pragma unroll
  for (int p = 0; p < VEC / 2; ++p) u2[p] = make_float2(u[2 * p], u[2 * p + 1]);
}

// S'[k][v] = d_k S[k][v] + k_k u_v for one fragment row (decay d, key k).
template <int NP2>
__device__ __forceinline__ void update_row(float d, float k, const float2* x2, const float2 (&u2)[NP2],
                                           float2 (&y2)[NP2]) {
  const float2 dd = dup2(d), kk = dup2(k);
#pragma unroll
  for (int p = 0; p < NP2; ++p) y2[p] = fma2(dd, x2[p], mul2(kk, u2[p]));
}

// S' = d S + k u^T, written straight back (T=1).
template <typename StateT, typename G>
__device__ __forceinline__ void strip_update_store(StateT* sp, int row0, int col0, const RawRegs<StateT, G>& R,
                                                   const float4* coef, const float (&u)[G::VEC]) {
  float2 u2[G::VEC / 2];
  pairs_of<G::VEC>(u, u2);
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    const float4 c = coef[row0 + i * G::RPI];
    float2 x2[G::VEC / 2], y2[G::VEC / 2];
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) x2[p] = R.at2(i, p);
    update_row<G::VEC / 2>(c.z, c.w, x2, u2, y2);
    Frag<StateT>::store(sp + (row0 + i * G::RPI) * kD + col0, Frag<StateT>::pack2(y2));
  }
}

// Same update kept in float registers (speculative token loop).
template <typename G>
__device__ __forceinline__ void strip_update(FltRegs<G>& F, const float4* coef, int row0, const float (&u)[G::VEC]) {
  float2 u2[G::VEC / 2];
  pairs_of<G::VEC>(u, u2);
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    const float4 c = coef[row0 + i * G::RPI];
    update_row<G::VEC / 2>(c.z, c.w, F.s[i], u2, F.s[i]);
  }
}

template <typename StateT, typename G>
__device__ __forceinline__ void strip_store(StateT* sp, int row0, int col0, const FltRegs<G>& F) {
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) Frag<StateT>::store(sp + (row0 + i * G::RPI) * kD + col0, Frag<StateT>::pack2(F.s[i]));
}

// Minimum resident CTAs per SM for a CTA of NW warps: keeps >= 16 warps per
// SM, i.e. at most 128 registers per thread.
template <int NW>
struct MinBlocks {
  static constexpr int value = NW >= 16 ? 1 : 16 / NW;
};

}  // namespace kda
