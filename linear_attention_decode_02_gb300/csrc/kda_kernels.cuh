// KDA decode kernels for sm_103a.
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

// =====================================================================================
// T=1: one CTA per (row, head, split); NW warps x CW columns = 128/split columns.
// =====================================================================================
template <typename StateT, int CW, int NW>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW>::value) kda_t1_kernel(const T1Args a) {
  using G = Strip<StateT, CW>;
  constexpr int SPLIT = kD / (CW * NW);
  static_assert(SPLIT * CW * NW == kD, "split must tile the 128 value columns");
  __shared__ float4 s_coef[NW][kD];

  const int split = blockIdx.x % SPLIT;
  const int unit = blockIdx.x / SPLIT;
  const int h = unit % a.H;
  const int b = unit / a.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int col0 = (split * NW + warp) * CW + (lane % G::LPR) * G::VEC;
  const int row0 = lane / G::LPR;
  const int c4 = lane * 4;

  // Activation loads first: they do not depend on the slot.
  const float4 q = load4(a.q, (int64_t)b * a.q_rs + (int64_t)h * a.q_hs + c4, a.qkv_dtype);
  const float4 k = load4(a.k, (int64_t)b * a.k_rs + (int64_t)h * a.k_hs + c4, a.qkv_dtype);
  const float4 gr = load4(a.gate, (int64_t)b * a.g_rs + (int64_t)h * a.g_hs + c4, a.gate_dtype);
  const float4 dtb = __ldg(reinterpret_cast<const float4*>(a.dt_bias + h * kD + c4));
  const float A = expf(__ldg(a.A_log + h));
  const float braw = load1(a.beta, (int64_t)b * a.b_rs + (int64_t)h * a.b_hs, a.beta_dtype);
  float vv[G::VEC];
  load_cols<G::VEC>(a.v, (int64_t)b * a.v_rs + (int64_t)h * a.v_hs + col0, a.qkv_dtype, vv);

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)b * a.H + h) * kD;
  const int slot = __ldg(a.idx + b);
  if (slot <= 0 || slot >= a.num_slots) {  // null row: zero output, no cache access
    if (row0 == 0) store_out_zero<G::VEC>(out + col0);
    return;
  }

  StateT* sp = static_cast<StateT*>(a.state) + (int64_t)slot * a.slot_stride + (int64_t)h * kD * kD;
  RawRegs<StateT, G> S;
  strip_load<StateT, G>(sp, row0, col0, S);

  float4 d;
  d.x = expf(log_decay(gr.x + dtb.x, A, a.gate_mode, a.lower_bound));
  d.y = expf(log_decay(gr.y + dtb.y, A, a.gate_mode, a.lower_bound));
  d.z = expf(log_decay(gr.z + dtb.z, A, a.gate_mode, a.lower_bound));
  d.w = expf(log_decay(gr.w + dtb.w, A, a.gate_mode, a.lower_bound));
  float4* coef = s_coef[warp];
  const float qk = token_coefficients(q, k, d, lane, coef);
  const float beta = sigmoidf_(braw);
  __syncwarp();

  float acc_a[G::VEC], acc_b[G::VEC];
  strip_reduce<G>(S, coef, row0, acc_a, acc_b);
  float u[G::VEC], o[G::VEC];
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) {
    u[j] = beta * (vv[j] - acc_a[j]);
    o[j] = a.scale * (acc_b[j] + qk * u[j]);
  }
  strip_update_store<StateT, G>(sp, row0, col0, S, coef, u);
  if (row0 == 0) store_out<G::VEC>(out + col0, o);
}

// =====================================================================================
// Fused conv + SiLU + KDA + gated RMSNorm: one CTA of 8 warps per (row, head).
// =====================================================================================
template <typename StateT>
__global__ void __launch_bounds__(256, 2) kda_fused_kernel(const FusedArgs a) {
  constexpr int CW = 16, NW = 8, NT = NW * 32;
  using G = Strip<StateT, CW>;
  static_assert(CW * NW == kD, "one CTA covers all value columns");
  __shared__ float s_a[3 * kD];  // SiLU(conv) of this head's q | k | v channels
  __shared__ float s_d[kD];      // decay exp(g)
  __shared__ float4 s_coef[NW][kD];
  __shared__ float s_ss[NW];

  const int unit = blockIdx.x;
  const int h = unit % a.H;
  const int r = unit / a.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = warp * CW + (lane % G::LPR) * G::VEC;
  const int row0 = lane / G::LPR;

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)r * a.H + h) * kD;
  const int slot = __ldg(a.idx + r);
  if (slot <= 0 || slot >= a.num_slots) {  // null row: zero output, neither cache touched
    if (row0 == 0) store_out_zero<G::VEC>(out + col0);
    return;
  }

  StateT* sp = static_cast<StateT*>(a.state) + (int64_t)slot * a.slot_stride + (int64_t)h * kD * kD;
  RawRegs<StateT, G> S;
  strip_load<StateT, G>(sp, row0, col0, S);

  // Short conv over [cache0, cache1, cache2, x] (oldest first) for the 384
  // channels of this head, then the cache shift.  Each channel is read and
  // written by the same thread; heads own disjoint channels.
  const int HD = a.H * kD;
  const __nv_bfloat16* xr = static_cast<const __nv_bfloat16*>(a.x) + (int64_t)r * a.x_rs;
  __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state) + (int64_t)slot * a.cs_slot_stride;
  for (int lc = tid; lc < 3 * kD; lc += NT) {
    const int sec = lc >> 7;
    const int ch = sec * HD + h * kD + (lc & (kD - 1));
    const __nv_bfloat16 xb = xr[ch];
    __nv_bfloat16* cp = cs + ch;
    const __nv_bfloat16 c0 = cp[0];
    const __nv_bfloat16 c1 = cp[a.cs_tap_stride];
    const __nv_bfloat16 c2 = cp[2 * a.cs_tap_stride];
    const float* w = a.conv_w + (int64_t)sec * 4 * HD + h * kD + (lc & (kD - 1));
    float y = __ldg(w) * __bfloat162float(c0);
    y = fmaf(__ldg(w + HD), __bfloat162float(c1), y);
    y = fmaf(__ldg(w + 2 * HD), __bfloat162float(c2), y);
    y = fmaf(__ldg(w + 3 * HD), __bfloat162float(xb), y);
    s_a[lc] = y * sigmoidf_(y);
    cp[0] = c1;
    cp[a.cs_tap_stride] = c2;
    cp[2 * a.cs_tap_stride] = xb;
  }
  if (tid < kD) {
    const float A = expf(__ldg(a.A_log + h));
    const float x = __bfloat162float(static_cast<const __nv_bfloat16*>(a.gate)[(int64_t)r * a.g_rs +
                                                                                (int64_t)h * a.g_hs + tid]) +
                    __ldg(a.dt_bias + h * kD + tid);
    s_d[tid] = expf(log_decay(x, A, a.gate_mode, a.lower_bound));
  }
  const float beta = sigmoidf_(
      __bfloat162float(static_cast<const __nv_bfloat16*>(a.beta)[(int64_t)r * a.b_rs + (int64_t)h * a.b_hs]));
  // Epilogue operands, loaded early.
  float nw[G::VEC], og[G::VEC];
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) nw[j] = __ldg(a.norm_w + col0 + j);
  load_cols<G::VEC>(a.out_gate, (int64_t)r * a.og_rs + (int64_t)h * a.og_hs + col0, KDA_DT_BF16, og);
  __syncthreads();

  const float4 q = *reinterpret_cast<const float4*>(s_a + 4 * lane);
  const float4 k = *reinterpret_cast<const float4*>(s_a + kD + 4 * lane);
  const float4 d = *reinterpret_cast<const float4*>(s_d + 4 * lane);
  float4* coef = s_coef[warp];
  const float qk = token_coefficients(q, k, d, lane, coef);
  float vv[G::VEC];
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) vv[j] = s_a[2 * kD + col0 + j];
  __syncwarp();

  float acc_a[G::VEC], acc_b[G::VEC];
  strip_reduce<G>(S, coef, row0, acc_a, acc_b);
  float u[G::VEC], o[G::VEC];
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) {
    u[j] = beta * (vv[j] - acc_a[j]);
    o[j] = a.scale * (acc_b[j] + qk * u[j]);
    ss = fmaf(o[j], o[j], ss);
  }
  strip_update_store<StateT, G>(sp, row0, col0, S, coef, u);

  // Gated RMSNorm over the 128 value columns: lanes with row0 == 0 hold
  // distinct columns; one barrier to combine the 8 warps.
  ss = warp_sum(row0 == 0 ? ss : 0.f);
  if (lane == 0) s_ss[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) tot += s_ss[w];
  const float rinv = rsqrtf(tot * (1.f / kD) + a.norm_eps);
  if (row0 == 0) {
    float y[G::VEC];
#pragma unroll
    for (int j = 0; j < G::VEC; ++j) y[j] = o[j] * rinv * nw[j] * sigmoidf_(og[j]);
    store_out<G::VEC>(out + col0, y);
  }
}

// =====================================================================================
// Speculative T >= 1: one CTA per (row, head, split); the state stays in
// float32 registers across the row's tokens.  Tokens are staged TC at a
// time.  Within a chunk the decay is deferred: with P_t the cumulative decay
// of each key row since the chunk start, the registers hold S~ = S / P_t, so
// the reductions use (P_t k, P_t q) and the update is one paired FMA,
// S~ += (k / P_t) u^T; the true state P_end S~ is restored at chunk end.  A
// chunk ends early once the sum over its tokens of the largest per-row decay
// exceeds e^-80, keeping P_t and 1/P_t finite in float32 (per-element log
// decays are clamped at -60: anything decayed further is below float32
// resolution of the rest of the row).
// Grid slice n == N zeroes the padding token rows outside [cu[0], cu[N]).
// VERIFY: the state is read-only (never stored); token position t < t_cap of
// a live row records its correction u_t and its raw key | log decay in the
// optional slot-indexed caches.
// =====================================================================================
constexpr float kSpecMaxLogDecay = 80.f;   // chunk bound on the summed per-token decay
constexpr float kSpecLogDecayFloor = -60.f;

template <typename StateT, int CW, int NW, bool VERIFY>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW>::value) kda_spec_kernel(const SpecArgs a) {
  using G = Strip<StateT, CW>;
  constexpr int SPLIT = kD / (CW * NW);
  constexpr int TC = 8;
  constexpr int NT = NW * 32;
  static_assert(SPLIT * CW * NW == kD, "split must tile the 128 value columns");
  __shared__ float4 s_coef[TC][kD];  // staged (q, k, g), then (P k, P q, k / P, k / P)
  __shared__ float4 s_tok[TC];       // (beta, q.k, largest per-row decay, -)
  __shared__ float s_P[kD];          // P at the chunk end, per key row
  __shared__ __align__(16) float s_v[TC][kD];  // the chunk's value vectors

  const int split = blockIdx.x % SPLIT;
  const int unit = blockIdx.x / SPLIT;
  const int h = unit % a.H;
  const int n = unit / a.H;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int col0 = (split * NW + warp) * CW + (lane % G::LPR) * G::VEC;
  const int row0 = lane / G::LPR;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)h * kD + col0;
  const int64_t out_rs = (int64_t)a.H * kD;

  if (n == a.N) {  // padding token rows
    const int lo = min(max(__ldg(a.cu), 0), a.R);
    const int hi = max(min(__ldg(a.cu + a.N), a.R), lo);
    for (int t = row0; t < lo; t += G::RPI) store_out_zero<G::VEC>(out + t * out_rs);
    for (int t = hi + row0; t < a.R; t += G::RPI) store_out_zero<G::VEC>(out + t * out_rs);
    return;
  }

  const int t0 = max(__ldg(a.cu + n), 0);
  const int t1 = min(__ldg(a.cu + n + 1), a.R);
  if (t1 <= t0) return;  // empty row
  const int slot = __ldg(a.idx + n);
  if (slot <= 0 || slot >= a.num_slots) {  // null row: zero its token rows
    for (int t = t0 + row0; t < t1; t += G::RPI) store_out_zero<G::VEC>(out + t * out_rs);
    return;
  }

  StateT* sp = static_cast<StateT*>(a.state) + (int64_t)slot * a.slot_stride + (int64_t)h * kD * kD;
  FltRegs<G> S;
  strip_load<StateT, G>(sp, row0, col0, S);

  for (int tc0 = t0; tc0 < t1;) {
    const int nt = min(TC, t1 - tc0);
    if (tc0 != t0) __syncthreads();  // previous chunk fully consumed
    // per-token prologue, one token per warp: normalised q, k and the log decay
    for (int j = warp; j < nt; j += NW) {
      const int t = tc0 + j;
      const float4 q = load4(a.q, (int64_t)t * a.q_rs + (int64_t)h * a.q_hs + 4 * lane, a.qkv_dtype);
      const float4 k = load4(a.k, (int64_t)t * a.k_rs + (int64_t)h * a.k_hs + 4 * lane, a.qkv_dtype);
      reinterpret_cast<float4*>(s_v[j])[lane] =
          load4(a.v, (int64_t)t * a.v_rs + (int64_t)h * a.v_hs + 4 * lane, a.qkv_dtype);
      float4 g = __ldg(reinterpret_cast<const float4*>(a.g + (int64_t)t * a.g_rs + (int64_t)h * a.g_hs + 4 * lane));
      if (VERIFY && a.kg != nullptr && split == 0 && t - t0 < a.t_cap) {
        float* kgp = a.kg + (((int64_t)slot * a.H + h) * a.t_cap + (t - t0)) * (2 * kD);
        reinterpret_cast<float4*>(kgp)[lane] = k;
        reinterpret_cast<float4*>(kgp + kD)[lane] = g;
      }
      g = make_float4(fmaxf(g.x, kSpecLogDecayFloor), fmaxf(g.y, kSpecLogDecayFloor),
                      fmaxf(g.z, kSpecLogDecayFloor), fmaxf(g.w, kSpecLogDecayFloor));
      float qq = q.x * q.x + q.y * q.y + q.z * q.z + q.w * q.w;
      float kk = k.x * k.x + k.y * k.y + k.z * k.z + k.w * k.w;
      float qk = q.x * k.x + q.y * k.y + q.z * k.z + q.w * k.w;
      float gm = fmaxf(fmaxf(-g.x, -g.y), fmaxf(-g.z, -g.w));
      qq = warp_sum(qq);
      kk = warp_sum(kk);
      qk = warp_sum(qk);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(0xffffffffu, gm, o));
      const float rq = rsqrtf(qq + kL2Eps), rk = rsqrtf(kk + kL2Eps);
#pragma unroll
      for (int i = 0; i < 4; ++i)
        s_coef[j][4 * lane + i] = make_float4(f4get(q, i) * rq, f4get(k, i) * rk, f4get(g, i), 0.f);
      if (lane == 0) {
        const float braw = load1(a.beta, (int64_t)t * a.b_rs + (int64_t)h * a.b_hs, a.beta_dtype);
        s_tok[j] = make_float4(a.beta_is_logit ? sigmoidf_(braw) : braw, qk * rq * rk, gm, 0.f);
      }
    }
    __syncthreads();
    // tokens of this chunk: the longest prefix whose summed decay stays within the bound
    int ne = 1;
    {
      float acc = s_tok[0].z;
      for (int j = 1; j < nt; ++j) {
        acc += s_tok[j].z;
        if (acc > kSpecMaxLogDecay) break;
        ne = j + 1;
      }
    }
    // cumulative decay per key row -> deferred-decay coefficients
    for (int r = threadIdx.x; r < kD; r += NT) {
      float Gs = 0.f, P = 1.f;
      for (int j = 0; j < ne; ++j) {
        const float4 c = s_coef[j][r];  // (q, k, g, -)
        Gs += c.z;
        P = expf(Gs);
        const float ku = c.y * expf(-Gs);
        s_coef[j][r] = make_float4(P * c.y, P * c.x, ku, ku);
      }
      s_P[r] = P;
    }
    __syncthreads();
    for (int j = 0; j < ne; ++j) {
      const int t = tc0 + j;
      float vv[G::VEC];
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) vv[jj] = s_v[j][col0 + jj];
      const float4 tk = s_tok[j];
      float acc_a[G::VEC], acc_b[G::VEC];
      strip_reduce<G>(S, s_coef[j], row0, acc_a, acc_b);
      float u[G::VEC], o[G::VEC];
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) {
        u[jj] = tk.x * (vv[jj] - acc_a[jj]);
        o[jj] = a.scale * (acc_b[jj] + tk.y * u[jj]);
      }
      if (VERIFY && a.corr != nullptr && row0 == 0 && t - t0 < a.t_cap) {
        float* cp = a.corr + (((int64_t)slot * a.H + h) * a.t_cap + (t - t0)) * kD + col0;
#pragma unroll
        for (int jj = 0; jj < G::VEC; jj += 4)
          *reinterpret_cast<float4*>(cp + jj) = make_float4(u[jj], u[jj + 1], u[jj + 2], u[jj + 3]);
      }
      // S~ += (k / P_t) u^T
      float2 u2[G::VEC / 2];
      pairs_of<G::VEC>(u, u2);
#pragma unroll
      for (int i = 0; i < G::PASSES; ++i) {
        const float4 c = s_coef[j][row0 + i * G::RPI];
        const float2 ku = make_float2(c.z, c.w);
#pragma unroll
        for (int p = 0; p < G::VEC / 2; ++p) S.s[i][p] = fma2(ku, u2[p], S.s[i][p]);
      }
      if (row0 == 0) store_out<G::VEC>(out + t * out_rs, o);
    }
    // restore the true state: S = P_end S~
#pragma unroll
    for (int i = 0; i < G::PASSES; ++i) {
      const float2 pp = dup2(s_P[row0 + i * G::RPI]);
#pragma unroll
      for (int p = 0; p < G::VEC / 2; ++p) S.s[i][p] = mul2(pp, S.s[i][p]);
    }
    tc0 += ne;
  }
  if (!VERIFY) strip_store<StateT, G>(sp, row0, col0, S);
}

}  // namespace kda
