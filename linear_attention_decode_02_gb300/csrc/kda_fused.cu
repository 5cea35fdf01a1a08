// Fused conv + SiLU + KDA + gated RMSNorm decode: kernel instantiations and launcher.
#include "kda_kernels.cuh"

namespace kda {

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
  pdl_wait();
  pdl_launch_dependents();
  const int slot = __ldg(a.idx + r);

  // Operands that do not depend on the slot are requested before the slot
  // index resolves, so their round trips overlap it: the conv input x and
  // taps of this thread's (at most two) channels, the gate, beta, and the
  // epilogue's norm weight and output gate.
  const int HD = a.H * kD;
  const __nv_bfloat16* xr = static_cast<const __nv_bfloat16*>(a.x) + (int64_t)r * a.x_rs;
  constexpr int CPT = (3 * kD + NT - 1) / NT;  // channels per thread
  __nv_bfloat16 xb[CPT];
  float cw[CPT][4];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int lc = tid + i * NT;
    if (lc < 3 * kD) {
      const int sec = lc >> 7;
      const int ch = sec * HD + h * kD + (lc & (kD - 1));
      xb[i] = xr[ch];
      const float* w = a.conv_w + (int64_t)sec * 4 * HD + h * kD + (lc & (kD - 1));
#pragma unroll
      for (int t = 0; t < 4; ++t) cw[i][t] = __ldg(w + t * HD);
    }
  }
  float graw = 0.f, gA = 0.f;
  if (tid < kD) {
    gA = __ldg(a.A_log + h);
    graw = __bfloat162float(static_cast<const __nv_bfloat16*>(a.gate)[(int64_t)r * a.g_rs +
                                                                     (int64_t)h * a.g_hs + tid]) +
           __ldg(a.dt_bias + h * kD + tid);
  }
  const float braw =
      __bfloat162float(static_cast<const __nv_bfloat16*>(a.beta)[(int64_t)r * a.b_rs + (int64_t)h * a.b_hs]);
  float nw[G::VEC], og[G::VEC];
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) nw[j] = __ldg(a.norm_w + col0 + j);
  load_cols<G::VEC>(a.out_gate, (int64_t)r * a.og_rs + (int64_t)h * a.og_hs + col0, KDA_DT_BF16, og);

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
  __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state) + (int64_t)slot * a.cs_slot_stride;
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int lc = tid + i * NT;
    if (lc < 3 * kD) {
      const int ch = (lc >> 7) * HD + h * kD + (lc & (kD - 1));
      __nv_bfloat16* cp = cs + ch;
      const __nv_bfloat16 c0 = cp[0];
      const __nv_bfloat16 c1 = cp[a.cs_tap_stride];
      const __nv_bfloat16 c2 = cp[2 * a.cs_tap_stride];
      float y = cw[i][0] * __bfloat162float(c0);
      y = fmaf(cw[i][1], __bfloat162float(c1), y);
      y = fmaf(cw[i][2], __bfloat162float(c2), y);
      y = fmaf(cw[i][3], __bfloat162float(xb[i]), y);
      s_a[lc] = y * sigmoidf_(y);
      cp[0] = c1;
      cp[a.cs_tap_stride] = c2;
      cp[2 * a.cs_tap_stride] = xb[i];
    }
  }
  if (tid < kD) s_d[tid] = expf(log_decay(graw, expf(gA), a.gate_mode, a.lower_bound));
  const float beta = sigmoidf_(braw);
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

cudaError_t launch_fused(const FusedArgs& a, int state_dtype, cudaStream_t s) {
  const int64_t blocks = (int64_t)a.rows * a.H;
  if (state_dtype == KDA_DT_F32)
    return launch_pdl(kda_fused_kernel<float>, dim3((unsigned)blocks), dim3(256), 0, s, 1, a);
  return launch_pdl(kda_fused_kernel<__nv_bfloat16>, dim3((unsigned)blocks), dim3(256), 0, s, 1, a);
}

}  // namespace kda
