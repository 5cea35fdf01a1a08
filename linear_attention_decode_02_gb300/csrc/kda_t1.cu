// T=1 recurrent / packed decode: kernel instantiations and launcher.
#include "kda_kernels.cuh"

namespace kda {

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
  pdl_wait();
  pdl_launch_dependents();

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

namespace {

template <typename StateT, int CW, int NW>
cudaError_t launch_t1_variant(const T1Args& a, cudaStream_t s) {
  constexpr int SPLIT = kD / (CW * NW);
  const int64_t blocks = (int64_t)a.B * a.H * SPLIT;
  return launch_pdl(kda_t1_kernel<StateT, CW, NW>, dim3((unsigned)blocks), dim3(NW * 32), 0, s, 1, a);
}

template <typename StateT>
cudaError_t launch_t1_typed(const T1Args& a, int split, cudaStream_t s) {
  switch (split) {
    case 1: return launch_t1_variant<StateT, 16, 8>(a, s);
    case 2: return launch_t1_variant<StateT, 16, 4>(a, s);
    case 4: return launch_t1_variant<StateT, 16, 2>(a, s);
    case 8: return launch_t1_variant<StateT, 16, 1>(a, s);
    case 16: return launch_t1_variant<StateT, 8, 1>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

bool split_supported(int split) {
  return split == 1 || split == 2 || split == 4 || split == 8 || split == 16;
}

cudaError_t launch_t1(const T1Args& a, int state_dtype, int split, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_t1_typed<float>(a, split, s);
  return launch_t1_typed<__nv_bfloat16>(a, split, s);
}

}  // namespace kda
