// Fused conv + SiLU + KDA + gated RMSNorm decode: kernel instantiations and launcher.
#include <cooperative_groups.h>

#include "kda_kernels.cuh"

namespace cg = cooperative_groups;

namespace kda {

// =====================================================================================
// Fused conv + SiLU + KDA + gated RMSNorm: a cluster of CL = 128 / (16 NW)
// CTAs of NW warps per (row, head); CTA `rank` owns the value columns
// [rank W, rank W + W), W = 16 NW, one 16-column strip per warp.  Every CTA
// convolves the head's q and k channels (all 128 key rows need them) and its
// slab of v; it writes the conv-cache shift of its own slab of each section,
// so every channel of the cache is written once.  With CL > 1:
//  - a split cluster barrier (arrive after the cache history is read, wait
//    before the shifted cache is written) orders every CTA's history reads
//    before any peer's writes, and has every CTA of the cluster running
//    before the distributed-shared-memory exchange below;
//  - the RMSNorm's sums of squares meet through distributed shared memory:
//    each CTA writes its partial into every peer, then one cluster barrier.
// Every CTA of a cluster reads the same slot, so all take the same branches
// and reach each cluster barrier once.
// =====================================================================================
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait;" ::: "memory"); }

template <typename StateT, int NW>
__global__ void __launch_bounds__(NW * 32, 16 / NW) kda_fused_kernel(const FusedArgs a) {
  constexpr int CW = 16, NT = NW * 32, W = NW * CW, CL = kD / W;
  constexpr int NCH = 2 * kD + W;               // conv channels: all of q and k, this slab of v
  constexpr int CPT = (NCH + NT - 1) / NT;      // channels per thread
  using G = Strip<StateT, CW>;
  static_assert(CL * W == kD && (CL == 1 || CL == 2 || CL == 4), "slabs must tile the 128 columns");
  __shared__ float s_a[NCH];     // SiLU(conv): q (128) | k (128) | this slab of v (W)
  __shared__ float s_d[kD];      // decay exp(g)
  __shared__ float4 s_coef[NW][kD];
  __shared__ float s_ss[NW];
  __shared__ float s_part[CL];   // the cluster CTAs' sums of squares

  const int rank = CL == 1 ? 0 : (int)(blockIdx.x % CL);
  const int slab0 = rank * W;
  const int unit = blockIdx.x / CL;
  const int h = unit % a.H;
  const int r = unit / a.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = slab0 + warp * CW + (lane % G::LPR) * G::VEC;  // value column within the head
  const int row0 = lane / G::LPR;
  // Local conv channel lc -> (section, channel within the head's section).
  auto sec_of = [](int lc) { return lc < kD ? 0 : (lc < 2 * kD ? 1 : 2); };
  auto cis_of = [slab0](int lc) { return lc < 2 * kD ? (lc & (kD - 1)) : slab0 + lc - 2 * kD; };

  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)r * a.H + h) * kD;
  pdl_wait();
  pdl_launch_dependents();
  const int slot = __ldg(a.idx + r);

  // Operands that do not depend on the slot are requested before the slot
  // index resolves, so their round trips overlap it: the conv input x and
  // taps of this thread's channels, the gate, beta, and the epilogue's norm
  // weight and output gate.
  const int HD = a.H * kD;
  const __nv_bfloat16* xr = static_cast<const __nv_bfloat16*>(a.x) + (int64_t)r * a.x_rs;
  __nv_bfloat16 xb[CPT];
  float cw[CPT][4];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int lc = tid + i * NT;
    if (lc < NCH) {
      const int sec = sec_of(lc);
      const int ch = sec * HD + h * kD + cis_of(lc);
      xb[i] = xr[ch];
      const float* w = a.conv_w + (int64_t)sec * 4 * HD + h * kD + cis_of(lc);
#pragma unroll
      for (int t = 0; t < 4; ++t) cw[i][t] = __ldg(w + t * HD);
    }
  }
  constexpr int GPT = kD / NT > 0 ? kD / NT : 1;  // gate entries per thread
  const float gA = __ldg(a.A_log + h);
  float graw[GPT];
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    const int e = tid + i * NT;
    graw[i] = e < kD ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.gate)[(int64_t)r * a.g_rs +
                                                                                (int64_t)h * a.g_hs + e]) +
                           __ldg(a.dt_bias + h * kD + e)
                     : 0.f;
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

  // Short conv over [cache0, cache1, cache2, x] (oldest first) of this CTA's
  // channels, then the cache shift of the channels this CTA owns.
  __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state) + (int64_t)slot * a.cs_slot_stride;
  __nv_bfloat16 c1s[CPT], c2s[CPT];
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int lc = tid + i * NT;
    if (lc < NCH) {
      const __nv_bfloat16* cp = cs + sec_of(lc) * HD + h * kD + cis_of(lc);
      const __nv_bfloat16 c0 = cp[0];
      c1s[i] = cp[a.cs_tap_stride];
      c2s[i] = cp[2 * a.cs_tap_stride];
      float y = cw[i][0] * __bfloat162float(c0);
      y = fmaf(cw[i][1], __bfloat162float(c1s[i]), y);
      y = fmaf(cw[i][2], __bfloat162float(c2s[i]), y);
      y = fmaf(cw[i][3], __bfloat162float(xb[i]), y);
      s_a[lc] = y * sigmoidf_(y);
    }
  }
  if constexpr (CL > 1) cluster_arrive();  // this CTA's history reads are done
#pragma unroll
  for (int i = 0; i < GPT; ++i)
    if (tid + i * NT < kD) s_d[tid + i * NT] = expf(log_decay(graw[i], expf(gA), a.gate_mode, a.lower_bound));
  if constexpr (CL > 1) cluster_wait();  // ... and every peer's
#pragma unroll
  for (int i = 0; i < CPT; ++i) {
    const int lc = tid + i * NT;
    const int cis = lc < NCH ? cis_of(lc) : -1;
    if (lc < NCH && cis >= slab0 && cis < slab0 + W) {
      __nv_bfloat16* cp = cs + sec_of(lc) * HD + h * kD + cis;
      cp[0] = c1s[i];
      cp[a.cs_tap_stride] = c2s[i];
      cp[2 * a.cs_tap_stride] = xb[i];
    }
  }
  const float beta = sigmoidf_(braw);
  __syncthreads();

  const float4 q = *reinterpret_cast<const float4*>(s_a + 4 * lane);
  const float4 k = *reinterpret_cast<const float4*>(s_a + kD + 4 * lane);
  const float4 d = *reinterpret_cast<const float4*>(s_d + 4 * lane);
  float4* coef = s_coef[warp];
  const float qk = token_coefficients(q, k, d, lane, coef);
  float vv[G::VEC];
#pragma unroll
  for (int j = 0; j < G::VEC; ++j) vv[j] = s_a[2 * kD + col0 - slab0 + j];
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
  // distinct columns; one barrier combines the warps, then (cluster) the CTAs.
  ss = warp_sum(row0 == 0 ? ss : 0.f);
  if (lane == 0) s_ss[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) tot += s_ss[w];
  if constexpr (CL > 1) {
    if (tid < CL) *cg::this_cluster().map_shared_rank(&s_part[rank], tid) = tot;  // into CTA tid
    cg::this_cluster().sync();  // every CTA's sum has arrived in every CTA
    tot = 0.f;
#pragma unroll
    for (int c = 0; c < CL; ++c) tot += s_part[c];
  }
  const float rinv = rsqrtf(tot * (1.f / kD) + a.norm_eps);
  if (row0 == 0) {
    float y[G::VEC];
#pragma unroll
    for (int j = 0; j < G::VEC; ++j) y[j] = o[j] * rinv * nw[j] * sigmoidf_(og[j]);
    store_out<G::VEC>(out + col0, y);
  }
}

namespace {

template <typename StateT>
cudaError_t launch_fused_typed(const FusedArgs& a, int cluster, cudaStream_t s) {
  const int64_t units = (int64_t)a.rows * a.H;
  switch (cluster) {
    case 1: return launch_pdl(kda_fused_kernel<StateT, 8>, dim3((unsigned)units), dim3(256), 0, s, 1, a);
    case 2: return launch_pdl(kda_fused_kernel<StateT, 4>, dim3((unsigned)(2 * units)), dim3(128), 0, s, 2, a);
    case 4: return launch_pdl(kda_fused_kernel<StateT, 2>, dim3((unsigned)(4 * units)), dim3(64), 0, s, 4, a);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_fused(const FusedArgs& a, int state_dtype, int cluster, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_fused_typed<float>(a, cluster, s);
  return launch_fused_typed<__nv_bfloat16>(a, cluster, s);
}

}  // namespace kda
