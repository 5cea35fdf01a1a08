// Packed fused speculative decode (conv + SiLU + KDA + gated RMSNorm over
// T >= 1 token rows per sequence) with per-token checkpoints of both caches.
#include "kda_kernels.cuh"
#include "kda_packed_fused.h"

namespace kda {

// =====================================================================================
// One CTA of 8 warps per (sequence, head); warp w owns value columns
// 16w..16w+15 over all 128 key rows.  The state is loaded once from the
// start slot (the checkpoint of the last accepted token) and carried in
// float32 registers across the sequence's tokens; after each token it is
// stored to that token's checkpoint slot (rounded once if bf16), so a call
// moves one state read plus one state write per token.
//
// Tokens go in chunks of up to TC:
//  A. conv + SiLU of the chunk's tokens for this head's 384 channels (each
//     thread carries the raw history of its channels in registers and writes
//     the per-token conv checkpoints), decays and betas;
//  B. warp j normalises q, k of token j and writes its per-row coefficients;
//  C. every warp runs the chunk's tokens on its strip with no CTA barrier:
//     reduction, update, checkpoint store, raw output and its sum of squares;
//  D. warp j applies the gated RMSNorm to token j and writes the output row.
// Grid slice n == N zeroes the padding token rows outside [qsl[0], qsl[N]).
// =====================================================================================
template <typename StateT>
__global__ void __launch_bounds__(256, 2) kda_packed_fused_kernel(const PackedFusedArgs a) {
  constexpr int CW = 16, NW = 8, NT = NW * 32, TC = 8, NCH = 3 * kD;
  using G = Strip<StateT, CW>;
  static_assert(CW * NW == kD, "one CTA covers all value columns");
  static_assert(TC <= NW, "phases B and D give each token of a chunk one warp");
  __shared__ __align__(16) float s_act[TC][NCH];  // SiLU(conv): q | k | v channels of this head
  __shared__ __align__(16) float s_d[TC][kD];     // decay exp(g)
  __shared__ float4 s_coef[TC][kD];               // (d k_hat, d q_hat, d, k_hat) per key row
  __shared__ float2 s_tok[TC];                    // (beta, q_hat . k_hat)
  __shared__ int s_slot[TC];                      // checkpoint slot, 0 = none
  __shared__ __align__(16) float s_o[TC][kD];     // raw outputs
  __shared__ float s_ss[TC][NW];                  // per-warp sums of squares

  const int h = blockIdx.x % a.H;
  const int n = blockIdx.x / a.H;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int col0 = warp * CW + (lane % G::LPR) * G::VEC;
  const int row0 = lane / G::LPR;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)h * kD;

  if (n == a.N) {  // padding token rows
    const int lo = min(max(__ldg(a.qsl), 0), a.R);
    const int hi = max(min(__ldg(a.qsl + a.N), a.R), lo);
    for (int t = row0; t < lo; t += G::RPI) store_out_zero<G::VEC>(out + t * a.o_rs + col0);
    for (int t = hi + row0; t < a.R; t += G::RPI) store_out_zero<G::VEC>(out + t * a.o_rs + col0);
    return;
  }

  const int t0 = max(__ldg(a.qsl + n), 0);
  const int t1 = min(__ldg(a.qsl + n + 1), a.R);
  if (t1 <= t0) return;  // empty sequence: nothing written
  const int acc = __ldg(a.accepted + n);
  const int32_t* row_slots = a.idx + (int64_t)n * a.idx_rs;
  const int s0 = (acc >= 1 && acc <= a.cols) ? __ldg(row_slots + acc - 1) : 0;
  if (s0 <= 0 || s0 >= a.num_slots) {  // null sequence: zero its rows, touch no cache
    for (int t = t0 + row0; t < t1; t += G::RPI) store_out_zero<G::VEC>(out + t * a.o_rs + col0);
    return;
  }

  const int64_t head_off = (int64_t)h * kD * kD;
  FltRegs<G> S;
  strip_load<StateT, G>(static_cast<const StateT*>(a.state) + (int64_t)s0 * a.slot_stride + head_off, row0, col0, S);

  // Raw conv history (oldest first) of the thread's channels lc = tid, tid + 256.
  const int HD = a.H * kD;
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(a.x);
  __nv_bfloat16* cs = static_cast<__nv_bfloat16*>(a.conv_state);
  constexpr int NC = (NCH + NT - 1) / NT;
  __nv_bfloat16 hist[NC][3];
  int chan[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const int lc = tid + c * NT;
    chan[c] = lc < NCH ? (lc >> 7) * HD + h * kD + (lc & (kD - 1)) : 0;
    if (lc < NCH) {
      const __nv_bfloat16* cp = cs + (int64_t)s0 * a.cs_slot_stride + chan[c];
#pragma unroll
      for (int p = 0; p < 3; ++p) hist[c][p] = cp[p * a.cs_tap_stride];
    }
  }
  const float A = expf(__ldg(a.A_log + h));
  const float dtb = tid < kD ? __ldg(a.dt_bias + h * kD + tid) : 0.f;
  const float4 nw = __ldg(reinterpret_cast<const float4*>(a.norm_w) + lane);

  for (int tc0 = t0; tc0 < t1; tc0 += TC) {
    const int nt = min(TC, t1 - tc0);
    const int p0 = tc0 - t0;  // position of the chunk's first token in its sequence
    if (tc0 != t0) __syncthreads();  // previous chunk's epilogue done with the shared arrays

    // ---- A: conv + SiLU, conv checkpoints, decays, betas, checkpoint slots
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const int lc = tid + c * NT;
      if (lc >= NCH) continue;
      const int sec = lc >> 7;
      const float* w = a.conv_w + (int64_t)sec * 4 * HD + h * kD + (lc & (kD - 1));
      const float w0 = __ldg(w), w1 = __ldg(w + HD), w2 = __ldg(w + 2 * HD), w3 = __ldg(w + 3 * HD);
      for (int j = 0; j < nt; ++j) {
        const int t = tc0 + j;
        const __nv_bfloat16 xn = xb[(int64_t)t * a.x_rs + chan[c]];
        float y = w0 * __bfloat162float(hist[c][0]);
        y = fmaf(w1, __bfloat162float(hist[c][1]), y);
        y = fmaf(w2, __bfloat162float(hist[c][2]), y);
        y = fmaf(w3, __bfloat162float(xn), y);
        s_act[j][lc] = y * sigmoidf_(y);
        hist[c][0] = hist[c][1];
        hist[c][1] = hist[c][2];
        hist[c][2] = xn;
        if (p0 + j < a.cols) {
          const int sl = __ldg(row_slots + p0 + j);
          if (sl > 0 && sl < a.num_slots) {
            __nv_bfloat16* cp = cs + (int64_t)sl * a.cs_slot_stride + chan[c];
#pragma unroll
            for (int p = 0; p < 3; ++p) cp[p * a.cs_tap_stride] = hist[c][p];
          }
        }
      }
    }
    if (tid < kD) {
      const __nv_bfloat16* gp = static_cast<const __nv_bfloat16*>(a.gate) + (int64_t)h * a.g_hs + tid;
      for (int j = 0; j < nt; ++j)
        s_d[j][tid] = expf(log_decay(__bfloat162float(gp[(int64_t)(tc0 + j) * a.g_rs]) + dtb, A, a.gate_mode,
                                     a.lower_bound));
    }
    if (tid < nt) {
      const float braw = __bfloat162float(
          static_cast<const __nv_bfloat16*>(a.beta)[(int64_t)(tc0 + tid) * a.b_rs + (int64_t)h * a.b_hs]);
      s_tok[tid].x = sigmoidf_(braw);
      int sl = p0 + tid < a.cols ? __ldg(row_slots + p0 + tid) : 0;
      s_slot[tid] = (sl > 0 && sl < a.num_slots) ? sl : 0;
    }
    __syncthreads();

    // ---- B: per-token coefficients, one warp per token
    if (warp < nt) {
      const float4 q = *reinterpret_cast<const float4*>(&s_act[warp][4 * lane]);
      const float4 k = *reinterpret_cast<const float4*>(&s_act[warp][kD + 4 * lane]);
      const float4 d = *reinterpret_cast<const float4*>(&s_d[warp][4 * lane]);
      const float qk = token_coefficients(q, k, d, lane, s_coef[warp]);
      if (lane == 0) s_tok[warp].y = qk;
    }
    __syncthreads();

    // ---- C: the chunk's tokens on this warp's strip
    for (int j = 0; j < nt; ++j) {
      const float2 tk = s_tok[j];
      float acc_a[G::VEC], acc_b[G::VEC];
      strip_reduce<G>(S, s_coef[j], row0, acc_a, acc_b);
      float u[G::VEC], o[G::VEC];
      float ss = 0.f;
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) {
        u[jj] = tk.x * (s_act[j][2 * kD + col0 + jj] - acc_a[jj]);
        o[jj] = a.scale * (acc_b[jj] + tk.y * u[jj]);
        ss = fmaf(o[jj], o[jj], ss);
      }
      strip_update<G>(S, s_coef[j], row0, u);
      const int sl = s_slot[j];
      if (sl != 0)
        strip_store<StateT, G>(static_cast<StateT*>(a.state) + (int64_t)sl * a.slot_stride + head_off, row0, col0, S);
      if (row0 == 0) {
#pragma unroll
        for (int jj = 0; jj < G::VEC; ++jj) s_o[j][col0 + jj] = o[jj];
      }
      ss = warp_sum(row0 == 0 ? ss : 0.f);
      if (lane == 0) s_ss[j][warp] = ss;
    }
    __syncthreads();

    // ---- D: gated RMSNorm and the output row, one warp per token
    if (warp < nt) {
      const int t = tc0 + warp;
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) tot += s_ss[warp][w];
      const float rinv = rsqrtf(tot * (1.f / kD) + a.norm_eps);
      const float4 o4 = *reinterpret_cast<const float4*>(&s_o[warp][4 * lane]);
      const float4 g4 = load4(a.out_gate, (int64_t)t * a.og_rs + (int64_t)h * a.og_hs + 4 * lane, KDA_DT_BF16);
      float y[4] = {o4.x * rinv * nw.x * sigmoidf_(g4.x), o4.y * rinv * nw.y * sigmoidf_(g4.y),
                    o4.z * rinv * nw.z * sigmoidf_(g4.z), o4.w * rinv * nw.w * sigmoidf_(g4.w)};
      store_out<4>(out + (int64_t)t * a.o_rs + 4 * lane, y);
    }
  }
}

cudaError_t launch_packed_fused(const PackedFusedArgs& a, int state_dtype, cudaStream_t s) {
  const int64_t blocks = (int64_t)(a.N + 1) * a.H;  // slice N zeroes padding rows
  if (state_dtype == KDA_DT_F32) {
    kda_packed_fused_kernel<float><<<dim3((unsigned)blocks), dim3(256), 0, s>>>(a);
  } else {
    kda_packed_fused_kernel<__nv_bfloat16><<<dim3((unsigned)blocks), dim3(256), 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kda
