// Packed speculative (T >= 1, ragged cu_seqlens) decode: kernel instantiations and launcher.
#include "kda_kernels.cuh"

namespace kda {

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

// Column sums of a 16-column strip's two k-reductions by reduce-scatter over
// the strip's 2 VEC row groups: at each level a lane keeps one half of its
// values and adds its partner's copy of that half, so the lane of row group
// rg ends holding value rg of (a_0 .. a_{VEC-1}, b_0 .. b_{VEC-1}) summed
// over all rows.
template <typename G>
__device__ __forceinline__ float spec_reduce_scatter(const float2 (&a2)[G::VEC / 2], const float2 (&b2)[G::VEC / 2],
                                                     int rg) {
  constexpr int NV = 2 * G::VEC;
  static_assert(NV == G::RPI, "one value per row group");
  constexpr int LEVELS = NV == 8 ? 3 : (NV == 16 ? 4 : 0);
  static_assert(LEVELS > 0, "8 or 16 row groups");
  float v[NV];
#pragma unroll
  for (int p = 0; p < G::VEC / 2; ++p) {
    v[2 * p] = a2[p].x; v[2 * p + 1] = a2[p].y;
    v[G::VEC + 2 * p] = b2[p].x; v[G::VEC + 2 * p + 1] = b2[p].y;
  }
#pragma unroll
  for (int l = 0; l < LEVELS; ++l) {
    const int half = NV >> (l + 1);
    const int bit = LEVELS - 1 - l;  // the row-group bit of this level, most significant first
    const bool hi = (rg >> bit) & 1;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = hi ? v[i] : v[i + half];
      const float keep = hi ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, G::LPR << bit);
    }
  }
  return v[0];
}

template <typename StateT, int CW, int NW, bool VERIFY>
__global__ void __launch_bounds__(NW * 32, MinBlocks<NW>::value) kda_spec_kernel(const SpecArgs a) {
  using G = Strip<StateT, CW>;
  constexpr int SPLIT = kD / (CW * NW);
  constexpr int TC = 8;
  constexpr int NT = NW * 32;
  static_assert(SPLIT * CW * NW == kD, "split must tile the 128 value columns");
  // Per key row: staged (q, k) and g, then (P k, P q) and k / P; the reduction
  // reads one 8-byte pair a row, the update one float.
  __shared__ __align__(16) float2 s_ab[TC][kD];
  __shared__ __align__(16) float s_ku[TC][kD];
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
  pdl_wait();
  pdl_launch_dependents();

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
      float4* ab = reinterpret_cast<float4*>(&s_ab[j][4 * lane]);
      ab[0] = make_float4(q.x * rq, k.x * rk, q.y * rq, k.y * rk);
      ab[1] = make_float4(q.z * rq, k.z * rk, q.w * rq, k.w * rk);
      reinterpret_cast<float4*>(s_ku[j])[lane] = g;
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
        const float2 c = s_ab[j][r];  // (q, k)
        Gs += s_ku[j][r];  // g
        P = expf(Gs);
        const float ku = c.y * expf(-Gs);
        s_ab[j][r] = make_float2(P * c.y, P * c.x);
        s_ku[j][r] = ku;
      }
      s_P[r] = P;
    }
    __syncthreads();
    for (int j = 0; j < ne; ++j) {
      const int t = tc0 + j;
      const float4 tk = s_tok[j];
      // bf16 state (16 row groups): the column sums by reduce-scatter, 24
      // shuffles instead of 64; the lane of row group rg < VEC forms u for
      // column rg, the lane VEC groups up forms o for it, every lane gathers u
      constexpr bool kScatter = sizeof(StateT) == 2 && 2 * G::VEC == G::RPI;
      float u[G::VEC], o[G::VEC];
      {
        float2 a2[G::VEC / 2], b2[G::VEC / 2];
#pragma unroll
        for (int p = 0; p < G::VEC / 2; ++p) { a2[p] = make_float2(0.f, 0.f); b2[p] = make_float2(0.f, 0.f); }
#pragma unroll
        for (int i = 0; i < G::PASSES; ++i) {
          const float2 c = s_ab[j][row0 + i * G::RPI];
          accumulate_row<G::VEC / 2>(make_float4(c.x, c.y, 0.f, 0.f), S.s[i], a2, b2);
        }
        if constexpr (kScatter) {
          const float tot = spec_reduce_scatter<G>(a2, b2, row0);
          const float uc = row0 < G::VEC ? tk.x * (s_v[j][col0 + row0] - tot) : 0.f;
          const float u_lo = __shfl_xor_sync(0xffffffffu, uc, G::LPR * G::VEC);
          if (row0 >= G::VEC) out[t * out_rs + row0 - G::VEC] = __float2bfloat16_rn(a.scale * (tot + tk.y * u_lo));
#pragma unroll
          for (int c = 0; c < G::VEC; ++c) u[c] = __shfl_sync(0xffffffffu, uc, c * G::LPR + lane % G::LPR);
        } else {
          float acc_a[G::VEC], acc_b[G::VEC];
          strip_allreduce<G>(a2, b2, acc_a, acc_b);
#pragma unroll
          for (int jj = 0; jj < G::VEC; ++jj) {
            u[jj] = tk.x * (s_v[j][col0 + jj] - acc_a[jj]);
            o[jj] = a.scale * (acc_b[jj] + tk.y * u[jj]);
          }
        }
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
        const float2 ku = dup2(s_ku[j][row0 + i * G::RPI]);
#pragma unroll
        for (int p = 0; p < G::VEC / 2; ++p) S.s[i][p] = fma2(ku, u2[p], S.s[i][p]);
      }
      if (!kScatter && row0 == 0) store_out<G::VEC>(out + t * out_rs, o);
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

namespace {

template <typename StateT, int CW, int NW, bool VERIFY>
cudaError_t launch_spec_variant(const SpecArgs& a, cudaStream_t s) {
  constexpr int SPLIT = kD / (CW * NW);
  const int64_t blocks = (int64_t)(a.N + 1) * a.H * SPLIT;  // slice N zeroes padding rows
  return launch_pdl(kda_spec_kernel<StateT, CW, NW, VERIFY>, dim3((unsigned)blocks), dim3(NW * 32), 0, s, 1, a);
}

template <typename StateT, bool VERIFY>
cudaError_t launch_spec_typed(const SpecArgs& a, int split, cudaStream_t s) {
  switch (split) {
    case 1: return launch_spec_variant<StateT, 16, 8, VERIFY>(a, s);
    case 2: return launch_spec_variant<StateT, 16, 4, VERIFY>(a, s);
    case 4: return launch_spec_variant<StateT, 16, 2, VERIFY>(a, s);
    case 8: return launch_spec_variant<StateT, 16, 1, VERIFY>(a, s);
    case 16: return launch_spec_variant<StateT, 8, 1, VERIFY>(a, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_spec(const SpecArgs& a, int state_dtype, int split, bool verify, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32)
    return verify ? launch_spec_typed<float, true>(a, split, s) : launch_spec_typed<float, false>(a, split, s);
  return verify ? launch_spec_typed<__nv_bfloat16, true>(a, split, s)
                : launch_spec_typed<__nv_bfloat16, false>(a, split, s);
}

}  // namespace kda
