// Persistent streaming T=1 decode: one CTA per SM walks its share of the
// (row, head) units.  A producer warp moves each unit's whole state block
// (and the unit's q, k, v, raw gate and dt_bias vectors) into a shared-memory
// stage with bulk asynchronous copies; eight consumer warps take the stages
// in order, each reducing its 16-column strip from shared memory and writing
// the updated state straight from registers to global memory.  With three
// (float32) or five (bfloat16) stages the SM keeps ~200 KB of state loads in
// flight regardless of register pressure.
//
// Every wait is bounded in time; on a timeout the warp records a bit in
// g_kda_device_error and returns (no barrier spans the warps after set-up).
#include "kda_async.cuh"
#include "kda_kernels.cuh"

namespace kda {

// bit 0: a stage-full wait timed out; bit 1: a stage-free wait timed out.
__device__ unsigned int g_kda_device_error = 0;

template <typename StateT>
struct StreamCfg {
  static constexpr int NW = 8;   // consumer warps
  static constexpr int CW = 16;  // columns per consumer warp
  static constexpr int NSTAGE = sizeof(StateT) == 4 ? 3 : 5;
  static constexpr uint32_t STATE_BYTES = kD * kD * sizeof(StateT);
  static constexpr uint32_t ACT_SLOT = 512;                   // one 128-vector, up to float32
  static constexpr uint32_t ACT_BYTES = 5 * ACT_SLOT;         // q, k, v, raw gate, dt_bias
  static constexpr uint32_t STAGE_BYTES = STATE_BYTES + ACT_BYTES;
  static constexpr size_t COEF_OFF = (size_t)NSTAGE * STAGE_BYTES;
  static constexpr size_t SCAL_OFF = COEF_OFF + (size_t)NW * kD * sizeof(float4);
  static constexpr size_t BAR_OFF = SCAL_OFF + (size_t)NSTAGE * sizeof(int4);
  static constexpr size_t SMEM = BAR_OFF + 2 * NSTAGE * sizeof(uint64_t);
  static_assert(CW * NW == kD, "consumers cover the 128 value columns");
  static_assert(SMEM <= 232448, "stages exceed the 227 KB shared memory of a CTA");
};

__device__ __forceinline__ float4 lds4(const unsigned char* base, int i, int dtype) {
  if (dtype == KDA_DT_F32) return reinterpret_cast<const float4*>(base)[i >> 2];
  const uint2 u = reinterpret_cast<const uint2*>(base)[i >> 2];
  return make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
}

template <typename StateT>
__global__ void __launch_bounds__((StreamCfg<StateT>::NW + 1) * 32, 1)
    kda_t1_stream_kernel(const T1Args a, const int units) {
  using C = StreamCfg<StateT>;
  using G = Strip<StateT, C::CW>;
  extern __shared__ __align__(128) unsigned char smem[];
  float4* coef_all = reinterpret_cast<float4*>(smem + C::COEF_OFF);
  int4* scal = reinterpret_cast<int4*>(smem + C::SCAL_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* empty = full + C::NSTAGE;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], C::NW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  const int P = gridDim.x;
  const int n_my = (units - (int)blockIdx.x + P - 1) / P;  // units blockIdx.x + j*P
  const int qsz = a.qkv_dtype == KDA_DT_F32 ? 4 : 2;
  const int gsz = a.gate_dtype == KDA_DT_F32 ? 4 : 2;

  if (warp == C::NW) {
    // ---------------- producer ----------------
    for (int j0 = 0; j0 < n_my; j0 += 32) {
      int slot = -1;
      float beta = 0.f, A = 0.f;
      if (j0 + lane < n_my) {  // per-unit scalars, 32 units at a time
        const int u = blockIdx.x + (j0 + lane) * P;
        const int h = u % a.H, b = u / a.H;
        slot = __ldg(a.idx + b);
        beta = sigmoidf_(load1(a.beta, (int64_t)b * a.b_rs + (int64_t)h * a.b_hs, a.beta_dtype));
        A = expf(__ldg(a.A_log + h));
      }
      const int cnt = min(32, n_my - j0);
      for (int t = 0; t < cnt; ++t) {
        const int j = j0 + t;
        const int s = j % C::NSTAGE;
        const uint32_t round = j / C::NSTAGE;
        const int slot_t = __shfl_sync(0xffffffffu, slot, t);
        const float beta_t = __shfl_sync(0xffffffffu, beta, t);
        const float A_t = __shfl_sync(0xffffffffu, A, t);
        const bool ok = round == 0 || mbar_wait(&empty[s], (round - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {  // the whole warp leaves together
          if (lane == 0) atomicOr(&g_kda_device_error, 2u);
          return;
        }
        if (lane == 0) {
          const int u = blockIdx.x + j * P;
          const int h = u % a.H, b = u / a.H;
          const bool live = slot_t > 0 && slot_t < a.num_slots;
          scal[s] = make_int4(live ? slot_t : -1, __float_as_int(beta_t), __float_as_int(A_t), 0);
          if (live) {
            unsigned char* st = smem + (size_t)s * C::STAGE_BYTES;
            const uint32_t qb = kD * qsz, gb = kD * gsz;
            mbar_arrive_expect_tx(&full[s], C::STATE_BYTES + 3 * qb + gb + kD * 4);
            const StateT* src = static_cast<const StateT*>(a.state) + (int64_t)slot_t * a.slot_stride +
                                (int64_t)h * kD * kD;
            bulk_load(st, src, C::STATE_BYTES, &full[s]);
            unsigned char* act = st + C::STATE_BYTES;
            bulk_load(act, static_cast<const char*>(a.q) + ((int64_t)b * a.q_rs + (int64_t)h * a.q_hs) * qsz, qb,
                      &full[s]);
            bulk_load(act + C::ACT_SLOT,
                      static_cast<const char*>(a.k) + ((int64_t)b * a.k_rs + (int64_t)h * a.k_hs) * qsz, qb, &full[s]);
            bulk_load(act + 2 * C::ACT_SLOT,
                      static_cast<const char*>(a.v) + ((int64_t)b * a.v_rs + (int64_t)h * a.v_hs) * qsz, qb, &full[s]);
            bulk_load(act + 3 * C::ACT_SLOT,
                      static_cast<const char*>(a.gate) + ((int64_t)b * a.g_rs + (int64_t)h * a.g_hs) * gsz, gb,
                      &full[s]);
            bulk_load(act + 4 * C::ACT_SLOT, a.dt_bias + h * kD, kD * 4, &full[s]);
          } else {
            mbar_arrive(&full[s]);
          }
        }
        __syncwarp();
      }
    }
    return;
  }

  // ---------------- consumers ----------------
  const int col0 = warp * C::CW + (lane % G::LPR) * G::VEC;
  const int row0 = lane / G::LPR;
  float4* coef = coef_all + warp * kD;
  for (int j = 0; j < n_my; ++j) {
    const int s = j % C::NSTAGE;
    const uint32_t round = j / C::NSTAGE;
    const bool ok = mbar_wait(&full[s], round & 1);
    if (!__all_sync(0xffffffffu, ok)) {  // the whole warp leaves together
      if (lane == 0) atomicOr(&g_kda_device_error, 1u);
      return;
    }
    const int u = blockIdx.x + j * P;
    const int h = u % a.H, b = u / a.H;
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + ((int64_t)b * a.H + h) * kD;
    const int4 sc = scal[s];
    if (sc.x < 0) {  // null row: zero output, no cache access
      if (row0 == 0) store_out_zero<G::VEC>(out + col0);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    const unsigned char* st = smem + (size_t)s * C::STAGE_BYTES;
    const unsigned char* act = st + C::STATE_BYTES;
    const float beta = __int_as_float(sc.y);
    const float A = __int_as_float(sc.z);
    const float4 q = lds4(act, 4 * lane, a.qkv_dtype);
    const float4 k = lds4(act + C::ACT_SLOT, 4 * lane, a.qkv_dtype);
    const float4 gr = lds4(act + 3 * C::ACT_SLOT, 4 * lane, a.gate_dtype);
    const float4 dtb = reinterpret_cast<const float4*>(act + 4 * C::ACT_SLOT)[lane];
    float vv[G::VEC];
#pragma unroll
    for (int jj = 0; jj < G::VEC; jj += 4) {
      const float4 t = lds4(act + 2 * C::ACT_SLOT, col0 + jj, a.qkv_dtype);
      vv[jj] = t.x; vv[jj + 1] = t.y; vv[jj + 2] = t.z; vv[jj + 3] = t.w;
    }
    float4 d;
    d.x = expf(log_decay(gr.x + dtb.x, A, a.gate_mode, a.lower_bound));
    d.y = expf(log_decay(gr.y + dtb.y, A, a.gate_mode, a.lower_bound));
    d.z = expf(log_decay(gr.z + dtb.z, A, a.gate_mode, a.lower_bound));
    d.w = expf(log_decay(gr.w + dtb.w, A, a.gate_mode, a.lower_bound));
    const float qk = token_coefficients(q, k, d, lane, coef);
    __syncwarp();

    RawRegs<StateT, G> S;
    const StateT* ss = reinterpret_cast<const StateT*>(st);
#pragma unroll
    for (int i = 0; i < G::PASSES; ++i)
      S.r[i] = *reinterpret_cast<const typename Frag<StateT>::Raw*>(ss + (row0 + i * G::RPI) * kD + col0);
    float acc_a[G::VEC], acc_b[G::VEC];
    strip_reduce<G>(S, coef, row0, acc_a, acc_b);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // the stage is no longer read by this warp

    float u_[G::VEC], o[G::VEC];
#pragma unroll
    for (int jj = 0; jj < G::VEC; ++jj) {
      u_[jj] = beta * (vv[jj] - acc_a[jj]);
      o[jj] = a.scale * (acc_b[jj] + qk * u_[jj]);
    }
    StateT* sp = static_cast<StateT*>(a.state) + (int64_t)sc.x * a.slot_stride + (int64_t)h * kD * kD;
    strip_update_store<StateT, G>(sp, row0, col0, S, coef, u_);
    if (row0 == 0) store_out<G::VEC>(out + col0, o);
  }
}

template <typename StateT>
cudaError_t launch_stream_typed(const T1Args& a, int sm_count, cudaStream_t s) {
  using C = StreamCfg<StateT>;
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !attr_set[dev]) {
    cudaError_t e = cudaFuncSetAttribute(kda_t1_stream_kernel<StateT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM);
    if (e != cudaSuccess) return e;
    attr_set[dev] = true;
  }
  const int units = a.B * a.H;
  const int grid = units < sm_count ? units : sm_count;
  kda_t1_stream_kernel<StateT><<<grid, (C::NW + 1) * 32, C::SMEM, s>>>(a, units);
  return cudaGetLastError();
}

cudaError_t launch_t1_stream(const T1Args& a, int state_dtype, int sm_count, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_stream_typed<float>(a, sm_count, s);
  return launch_stream_typed<__nv_bfloat16>(a, sm_count, s);
}

cudaError_t read_device_error(unsigned int* flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_kda_device_error, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
