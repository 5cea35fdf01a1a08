// Persistent streaming decode kernels: one CTA per SM walks its share of the
// (row, head) units through rings of shared-memory stages.
//
//   loader warp    per unit: the slot index, beta and A_log; TMA tensor
//                  copies of the 128 x 128 state block (128-byte swizzled,
//                  in 128-byte-wide column blocks) and bulk copies of the
//                  unit's activation vectors.  T=1: one ring, state and
//                  activations on the stage's `full` barrier.  Fused: two
//                  rings, the activations a few units ahead of the state.
//   prologue warps per unit, once, units dealt round-robin: (fused: the short conv + SiLU of the
//                  head's 384 channels, the conv-cache shift written back
//                  from registers) the L2 norms, gate and decay of the 128 key
//                  channels into the coefficient array (d k, d q, d, k) and
//                  q.k; then `ready`.
//   8 consumers    per unit: a 16-column strip over all 128 key rows from
//                  shared memory: the two k-reductions (in-thread plus xor
//                  shuffles), u and o, release of the stage (`empty`), the
//                  update written straight from registers to global.
//   epilogue warp  (fused) per unit: the gated RMSNorm of the consumers' o.
//
// The state rings keep 160-200 KB of loads in flight per SM.  Every mbarrier
// wait is bounded in time; a warp whose wait times out records a bit in
// g_kda_device_error and leaves, and the warps waiting on it time out in turn.
// No barrier spans warps after set-up.
#include <atomic>

#include "kda_stream_common.cuh"

namespace kda {

// bit 0: a stage-full/ready wait timed out; bit 1: a stage-free wait timed
// out; bit 2: the self-test wait timed out (expected).
__device__ unsigned int g_kda_device_error = 0;

__device__ __forceinline__ void record_error(unsigned int bit) { atomicOr(&g_kda_device_error, bit); }

// Consumer core shared by the stream kernels: reads the lane's fragments of
// a swizzled stage into registers, keeps each row's (decay, key) pair, and
// accumulates the column-pair sums of the two k-reductions.
template <typename StateT, typename G>
__device__ __forceinline__ void reduce_stage(const unsigned char* st, const float4* coef, int row0, int col0,
                                             typename Frag<StateT>::Raw (&S)[G::PASSES], float2 (&dk)[G::PASSES],
                                             float2 (&acc_a)[G::VEC / 2], float2 (&acc_b)[G::VEC / 2]) {
#pragma unroll
  for (int p = 0; p < G::VEC / 2; ++p) { acc_a[p] = make_float2(0.f, 0.f); acc_b[p] = make_float2(0.f, 0.f); }
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    const int r = row0 + i * G::RPI;
    S[i] = *reinterpret_cast<const typename Frag<StateT>::Raw*>(st + swz_offset<StateT>(r, col0));
    const float4 c = coef[r];
    dk[i] = make_float2(c.z, c.w);
    float2 x2[G::VEC / 2];
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) x2[p] = Frag<StateT>::get2(S[i], p);
    accumulate_row<G::VEC / 2>(c, x2, acc_a, acc_b);
  }
}

// The column sums by reduce-scatter (strip_reduce_scatter) where a strip has
// 2 VEC row groups, i.e. with a bf16 state: 24 shuffles instead of 64.
template <typename StateT, typename G>
constexpr bool kStreamScatter = sizeof(StateT) == 2 && 2 * G::VEC == G::RPI;

// S' = d S + k u^T from the registers of reduce_stage, stored to global.
template <typename StateT, typename G>
__device__ __forceinline__ void update_store_regs(StateT* sp, int row0, int col0,
                                                  const typename Frag<StateT>::Raw (&S)[G::PASSES],
                                                  const float2 (&dk)[G::PASSES], const float (&u)[G::VEC]) {
  float2 u2[G::VEC / 2];
  pairs_of<G::VEC>(u, u2);
#pragma unroll
  for (int i = 0; i < G::PASSES; ++i) {
    float2 x2[G::VEC / 2], y2[G::VEC / 2];
#pragma unroll
    for (int p = 0; p < G::VEC / 2; ++p) x2[p] = Frag<StateT>::get2(S[i], p);
    update_row<G::VEC / 2>(dk[i].x, dk[i].y, x2, u2, y2);
    Frag<StateT>::store(sp + (row0 + i * G::RPI) * kD + col0, Frag<StateT>::pack2(y2));
  }
}

// =====================================================================================
// T=1 recurrent / packed
// =====================================================================================
constexpr uint32_t T1_ACT_SLOT = 512;  // one 128-vector, up to float32: q, k, v, raw gate, dt_bias

template <typename StateT>
using T1Stream = StageCfg<StateT, 5 * T1_ACT_SLOT, sizeof(StateT) == 4 ? 3 : 5>;
// bfloat16 state in halves: a work item is one 64-column TMA block of a unit,
// which halves the last round's share of the persistent CTAs.
template <typename StateT, int PARTS>
using T1StreamP = StageCfg<StateT, 5 * T1_ACT_SLOT, PARTS == 1 ? (sizeof(StateT) == 4 ? 3 : 5) : 10, 0, PARTS>;
// Prologue warps.  Units are dealt to them round-robin; NP must divide
// NSTAGE so each stage is always served by the same prologue warp in round
// order (a parity wait cannot tell a phase from the one two rounds later).
template <int PARTS>
__host__ __device__ constexpr int t1_np() {
  return PARTS;  // every work item repeats its unit's coefficients: one prologue warp per part
}

template <typename StateT, int PARTS>
__host__ __device__ constexpr size_t t1_stream_smem() {
  return T1StreamP<StateT, PARTS>::TAIL_OFF + 1024;  // + base alignment slack
}

template <typename StateT, int PARTS>
__global__ void __launch_bounds__((T1StreamP<StateT, PARTS>::NW + 1 + t1_np<PARTS>()) * 32, 1)
    kda_t1_stream_kernel(const T1Args a, const __grid_constant__ CUtensorMap state_map, const int items) {
  using C = T1StreamP<StateT, PARTS>;
  using G = Strip<StateT, C::CW>;
  static_assert(t1_stream_smem<StateT, PARTS>() <= 232448, "stages exceed the 227 KB shared memory of a CTA");
  static_assert(C::NSTAGE % t1_np<PARTS>() == 0, "each stage must be served by one prologue warp");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  float4* coef_all = reinterpret_cast<float4*>(smem + C::COEF_OFF);
  int4* scal = reinterpret_cast<int4*>(smem + C::SCAL_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
  uint64_t* ready = full + C::NSTAGE;
  uint64_t* empty = ready + C::NSTAGE;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NSTAGE; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&ready[s], 1);
      mbar_init(&empty[s], C::GROUP_WARPS);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int P = gridDim.x;
  const int n_my = (items - (int)blockIdx.x + P - 1) / P;  // items blockIdx.x + j*P; item i = unit i / PARTS
  const int qsz = a.qkv_dtype == KDA_DT_F32 ? 4 : 2;
  const int gsz = a.gate_dtype == KDA_DT_F32 ? 4 : 2;

  if (warp == C::NW) {
    // ---------------- loader ----------------
    for (int j0 = 0; j0 < n_my; j0 += 32) {
      int slot = -1;
      float beta = 0.f, A = 0.f;
      if (j0 + lane < n_my) {  // per-item scalars, 32 items at a time
        const int u = (blockIdx.x + (j0 + lane) * P) / PARTS;
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
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_error(2u);
          return;
        }
        if (lane == 0) {
          const int item = blockIdx.x + j * P;
          const int u = item / PARTS, part = item % PARTS;
          const int h = u % a.H, b = u / a.H;
          const bool live = slot_t > 0 && slot_t < a.num_slots;
          scal[s] = make_int4(live ? slot_t : -1, __float_as_int(beta_t), __float_as_int(A_t), 0);
          if (live) {
            unsigned char* st = smem + (size_t)s * C::STAGE_BYTES;
            const uint32_t qb = kD * qsz, gb = kD * gsz;
            mbar_arrive_expect_tx(&full[s], C::PART_BYTES + 3 * qb + gb + kD * 4);
#pragma unroll
            for (int blk = 0; blk < C::PART_BLKS; ++blk)
              tma_load_3d(st + blk * C::BLK_BYTES, &state_map, (part * C::PART_BLKS + blk) * C::BLK_COLS, h * kD,
                          slot_t, &full[s]);
            unsigned char* act = st + C::PART_BYTES;
            const char* q = static_cast<const char*>(a.q) + ((int64_t)b * a.q_rs + (int64_t)h * a.q_hs) * qsz;
            const char* k = static_cast<const char*>(a.k) + ((int64_t)b * a.k_rs + (int64_t)h * a.k_hs) * qsz;
            const char* v = static_cast<const char*>(a.v) + ((int64_t)b * a.v_rs + (int64_t)h * a.v_hs) * qsz;
            const char* g = static_cast<const char*>(a.gate) + ((int64_t)b * a.g_rs + (int64_t)h * a.g_hs) * gsz;
            bulk_load(act, q, qb, &full[s]);
            bulk_load(act + T1_ACT_SLOT, k, qb, &full[s]);
            bulk_load(act + 2 * T1_ACT_SLOT, v, qb, &full[s]);
            bulk_load(act + 3 * T1_ACT_SLOT, g, gb, &full[s]);
            bulk_load(act + 4 * T1_ACT_SLOT, a.dt_bias + h * kD, kD * 4, &full[s]);
          } else {
            mbar_arrive(&full[s]);
          }
        }
        __syncwarp();
      }
    }
    return;
  }

  if (warp > C::NW) {
    // ---------------- prologue warps (units round-robin): per-key-channel coefficients, once ----------------
    for (int j = warp - C::NW - 1; j < n_my; j += t1_np<PARTS>()) {
      const int s = j % C::NSTAGE;
      const bool ok = mbar_wait(&full[s], (j / C::NSTAGE) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(1u);
        return;
      }
      const int4 sc = scal[s];
      if (sc.x >= 0) {
        const unsigned char* act = smem + (size_t)s * C::STAGE_BYTES + C::PART_BYTES;
        const float A = __int_as_float(sc.z);
        const float4 q = lds4(act, 4 * lane, a.qkv_dtype);
        const float4 k = lds4(act + T1_ACT_SLOT, 4 * lane, a.qkv_dtype);
        const float4 gr = lds4(act + 3 * T1_ACT_SLOT, 4 * lane, a.gate_dtype);
        const float4 dtb = reinterpret_cast<const float4*>(act + 4 * T1_ACT_SLOT)[lane];
        float4 d;
        d.x = expf(log_decay(gr.x + dtb.x, A, a.gate_mode, a.lower_bound));
        d.y = expf(log_decay(gr.y + dtb.y, A, a.gate_mode, a.lower_bound));
        d.z = expf(log_decay(gr.z + dtb.z, A, a.gate_mode, a.lower_bound));
        d.w = expf(log_decay(gr.w + dtb.w, A, a.gate_mode, a.lower_bound));
        const float qk = token_coefficients(q, k, d, lane, coef_all + s * kD);
        if (lane == 0) scal[s].w = __float_as_int(qk);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ready[s]);
    }
    return;
  }

  // ---------------- consumers: group warp / GROUP_WARPS takes items j = group, group + PARTS, ... ----------------
  const int col0 = (warp % C::GROUP_WARPS) * C::CW + (lane % G::LPR) * G::VEC;  // column within the staged part
  const int row0 = stream_row0<G::LPR>(lane);
  // The unit advances by P from one of this group's items to the next, so
  // with a bf16 state (whose consumers set the pace) its head is kept by one
  // conditional subtraction instead of a division; the float32 kernel, at its
  // register cap, divides.
  constexpr bool kStepH = sizeof(StateT) == 2;
  const int h_step = P % a.H;
  int h_run = (int)(((blockIdx.x + (warp / C::GROUP_WARPS) * P) / PARTS) % a.H);
  for (int j = warp / C::GROUP_WARPS; j < n_my;
       j += PARTS, h_run = h_run + h_step >= a.H ? h_run + h_step - a.H : h_run + h_step) {
    const int s = j % C::NSTAGE;
    const uint32_t par = (j / C::NSTAGE) & 1;
    const bool ok = mbar_wait(&full[s], par) && mbar_wait(&ready[s], par);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) record_error(1u);
      return;
    }
    const int item = blockIdx.x + j * P;
    const int u = item / PARTS;
    const int gcol = (item % PARTS) * C::PART_COLS + col0;  // column within the unit
    __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)u * kD;  // u = b * H + h
    const int h = kStepH ? h_run : u % a.H;
    const int4 sc = scal[s];
    if (sc.x < 0) {  // null row: zero output, no cache access
      if (row0 == 0) store_out_zero<G::VEC>(out + gcol);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      continue;
    }
    const unsigned char* st = smem + (size_t)s * C::STAGE_BYTES;
    const unsigned char* vact = st + C::PART_BYTES + 2 * T1_ACT_SLOT;
    const float4* coef = coef_all + s * kD;
    float2 acc2_a[G::VEC / 2], acc2_b[G::VEC / 2];
    // v before the stage is released: the lane's VEC columns, or with the
    // scatter the one column its row group forms u for
    const int rg = lane / G::LPR;
    float vv[G::VEC];
    if constexpr (kStreamScatter<StateT, G>) {
      vv[0] = rg < G::VEC ? (a.qkv_dtype == KDA_DT_F32
                                 ? reinterpret_cast<const float*>(vact)[gcol + rg]
                                 : __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(vact)[gcol + rg]))
                          : 0.f;
    } else {
#pragma unroll
      for (int jj = 0; jj < G::VEC; jj += 4) {
        const float4 t = lds4(vact, gcol + jj, a.qkv_dtype);
        vv[jj] = t.x; vv[jj + 1] = t.y; vv[jj + 2] = t.z; vv[jj + 3] = t.w;
      }
    }
    // k-reductions; the decay and key coefficients of each row stay in registers
    typename Frag<StateT>::Raw S[G::PASSES];
    float2 dk[G::PASSES];
    reduce_stage<StateT, G>(st, coef, row0, col0, S, dk, acc2_a, acc2_b);
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp no longer reads the stage
    const float beta = __int_as_float(sc.y);
    const float qk = __int_as_float(sc.w);
    float u_[G::VEC];
    if constexpr (kStreamScatter<StateT, G>) {
      // bf16 (16 row groups): the lane of row group rg < VEC forms u for
      // column rg of its VEC, the lane VEC groups up forms o for it and
      // writes it; every lane then gathers the VEC u
      const float tot = strip_reduce_scatter<G>(acc2_a, acc2_b, rg);
      const float uc = rg < G::VEC ? beta * (vv[0] - tot) : 0.f;
      const float u_lo = __shfl_xor_sync(0xffffffffu, uc, G::LPR * G::VEC);
      if (rg >= G::VEC) out[gcol + rg - G::VEC] = __float2bfloat16_rn(a.scale * (tot + qk * u_lo));
#pragma unroll
      for (int c = 0; c < G::VEC; ++c) u_[c] = __shfl_sync(0xffffffffu, uc, c * G::LPR + lane % G::LPR);
    } else {
      float acc_a[G::VEC], acc_b[G::VEC], o[G::VEC];
      strip_allreduce<G>(acc2_a, acc2_b, acc_a, acc_b);
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) {
        u_[jj] = beta * (vv[jj] - acc_a[jj]);
        o[jj] = a.scale * (acc_b[jj] + qk * u_[jj]);
      }
      if (row0 == 0) store_out<G::VEC>(out + gcol, o);
    }
    StateT* sp = static_cast<StateT*>(a.state) + (int64_t)sc.x * a.slot_stride + (int64_t)h * kD * kD;
    update_store_regs<StateT, G>(sp, row0, gcol, S, dk, u_);
  }
}

// =====================================================================================
// Fused short conv + SiLU + KDA + gated RMSNorm
// =====================================================================================
// Activation entry (bf16 unless noted): x of the head's q|k|v channels
// (3 x 256 B), the conv cache taps (3 taps x 3 sections x 256 B), the raw
// gate (256 B), dt_bias (512 B, f32) and the output gate (256 B); then the
// prologue's results: the coefficients (128 float4) and SiLU(conv) of the
// 128 v channels (f32); the consumers' o before the norm (f32); and the
// unit's scalars (slot, beta, A, q.k).
constexpr uint32_t F_X = 0, F_CS = 768, F_G = 3072, F_DT = 3328, F_OG = 3840, F_ACT = 4096;
constexpr uint32_t F_COEF = F_ACT, F_V = F_COEF + kD * 16, F_O = F_V + kD * 4, F_SCAL = F_O + kD * 4,
                   F_ENTRY = F_SCAL + 16;

// Two rings: NS state stages (TMA destinations, 1024-byte aligned) and NA
// activation entries.  The loader fills the entries LA = NA - NS units ahead
// of the state, so the prologue (conv, decay, coefficients: ~2.5 us a unit
// on one warp) is done before the unit's state lands and is not part of a
// state stage's turnaround.  NP prologue warps serve the entries
// round-robin; NP divides NA, so an entry is always served by the same warp
// in round order (a parity wait cannot tell a phase from the one two rounds
// later).  The gated RMSNorm runs on an epilogue warp from the consumers' o
// in the entry, so the consumer warps never wait on one another.
template <typename StateT>
struct FusedRing : SwzCfg<StateT> {
  static constexpr int NS = sizeof(StateT) == 4 ? 3 : 5;
  static constexpr int NA = sizeof(StateT) == 4 ? 4 : 8;
  static constexpr int LA = NA - NS;
  static constexpr int NP = 2;
  static constexpr int NW = 8;   // consumer warps
  static constexpr int CW = 16;  // columns per consumer warp
  static constexpr int WARPS = NW + 1 + NP + 1;  // consumers, loader, prologue, epilogue
  static constexpr size_t ACT_OFF = (size_t)NS * SwzCfg<StateT>::STATE_BYTES;
  static constexpr size_t BAR_OFF = ACT_OFF + (size_t)NA * F_ENTRY;
  static constexpr size_t TAIL_OFF = BAR_OFF + (size_t)(2 * NS + 4 * NA) * sizeof(uint64_t);
  static_assert(LA >= 0 && NA % NP == 0 && F_ENTRY % 16 == 0 && NW * CW == kD, "fused ring geometry");
};

template <typename StateT>
__host__ __device__ constexpr size_t fused_stream_smem() {
  return FusedRing<StateT>::TAIL_OFF + 1024;
}

template <typename StateT>
__global__ void __launch_bounds__(FusedRing<StateT>::WARPS * 32, 1)
    kda_fused_stream_kernel(const FusedArgs a, const __grid_constant__ CUtensorMap state_map, const int units) {
  using C = FusedRing<StateT>;
  using G = Strip<StateT, C::CW>;
  static_assert(fused_stream_smem<StateT>() <= 232448, "rings exceed the 227 KB shared memory of a CTA");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* smem = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  auto entry = [&](int e) { return smem + C::ACT_OFF + (size_t)e * F_ENTRY; };
  auto scal = [&](int e) { return reinterpret_cast<int4*>(entry(e) + F_SCAL); };
  uint64_t* sfull = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);  // state landed
  uint64_t* sempty = sfull + C::NS;                                   // consumers done with the stage
  uint64_t* afull = sempty + C::NS;                                   // activations landed
  uint64_t* aready = afull + C::NA;                                   // prologue results written
  uint64_t* aempty = aready + C::NA;                                  // consumers and epilogue done with it
  uint64_t* odone = aempty + C::NA;                                   // the unit's o written

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < C::NS; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], C::NW);
    }
    for (int e = 0; e < C::NA; ++e) {
      mbar_init(&afull[e], 1);
      mbar_init(&aready[e], 1);
      // consumers + the epilogue warp; the prologue has finished reading the
      // entry before it marks it ready, so it need not arrive
      mbar_init(&aempty[e], C::NW + 1);
      mbar_init(&odone[e], C::NW);
    }
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();

  const int P = gridDim.x;
  const int n_my = (units - (int)blockIdx.x + P - 1) / P;
  const int HD = a.H * kD;

  if (warp == C::NW) {
    // ---------------- loader: step k issues unit k's activations and unit k - LA's state ----------------
    int slot = -1;
    float beta = 0.f, A = 0.f;
    for (int k = 0; k < n_my + C::LA; ++k) {
      if (k < n_my) {
        if ((k & 31) == 0) {  // slot, beta and A of units k .. k+31, one per lane
          slot = -1;
          if (k + lane < n_my) {
            const int u = blockIdx.x + (k + lane) * P;
            const int h = u % a.H, r = u / a.H;
            slot = __ldg(a.idx + r);
            beta = sigmoidf_(load1(a.beta, (int64_t)r * a.b_rs + (int64_t)h * a.b_hs, KDA_DT_BF16));
            A = expf(__ldg(a.A_log + h));
          }
        }
        const int slot_t = __shfl_sync(0xffffffffu, slot, k & 31);
        const float beta_t = __shfl_sync(0xffffffffu, beta, k & 31);
        const float A_t = __shfl_sync(0xffffffffu, A, k & 31);
        const int e = k % C::NA;
        const uint32_t round = k / C::NA;
        const bool ok = round == 0 || mbar_wait(&aempty[e], (round - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_error(2u);
          return;
        }
        if (lane == 0) {
          const int u = blockIdx.x + k * P;
          const int h = u % a.H, r = u / a.H;
          const bool live = slot_t > 0 && slot_t < a.num_slots;
          *scal(e) = make_int4(live ? slot_t : -1, __float_as_int(beta_t), __float_as_int(A_t), 0);
          if (live) {
            unsigned char* act = entry(e);
            mbar_arrive_expect_tx(&afull[e], F_ACT);
            const __nv_bfloat16* xr = static_cast<const __nv_bfloat16*>(a.x) + (int64_t)r * a.x_rs + h * kD;
            const __nv_bfloat16* cs = static_cast<const __nv_bfloat16*>(a.conv_state) +
                                      (int64_t)slot_t * a.cs_slot_stride + h * kD;
#pragma unroll
            for (int sec = 0; sec < 3; ++sec) {
              bulk_load(act + F_X + sec * 256, xr + sec * HD, 256, &afull[e]);
#pragma unroll
              for (int tap = 0; tap < 3; ++tap)
                bulk_load(act + F_CS + (tap * 3 + sec) * 256, cs + tap * a.cs_tap_stride + sec * HD, 256, &afull[e]);
            }
            bulk_load(act + F_G,
                      static_cast<const __nv_bfloat16*>(a.gate) + (int64_t)r * a.g_rs + (int64_t)h * a.g_hs, 256,
                      &afull[e]);
            bulk_load(act + F_DT, a.dt_bias + h * kD, 512, &afull[e]);
            bulk_load(act + F_OG,
                      static_cast<const __nv_bfloat16*>(a.out_gate) + (int64_t)r * a.og_rs + (int64_t)h * a.og_hs,
                      256, &afull[e]);
          } else {
            mbar_arrive(&afull[e]);
          }
        }
        __syncwarp();
      }
      if (k >= C::LA) {
        const int js = k - C::LA;
        const int s = js % C::NS;
        const uint32_t round = js / C::NS;
        const bool ok = round == 0 || mbar_wait(&sempty[s], (round - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) {
          if (lane == 0) record_error(2u);
          return;
        }
        if (lane == 0) {
          const int slot_s = scal(js % C::NA)->x;  // written above by this thread; the entry is not reused yet
          if (slot_s >= 0) {
            mbar_arrive_expect_tx(&sfull[s], C::STATE_BYTES);
            tma_load_state<StateT>(smem + (size_t)s * C::STATE_BYTES, &state_map, (blockIdx.x + js * P) % a.H,
                                   slot_s, &sfull[s]);
          } else {
            mbar_arrive(&sfull[s]);
          }
        }
        __syncwarp();
      }
    }
    return;
  }

  if (warp == C::NW + 1 + C::NP) {
    // ---------------- epilogue: gated RMSNorm of each unit, lane l on columns 4l..4l+3 ----------------
    const float4 nw = __ldg(reinterpret_cast<const float4*>(a.norm_w) + lane);
    for (int j = 0; j < n_my; ++j) {
      const int e = j % C::NA;
      // the output gate arrived by bulk copy on the entry's afull barrier
      const bool ok = mbar_wait(&odone[e], (j / C::NA) & 1) && mbar_wait(&afull[e], (j / C::NA) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(1u);
        return;
      }
      const int u = blockIdx.x + j * P;
      __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.out) + (int64_t)u * kD + 4 * lane;  // u = r * H + h
      const unsigned char* act = entry(e);
      float y[4] = {0.f, 0.f, 0.f, 0.f};
      if (scal(e)->x >= 0) {
        const float4 o = reinterpret_cast<const float4*>(act + F_O)[lane];
        const float4 og = lds4(act + F_OG, 4 * lane, KDA_DT_BF16);
        const float ss = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
        const float rinv = rsqrtf(ss * (1.f / kD) + a.norm_eps);
        y[0] = o.x * rinv * nw.x * sigmoidf_(og.x);
        y[1] = o.y * rinv * nw.y * sigmoidf_(og.y);
        y[2] = o.z * rinv * nw.z * sigmoidf_(og.z);
        y[3] = o.w * rinv * nw.w * sigmoidf_(og.w);
      }
      store_out<4>(out, y);
      __syncwarp();
      if (lane == 0) mbar_arrive(&aempty[e]);
    }
    return;
  }

  if (warp > C::NW) {
    // ---------------- prologue warps (units round-robin): conv + SiLU, cache shift, coefficients ----------------
    // Lane l works on channels 4l..4l+3 of each section (q, k, v), the layout
    // of the coefficients.  The conv weights of a warp's next unit are loaded
    // while it works on the current one: an L2 read under the stream's DRAM
    // traffic takes about a microsecond.
    const int p = warp - C::NW - 1;
    float4 wv[3][4], wn[3][4];  // [section][tap]: current and next unit
    auto load_weights = [&](float4 (&w)[3][4], int j) {
      const int h = (blockIdx.x + j * P) % a.H;
#pragma unroll
      for (int sec = 0; sec < 3; ++sec)
#pragma unroll
        for (int tap = 0; tap < 4; ++tap)
          w[sec][tap] = __ldg(reinterpret_cast<const float4*>(a.conv_w + (int64_t)(sec * 4 + tap) * HD + h * kD) + lane);
    };
    if (p < n_my) load_weights(wn, p);
    for (int j = p; j < n_my; j += C::NP) {
#pragma unroll
      for (int sec = 0; sec < 3; ++sec)
#pragma unroll
        for (int tap = 0; tap < 4; ++tap) wv[sec][tap] = wn[sec][tap];
      if (j + C::NP < n_my) load_weights(wn, j + C::NP);
      const int e = j % C::NA;
      const bool ok = mbar_wait(&afull[e], (j / C::NA) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) record_error(1u);
        return;
      }
      const int4 sc = *scal(e);
      if (sc.x >= 0) {
        const int h = (blockIdx.x + j * P) % a.H;
        unsigned char* act = entry(e);
        // Raw taps, oldest first, then x: four bf16 channels per lane and section.
        // The shifted cache [tap1, tap2, x] goes back from registers.
        __nv_bfloat16* csg = static_cast<__nv_bfloat16*>(a.conv_state) + (int64_t)sc.x * a.cs_slot_stride + h * kD +
                             4 * lane;
        float4 y[3];
#pragma unroll
        for (int sec = 0; sec < 3; ++sec) {
          uint2 t[4];
#pragma unroll
          for (int tap = 0; tap < 3; ++tap)
            t[tap] = reinterpret_cast<const uint2*>(act + F_CS + (tap * 3 + sec) * 256)[lane];
          t[3] = reinterpret_cast<const uint2*>(act + F_X + sec * 256)[lane];
#pragma unroll
          for (int tap = 1; tap < 4; ++tap)
            *reinterpret_cast<uint2*>(csg + (int64_t)(tap - 1) * a.cs_tap_stride + sec * HD) = t[tap];
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int tap = 0; tap < 4; ++tap) {
            const float4 w = wv[sec][tap];
            acc.x = fmaf(w.x, bf_lo(t[tap].x), acc.x);
            acc.y = fmaf(w.y, bf_hi(t[tap].x), acc.y);
            acc.z = fmaf(w.z, bf_lo(t[tap].y), acc.z);
            acc.w = fmaf(w.w, bf_hi(t[tap].y), acc.w);
          }
          y[sec] = make_float4(acc.x * sigmoidf_(acc.x), acc.y * sigmoidf_(acc.y), acc.z * sigmoidf_(acc.z),
                               acc.w * sigmoidf_(acc.w));
        }
        reinterpret_cast<float4*>(act + F_V)[lane] = y[2];  // v, read by the consumers
        const float A = __int_as_float(sc.z);
        const float4 gr = lds4(act + F_G, 4 * lane, KDA_DT_BF16);
        const float4 dtb = reinterpret_cast<const float4*>(act + F_DT)[lane];
        float4 d;
        d.x = expf(log_decay(gr.x + dtb.x, A, a.gate_mode, a.lower_bound));
        d.y = expf(log_decay(gr.y + dtb.y, A, a.gate_mode, a.lower_bound));
        d.z = expf(log_decay(gr.z + dtb.z, A, a.gate_mode, a.lower_bound));
        d.w = expf(log_decay(gr.w + dtb.w, A, a.gate_mode, a.lower_bound));
        const float qk = token_coefficients(y[0], y[1], d, lane, reinterpret_cast<float4*>(act + F_COEF));
        if (lane == 0) scal(e)->w = __float_as_int(qk);
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&aready[e]);
    }
    return;
  }

  // ---------------- consumers ----------------
  const int col0 = warp * C::CW + (lane % G::LPR) * G::VEC;
  const int row0 = stream_row0<G::LPR>(lane);
  // the unit advances by P: with a bf16 state its head without a division
  constexpr bool kStepH = sizeof(StateT) == 2;
  const int h_step = P % a.H;
  int h_run = (int)(blockIdx.x % a.H);
  for (int j = 0; j < n_my; ++j, h_run = h_run + h_step >= a.H ? h_run + h_step - a.H : h_run + h_step) {
    const int s = j % C::NS, e = j % C::NA;
    const bool ok = mbar_wait(&sfull[s], (j / C::NS) & 1) && mbar_wait(&afull[e], (j / C::NA) & 1) &&
                    mbar_wait(&aready[e], (j / C::NA) & 1);
    if (!__all_sync(0xffffffffu, ok)) {
      if (lane == 0) record_error(1u);
      return;
    }
    const int4 sc = *scal(e);
    unsigned char* act = entry(e);
    if (sc.x >= 0) {
      const int h = kStepH ? h_run : (int)((blockIdx.x + j * P) % a.H);
      const unsigned char* st = smem + (size_t)s * C::STATE_BYTES;
      const float* vf = reinterpret_cast<const float*>(act + F_V);
      float* of = reinterpret_cast<float*>(act + F_O);  // o before the norm, for the epilogue warp
      typename Frag<StateT>::Raw S[G::PASSES];
      float2 dk[G::PASSES];
      float2 acc2_a[G::VEC / 2], acc2_b[G::VEC / 2];
      reduce_stage<StateT, G>(st, reinterpret_cast<const float4*>(act + F_COEF), row0, col0, S, dk, acc2_a, acc2_b);
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[s]);
      const float beta = __int_as_float(sc.y);
      const float qk = __int_as_float(sc.w);
      float u_[G::VEC];
      if constexpr (kStreamScatter<StateT, G>) {  // as in the T=1 kernel
        const int rg = lane / G::LPR;
        const float tot = strip_reduce_scatter<G>(acc2_a, acc2_b, rg);
        const float uc = rg < G::VEC ? beta * (vf[col0 + rg] - tot) : 0.f;
        const float u_lo = __shfl_xor_sync(0xffffffffu, uc, G::LPR * G::VEC);
        if (rg >= G::VEC) of[col0 + rg - G::VEC] = a.scale * (tot + qk * u_lo);
#pragma unroll
        for (int c = 0; c < G::VEC; ++c) u_[c] = __shfl_sync(0xffffffffu, uc, c * G::LPR + lane % G::LPR);
      } else {
        float acc_a[G::VEC], acc_b[G::VEC];
        strip_allreduce<G>(acc2_a, acc2_b, acc_a, acc_b);
#pragma unroll
        for (int jj = 0; jj < G::VEC; ++jj) u_[jj] = beta * (vf[col0 + jj] - acc_a[jj]);
        if (row0 == 0) {  // these lanes hold distinct columns
#pragma unroll
          for (int jj = 0; jj < G::VEC; jj += 4)
            reinterpret_cast<float4*>(of)[(col0 + jj) / 4] =
                make_float4(a.scale * (acc_b[jj] + qk * u_[jj]), a.scale * (acc_b[jj + 1] + qk * u_[jj + 1]),
                            a.scale * (acc_b[jj + 2] + qk * u_[jj + 2]), a.scale * (acc_b[jj + 3] + qk * u_[jj + 3]));
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&odone[e]);
        mbar_arrive(&aempty[e]);
      }
      StateT* sp = static_cast<StateT*>(a.state) + (int64_t)sc.x * a.slot_stride + (int64_t)h * kD * kD;
      update_store_regs<StateT, G>(sp, row0, col0, S, dk, u_);
    } else {
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&sempty[s]);
        mbar_arrive(&odone[e]);
        mbar_arrive(&aempty[e]);
      }
    }
  }
}

// Self-test of the bounded wait: one warp waits on a barrier that nothing
// completes; the wait gives up after kWaitNs and records bit 2.
__global__ void kda_selftest_wait_kernel() {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    mbar_fence_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_launch_dependents();
  const bool ok = mbar_wait(&bar, 0);
  if (!__all_sync(0xffffffffu, ok) && threadIdx.x == 0) record_error(4u);
}

// ---- host side ------------------------------------------------------------------------

namespace {

template <typename Kernel>
cudaError_t ensure_smem(Kernel k, size_t bytes, std::atomic<bool>* set_flags) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && !set_flags[dev].load(std::memory_order_acquire)) {
    // idempotent, so two host threads that both get here set the same value
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    set_flags[dev].store(true, std::memory_order_release);
  }
  return cudaSuccess;
}

template <typename StateT, int PARTS>
cudaError_t launch_t1_stream_typed(const T1Args& a, int sm_count, cudaStream_t s) {
  CUtensorMap map;
  if (!encode_state_map<StateT>(&map, a.state, a.H, a.num_slots, a.slot_stride)) return cudaErrorNotSupported;
  static std::atomic<bool> set[64];
  constexpr size_t smem = t1_stream_smem<StateT, PARTS>();
  cudaError_t e = ensure_smem(kda_t1_stream_kernel<StateT, PARTS>, smem, set);
  if (e != cudaSuccess) return e;
  const int items = a.B * a.H * PARTS;
  const int grid = items < sm_count ? items : sm_count;
  return launch_pdl(kda_t1_stream_kernel<StateT, PARTS>, dim3(grid),
                    dim3((T1StreamP<StateT, PARTS>::NW + 1 + t1_np<PARTS>()) * 32), smem, s, 1, a, map, items);
}

template <typename StateT>
cudaError_t launch_fused_stream_typed(const FusedArgs& a, int sm_count, cudaStream_t s) {
  CUtensorMap map;
  if (!encode_state_map<StateT>(&map, a.state, a.H, a.num_slots, a.slot_stride)) return cudaErrorNotSupported;
  static std::atomic<bool> set[64];
  constexpr size_t smem = fused_stream_smem<StateT>();
  cudaError_t e = ensure_smem(kda_fused_stream_kernel<StateT>, smem, set);
  if (e != cudaSuccess) return e;
  const int units = a.rows * a.H;
  const int grid = units < sm_count ? units : sm_count;
  return launch_pdl(kda_fused_stream_kernel<StateT>, dim3(grid),
                    dim3(FusedRing<StateT>::WARPS * 32), smem, s, 1, a, map, units);
}

}  // namespace

cudaError_t launch_t1_stream(const T1Args& a, int state_dtype, int sm_count, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_t1_stream_typed<float, 1>(a, sm_count, s);
  return launch_t1_stream_typed<__nv_bfloat16, 2>(a, sm_count, s);
}

cudaError_t launch_fused_stream(const FusedArgs& a, int state_dtype, int sm_count, cudaStream_t s) {
  if (state_dtype == KDA_DT_F32) return launch_fused_stream_typed<float>(a, sm_count, s);
  return launch_fused_stream_typed<__nv_bfloat16>(a, sm_count, s);
}

cudaError_t launch_selftest_wait(cudaStream_t s) {
  kda_selftest_wait_kernel<<<1, 32, 0, s>>>();
  return cudaGetLastError();
}

cudaError_t read_device_error(unsigned int* flags, bool clear) {
  cudaError_t e = cudaMemcpyFromSymbol(flags, g_kda_device_error, sizeof(unsigned int));
  if (e != cudaSuccess || !clear) return e;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(unsigned int));
}

}  // namespace kda
