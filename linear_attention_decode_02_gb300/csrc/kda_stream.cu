// Persistent streaming T=1 decode: one CTA per SM walks its share of the
// (row, head) units through a ring of shared-memory stages.
//
//   loader warp    per unit: the slot index, beta and A_log; TMA tensor
//                  copies of the 128 x 128 state block (128-byte swizzled,
//                  in 128-byte-wide column blocks) and bulk copies of the
//                  unit's q, k, v, raw gate and dt_bias vectors, all
//                  completing on the stage's `full` barrier.
//   prologue warp  per unit: L2 norms, gate and decay of the 128 key
//                  channels once, into the stage's coefficient array
//                  (d k, d q, d, k) and q.k; then the `ready` barrier.
//   8 consumers    per unit: a 16-column strip over all 128 key rows from
//                  shared memory: the two k-reductions (in-thread plus xor
//                  shuffles), u and o, release of the stage (`empty`), then
//                  the update written straight from registers to global.
//
// Three (float32) or five (bfloat16) stages keep ~200 KB of state loads in
// flight per SM.  Every wait is bounded in time; a warp whose wait times out
// records a bit in g_kda_device_error and leaves (no barrier spans warps
// after set-up, so the others time out in turn instead of hanging).
#include <cuda.h>

#include "kda_async.cuh"
#include "kda_kernels.cuh"

namespace kda {

// bit 0: a stage-full/ready wait timed out; bit 1: a stage-free wait timed out.
__device__ unsigned int g_kda_device_error = 0;

template <typename StateT>
struct StreamCfg {
  static constexpr int NW = 8;                                  // consumer warps
  static constexpr int CW = 16;                                 // columns per consumer warp
  static constexpr int NSTAGE = sizeof(StateT) == 4 ? 3 : 5;
  static constexpr int BLK_COLS = 128 / sizeof(StateT);         // columns of one 128-byte swizzle block
  static constexpr int NBLK = kD / BLK_COLS;                    // 4 (f32) or 2 (bf16) blocks per unit
  static constexpr uint32_t BLK_BYTES = kD * 128;               // 128 rows x 128 bytes
  static constexpr uint32_t STATE_BYTES = NBLK * BLK_BYTES;
  static constexpr uint32_t ACT_SLOT = 512;                     // one 128-vector, up to float32
  static constexpr uint32_t STAGE_BYTES = ((STATE_BYTES + 5 * ACT_SLOT + 1023) / 1024) * 1024;
  static constexpr size_t COEF_OFF = (size_t)NSTAGE * STAGE_BYTES;
  static constexpr size_t SCAL_OFF = COEF_OFF + (size_t)NSTAGE * kD * sizeof(float4);
  static constexpr size_t BAR_OFF = SCAL_OFF + (size_t)NSTAGE * sizeof(int4);
  static constexpr size_t SMEM = BAR_OFF + 3 * NSTAGE * sizeof(uint64_t) + 1024;  // + base alignment
  static_assert(CW * NW == kD, "consumers cover the 128 value columns");
  static_assert(SMEM <= 232448, "stages exceed the 227 KB shared memory of a CTA");
};

// Lane -> first key row of its fragments, chosen so that the rows read by
// one quarter-warp differ in bit 2 (f32: 2 rows) or bits 1-2 (bf16: 4 rows):
// under the 128-byte swizzle those rows' chunks land in distinct banks.
template <typename StateT>
__device__ __forceinline__ int stream_row0(int lane);
template <>
__device__ __forceinline__ int stream_row0<float>(int lane) {  // LPR 4, 8 rows per instruction
  return (lane >> 3) + ((lane >> 2) & 1) * 4;
}
template <>
__device__ __forceinline__ int stream_row0<__nv_bfloat16>(int lane) {  // LPR 2, 16 rows per instruction
  return ((lane >> 1) & 3) * 2 + ((lane >> 3) & 1) + ((lane >> 4) & 1) * 8;
}

// Byte offset of the 16-byte chunk holding (row, col) in a swizzled stage.
template <typename StateT>
__device__ __forceinline__ uint32_t swz_offset(int row, int col) {
  using C = StreamCfg<StateT>;
  const int blk = col / C::BLK_COLS;
  const int chunk = (col % C::BLK_COLS) * (int)sizeof(StateT) / 16;
  return blk * C::BLK_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4);
}

__device__ __forceinline__ float4 lds4(const unsigned char* base, int i, int dtype) {
  if (dtype == KDA_DT_F32) return reinterpret_cast<const float4*>(base)[i >> 2];
  const uint2 u = reinterpret_cast<const uint2*>(base)[i >> 2];
  return make_float4(bf_lo(u.x), bf_hi(u.x), bf_lo(u.y), bf_hi(u.y));
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int x, int y, int z, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], "
      "[%5];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
      : "memory");
}

template <typename StateT>
__global__ void __launch_bounds__((StreamCfg<StateT>::NW + 2) * 32, 1)
    kda_t1_stream_kernel(const T1Args a, const __grid_constant__ CUtensorMap state_map, const int units) {
  using C = StreamCfg<StateT>;
  using G = Strip<StateT, C::CW>;
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
    // ---------------- loader ----------------
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
        if (!__all_sync(0xffffffffu, ok)) {
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
#pragma unroll
            for (int blk = 0; blk < C::NBLK; ++blk)
              tma_load_3d(st + blk * C::BLK_BYTES, &state_map, blk * C::BLK_COLS, h * kD, slot_t, &full[s]);
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

  if (warp == C::NW + 1) {
    // ---------------- prologue: the unit's per-key-channel coefficients, once ----------------
    for (int j = 0; j < n_my; ++j) {
      const int s = j % C::NSTAGE;
      const bool ok = mbar_wait(&full[s], (j / C::NSTAGE) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        if (lane == 0) atomicOr(&g_kda_device_error, 1u);
        return;
      }
      const int4 sc = scal[s];
      if (sc.x >= 0) {
        const unsigned char* act = smem + (size_t)s * C::STAGE_BYTES + C::STATE_BYTES;
        const float A = __int_as_float(sc.z);
        const float4 q = lds4(act, 4 * lane, a.qkv_dtype);
        const float4 k = lds4(act + C::ACT_SLOT, 4 * lane, a.qkv_dtype);
        const float4 gr = lds4(act + 3 * C::ACT_SLOT, 4 * lane, a.gate_dtype);
        const float4 dtb = reinterpret_cast<const float4*>(act + 4 * C::ACT_SLOT)[lane];
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

  // ---------------- consumers ----------------
  const int col0 = warp * C::CW + (lane % G::LPR) * G::VEC;
  const int row0 = stream_row0<StateT>(lane);
  for (int j = 0; j < n_my; ++j) {
    const int s = j % C::NSTAGE;
    const uint32_t par = (j / C::NSTAGE) & 1;
    const bool ok = mbar_wait(&full[s], par) && mbar_wait(&ready[s], par);
    if (!__all_sync(0xffffffffu, ok)) {
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
    const float4* coef = coef_all + s * kD;
    float vv[G::VEC];
#pragma unroll
    for (int jj = 0; jj < G::VEC; jj += 4) {
      const float4 t = lds4(st + C::STATE_BYTES + 2 * C::ACT_SLOT, col0 + jj, a.qkv_dtype);
      vv[jj] = t.x; vv[jj + 1] = t.y; vv[jj + 2] = t.z; vv[jj + 3] = t.w;
    }
    // k-reductions; the decay and key coefficients of each row stay in registers
    typename Frag<StateT>::Raw S[G::PASSES];
    float2 dk[G::PASSES];
    float acc_a[G::VEC], acc_b[G::VEC];
#pragma unroll
    for (int jj = 0; jj < G::VEC; ++jj) { acc_a[jj] = 0.f; acc_b[jj] = 0.f; }
#pragma unroll
    for (int i = 0; i < G::PASSES; ++i) {
      const int r = row0 + i * G::RPI;
      S[i] = *reinterpret_cast<const typename Frag<StateT>::Raw*>(st + swz_offset<StateT>(r, col0));
      const float4 c = coef[r];
      dk[i] = make_float2(c.z, c.w);
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) {
        const float x = Frag<StateT>::get(S[i], jj);
        acc_a[jj] = fmaf(c.x, x, acc_a[jj]);
        acc_b[jj] = fmaf(c.y, x, acc_b[jj]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);  // this warp no longer reads the stage
#pragma unroll
    for (int o = G::LPR; o < 32; o <<= 1) {
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) {
        acc_a[jj] += __shfl_xor_sync(0xffffffffu, acc_a[jj], o);
        acc_b[jj] += __shfl_xor_sync(0xffffffffu, acc_b[jj], o);
      }
    }
    const float beta = __int_as_float(sc.y);
    const float qk = __int_as_float(sc.w);
    float u_[G::VEC], o[G::VEC];
#pragma unroll
    for (int jj = 0; jj < G::VEC; ++jj) {
      u_[jj] = beta * (vv[jj] - acc_a[jj]);
      o[jj] = a.scale * (acc_b[jj] + qk * u_[jj]);
    }
    StateT* sp = static_cast<StateT*>(a.state) + (int64_t)sc.x * a.slot_stride + (int64_t)h * kD * kD;
#pragma unroll
    for (int i = 0; i < G::PASSES; ++i) {
      float y[G::VEC];
#pragma unroll
      for (int jj = 0; jj < G::VEC; ++jj) y[jj] = fmaf(dk[i].x, Frag<StateT>::get(S[i], jj), dk[i].y * u_[jj]);
      Frag<StateT>::store(sp + (row0 + i * G::RPI) * kD + col0, Frag<StateT>::pack(y));
    }
    if (row0 == 0) store_out<G::VEC>(out + col0, o);
  }
}

// ---- host side ------------------------------------------------------------------------

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      p = nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

template <typename StateT>
cudaError_t launch_stream_typed(const T1Args& a, int sm_count, cudaStream_t s) {
  using C = StreamCfg<StateT>;
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return cudaErrorNotSupported;
  // The pool as a 3-d tensor [num_slots][H*128 rows][128 columns]; a box is
  // one 128-byte-wide column block of one (slot, head) state.
  CUtensorMap map;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)a.H * kD, (cuuint64_t)a.num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * sizeof(StateT), (cuuint64_t)a.slot_stride * sizeof(StateT)};
  const cuuint32_t box[3] = {(cuuint32_t)C::BLK_COLS, (cuuint32_t)kD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r =
      enc(&map, sizeof(StateT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, a.state,
          dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;

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
  kda_t1_stream_kernel<StateT><<<grid, (C::NW + 2) * 32, C::SMEM, s>>>(a, map, units);
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
