// Shared pieces of the persistent streaming kernels: stage geometry, the
// 128-byte swizzle of TMA-loaded state blocks, shared-memory activation
// reads, the 3-d tensor-map load, and the tensor-map encoder entry point.
#pragma once

#include <cuda.h>

#include "kda_async.cuh"
#include "kda_kernels.cuh"

namespace kda {

// A state block (128 x 128) arrives as NBLK column blocks of 128 rows x 128
// bytes, each 128-byte swizzled (16-byte chunk index XOR row % 8).
template <typename StateT>
struct SwzCfg {
  static constexpr int BLK_COLS = 128 / sizeof(StateT);  // 32 (f32) or 64 (bf16) columns
  static constexpr int NBLK = kD / BLK_COLS;             // 4 (f32) or 2 (bf16) blocks per state
  static constexpr uint32_t BLK_BYTES = kD * 128;        // 128 rows x 128 bytes
  static constexpr uint32_t STATE_BYTES = NBLK * BLK_BYTES;
};

// Ring of NSTAGE stages: [state part | ACT_BYTES of unit vectors] each
// (1024-byte aligned), then per stage a coefficient array (128 float4),
// DERIVED_BYTES of prologue results, scalars (int4) and three mbarriers.
// PARTS > 1 splits a unit's value columns into that many work items of
// 128 / PARTS columns (whole TMA column blocks), each staged on its own; the
// consumer warps then form PARTS groups of NW / PARTS warps that take the
// items in turn, each warp keeping a 16-column strip (whole 32-byte row
// segments for bf16, so every state store fills a sector).
template <typename StateT, uint32_t ACT_BYTES, int NSTAGE_, uint32_t DERIVED_BYTES = 0, int PARTS_ = 1>
struct StageCfg : SwzCfg<StateT> {
  static constexpr int NSTAGE = NSTAGE_;
  static constexpr int PARTS = PARTS_;
  static constexpr int NW = 8;            // consumer warps
  static constexpr int CW = 16;           // columns per consumer warp
  static constexpr int GROUP_WARPS = NW / PARTS;  // consumer warps per item
  static constexpr int PART_COLS = kD / PARTS;
  static constexpr int PART_BLKS = SwzCfg<StateT>::NBLK / PARTS;  // TMA column blocks of a part
  static constexpr uint32_t PART_BYTES = SwzCfg<StateT>::STATE_BYTES / PARTS;
  static_assert(PART_BLKS >= 1 && PART_BLKS * PARTS == SwzCfg<StateT>::NBLK, "parts must be whole column blocks");
  static constexpr uint32_t STAGE_BYTES = ((PART_BYTES + ACT_BYTES + 1023) / 1024) * 1024;
  static constexpr size_t COEF_OFF = (size_t)NSTAGE * STAGE_BYTES;
  static constexpr size_t DERIVED_OFF = COEF_OFF + (size_t)NSTAGE * kD * sizeof(float4);
  static constexpr size_t SCAL_OFF = DERIVED_OFF + (size_t)NSTAGE * DERIVED_BYTES;
  static constexpr size_t BAR_OFF = SCAL_OFF + (size_t)NSTAGE * sizeof(int4);
  static constexpr size_t TAIL_OFF = BAR_OFF + 3 * NSTAGE * sizeof(uint64_t);  // kernel-specific extras
  static_assert(CW * GROUP_WARPS * PARTS == kD, "a consumer group covers a part's value columns");
};

// Lane -> first key row of its fragments for LPR lanes per row segment,
// chosen so that the rows read by one quarter-warp differ in bit 2 (4 lanes
// per row: 2 rows), bits 1-2 (2 lanes: 4 rows) or bits 0-2 (1 lane: 8 rows):
// under the 128-byte swizzle those rows' chunks land in distinct banks.
template <int LPR>
__device__ __forceinline__ int stream_row0(int lane);
template <>
__device__ __forceinline__ int stream_row0<4>(int lane) {  // 8 rows per instruction
  return (lane >> 3) + ((lane >> 2) & 1) * 4;
}
template <>
__device__ __forceinline__ int stream_row0<2>(int lane) {  // 16 rows per instruction
  return ((lane >> 1) & 3) * 2 + ((lane >> 3) & 1) + ((lane >> 4) & 1) * 8;
}
template <>
__device__ __forceinline__ int stream_row0<1>(int lane) {  // 32 rows per instruction
  return lane;
}

// Byte offset of the 16-byte chunk holding (row, col) in a swizzled state block.
template <typename StateT>
__device__ __forceinline__ uint32_t swz_offset(int row, int col) {
  using C = SwzCfg<StateT>;
  const int blk = col / C::BLK_COLS;
  const int chunk = (col % C::BLK_COLS) * (int)sizeof(StateT) / 16;
  return blk * C::BLK_BYTES + row * 128 + ((chunk ^ (row & 7)) << 4);
}

// Four consecutive elements (float32 or bfloat16) of a shared-memory vector.
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

// All the unit's state blocks into `dst` (a 1024-byte aligned stage).
template <typename StateT>
__device__ __forceinline__ void tma_load_state(unsigned char* dst, const CUtensorMap* map, int h, int slot,
                                               uint64_t* bar) {
  using C = SwzCfg<StateT>;
#pragma unroll
  for (int blk = 0; blk < C::NBLK; ++blk) tma_load_3d(dst + blk * C::BLK_BYTES, map, blk * C::BLK_COLS, h * kD, slot, bar);
}

// Column sums of a 16-column strip's two k-reductions by reduce-scatter over
// the strip's RPI row groups (2 VEC of them): at each level a lane keeps one
// half of its values and adds its partner's copy of that half, so the lane of
// row group rg ends holding value rg of (a_0 .. a_{VEC-1}, b_0 .. b_{VEC-1})
// summed over all rows, after RPI - 1 shuffles instead of log2(RPI) * 2 VEC.
template <typename G>
__device__ __forceinline__ float strip_reduce_scatter(const float2 (&a2)[G::VEC / 2], const float2 (&b2)[G::VEC / 2],
                                                      int rg) {
  constexpr int NV = 2 * G::VEC;
  static_assert(NV == G::RPI, "one value per row group");
  float v[NV];
#pragma unroll
  for (int p = 0; p < G::VEC / 2; ++p) {
    v[2 * p] = a2[p].x; v[2 * p + 1] = a2[p].y;
    v[G::VEC + 2 * p] = b2[p].x; v[G::VEC + 2 * p + 1] = b2[p].y;
  }
  constexpr int LEVELS = NV == 8 ? 3 : (NV == 16 ? 4 : 0);
  static_assert(LEVELS > 0, "8 or 16 row groups");
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

// ---- host side -----------------------------------------------------------------------

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled() {
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

// The pool [num_slots][H*128 rows][128 columns] as a 3-d tensor map whose box
// is one 128-byte-wide column block of one (slot, head) state.
template <typename StateT>
inline bool encode_state_map(CUtensorMap* map, void* state, int H, int num_slots, int64_t slot_stride) {
  EncodeTiledFn enc = encode_tiled();
  if (enc == nullptr) return false;
  using C = SwzCfg<StateT>;
  const cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)H * kD, (cuuint64_t)num_slots};
  const cuuint64_t strides[2] = {(cuuint64_t)kD * sizeof(StateT), (cuuint64_t)slot_stride * sizeof(StateT)};
  const cuuint32_t box[3] = {(cuuint32_t)C::BLK_COLS, (cuuint32_t)kD, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return enc(map, sizeof(StateT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, state,
             dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace kda
