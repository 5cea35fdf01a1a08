// Packed fused speculative decode with per-token checkpoints: argument block
// and launcher.  Kept apart from kda_launch.h so the other kernels' sources
// do not change with it.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

// Conv + SiLU + KDA + gated RMSNorm over the ragged token rows of N packed
// sequences; checkpoint j of sequence n goes to slot idx[n * idx_rs + j].
struct PackedFusedArgs {
  const void* x; int64_t x_rs;                      // bf16 [R, 3*H*128], channel stride 1
  const float* conv_w;                              // [3, 4, H*128]
  void* conv_state;                                 // bf16, [slot][tap][channel]
  int64_t cs_slot_stride, cs_tap_stride;            // elements
  const void* gate; int64_t g_rs, g_hs;             // bf16 [R, H, 128]
  const void* beta; int64_t b_rs, b_hs;             // bf16 [R, H]
  const float* A_log; const float* dt_bias;
  const int32_t* qsl;                               // [N+1] query_start_loc
  const int32_t* idx; int64_t idx_rs; int32_t cols; // [N, cols] checkpoint slots
  const int32_t* accepted;                          // [N] num_accepted_tokens
  void* state; int64_t slot_stride; int32_t num_slots;
  const void* out_gate; int64_t og_rs, og_hs;       // bf16 [R, H, 128]
  const float* norm_w;                              // [128]
  void* out; int64_t o_rs;                          // bf16 [R, H, 128], head stride 128
  int32_t N, R, H;
  int32_t gate_mode;
  float lower_bound, norm_eps, scale;
};

// `cluster` CTAs (1, 2, 4 or 8) share each (sequence, head), one value slab
// each; with one, the grid is persistent (sized from `sms`).
cudaError_t launch_packed_fused(const PackedFusedArgs& a, int state_dtype, int cluster, int sms, cudaStream_t s);

}  // namespace kda
