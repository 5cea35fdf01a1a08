// Internal interface between the host dispatcher (kda_api.cu) and the kernel
// translation units.  Plain structs of device pointers and element strides,
// validated on the host before any launch.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

enum : int { KDA_DT_F32 = 0, KDA_DT_BF16 = 1 };
enum : int { KDA_GATE_SOFTPLUS = 0, KDA_GATE_LOWER_BOUND = 1 };

// One T=1 step over B rows x H heads with split q / k / v activations
// (the packed front end is the same with strided views into one row).
struct T1Args {
  const void* q; const void* k; const void* v; const void* gate; const void* beta;
  int64_t q_rs, q_hs, k_rs, k_hs, v_rs, v_hs, g_rs, g_hs, b_rs, b_hs;  // element strides
  int32_t qkv_dtype, gate_dtype, beta_dtype;
  const float* A_log;     // [H]
  const float* dt_bias;   // [H*128]
  const int32_t* idx;     // [B]
  void* state;            // [num_slots, H, 128, 128]
  int64_t slot_stride;    // elements
  int32_t num_slots;
  void* out;              // bf16 [B, H, 128] contiguous
  int32_t B, H;
  int32_t gate_mode;
  float lower_bound, scale;
};

// Fused conv + SiLU + KDA + gated RMSNorm, one token per row.
struct FusedArgs {
  const void* x; int64_t x_rs;            // bf16 [rows, 3*H*128]
  const float* conv_w;                    // [3, 4, H*128]
  void* conv_state;                       // bf16, [slot][tap][channel]
  int64_t cs_slot_stride, cs_tap_stride;  // elements
  const void* gate; int64_t g_rs, g_hs;   // bf16 [rows, H, 128]
  const void* beta; int64_t b_rs, b_hs;   // bf16 [rows, H]
  const float* A_log; const float* dt_bias;
  const int32_t* idx;
  void* state; int64_t slot_stride; int32_t num_slots;
  const void* out_gate; int64_t og_rs, og_hs;  // bf16 [rows, H, 128]
  const float* norm_w;                    // [128]
  void* out;                              // bf16 [rows, H, 128]
  int32_t rows, H;
  int32_t gate_mode;
  float lower_bound, norm_eps, scale;
};

// Packed speculative decode over N ragged rows of R token rows.
struct SpecArgs {
  const void* q; const void* k; const void* v;
  int64_t q_rs, q_hs, k_rs, k_hs, v_rs, v_hs;
  int32_t qkv_dtype;
  const float* g; int64_t g_rs, g_hs;     // f32 [R, H, 128] log decay
  const void* beta; int64_t b_rs, b_hs; int32_t beta_dtype; int32_t beta_is_logit;
  const int32_t* cu;                      // [N+1]
  const int32_t* idx;                     // [N]
  void* state; int64_t slot_stride; int32_t num_slots;
  void* out;                              // bf16 [R, H, 128]
  int32_t N, R, H;
  float scale;
  // verify mode (state read-only): optional slot-indexed caches, contiguous
  float* corr;                            // [num_slots, H, t_cap, 128] u_t
  float* kg;                              // [num_slots, H, t_cap, 256] raw k | g
  int32_t t_cap;
};

// Launches kernel<<<grid, block, smem, s>>>(args...) with programmatic
// stream serialization: the grid may begin (launch, CTA placement, on-chip
// set-up) while the previous kernel on the stream drains; every kernel of this
// library executes pdl_wait() before its first global-memory access, so
// nothing the previous kernel writes is read early.  `cluster` > 1 adds a
// thread-block cluster of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              int cluster, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// Launchers: return the launch error (cudaSuccess on success).
cudaError_t launch_t1(const T1Args& a, int state_dtype, int split, cudaStream_t s);
// `cluster` CTAs (1, 2 or 4) share each (row, head), one value slab each.
cudaError_t launch_fused(const FusedArgs& a, int state_dtype, int cluster, cudaStream_t s);
cudaError_t launch_spec(const SpecArgs& a, int state_dtype, int split, bool verify, cudaStream_t s);

// Persistent streaming T=1 kernel (bulk copies into shared-memory stages);
// needs 16-byte aligned q / k / v / gate head vectors.
cudaError_t launch_t1_stream(const T1Args& a, int state_dtype, int sm_count, cudaStream_t s);

// Persistent streaming fused kernel; needs 16-byte aligned x rows, conv-cache
// slots, raw-gate and output-gate head vectors.
cudaError_t launch_fused_stream(const FusedArgs& a, int state_dtype, int sm_count, cudaStream_t s);

// Speculative decode (and verify) in the chunked tensor-core form, bfloat16
// state only: persistent, one CTA per SM (sized from `sm_count`).
cudaError_t launch_spec_mma(const SpecArgs& a, bool verify, int sm_count, cudaStream_t s);

// Reads (and optionally clears) the error word of the tensor-core
// speculative kernel: bit 3 = one of its waits timed out.
cudaError_t read_mma_error(unsigned int* flags, bool clear);

// One warp waiting on a barrier nothing completes (bounded-wait self-test).
cudaError_t launch_selftest_wait(cudaStream_t s);

// Reads (and optionally clears) the device error word of the streaming
// kernels: bit 0 = a stage-full wait timed out, bit 1 = a stage-free wait.
cudaError_t read_device_error(unsigned int* flags, bool clear);

// Splits with a compiled kernel (1, 2, 4, 8, 16).
bool split_supported(int split);

}  // namespace kda
