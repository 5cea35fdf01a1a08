// Fused conv + SiLU + KDA + gated RMSNorm decode: kernel instantiations and launcher.
#include "kda_kernels.cuh"

namespace kda {

cudaError_t launch_fused(const FusedArgs& a, int state_dtype, cudaStream_t s) {
  const int64_t blocks = (int64_t)a.rows * a.H;
  if (state_dtype == KDA_DT_F32) {
    kda_fused_kernel<float><<<dim3((unsigned)blocks), dim3(256), 0, s>>>(a);
  } else {
    kda_fused_kernel<__nv_bfloat16><<<dim3((unsigned)blocks), dim3(256), 0, s>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace kda
