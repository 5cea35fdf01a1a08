// Packed speculative (T >= 1, ragged cu_seqlens) decode: kernel instantiations and launcher.
#include "kda_kernels.cuh"

namespace kda {

namespace {

template <typename StateT, int CW, int NW, bool VERIFY>
cudaError_t launch_spec_variant(const SpecArgs& a, cudaStream_t s) {
  constexpr int SPLIT = kD / (CW * NW);
  const int64_t blocks = (int64_t)(a.N + 1) * a.H * SPLIT;  // slice N zeroes padding rows
  kda_spec_kernel<StateT, CW, NW, VERIFY><<<dim3((unsigned)blocks), dim3(NW * 32), 0, s>>>(a);
  return cudaGetLastError();
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
