// stage1_tc.cu - instantiations of the tcgen05 stage-1 kernel (INT8 / INT4
// KV caches, head_dim 128).
#include "stage1_tc.cuh"

namespace fd {

cudaError_t stage1_tc_prepare(int kind) {
  if (kind == KV_I8) return stage1_tc_prepare_t<KV_I8>();
  if (kind == KV_I4) return stage1_tc_prepare_t<KV_I4>();
  return cudaErrorInvalidValue;
}

cudaError_t launch_stage1_tc(int kind, bool fused, const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const Stage1Params &p, dim3 grid, cudaStream_t stream) {
  if (kind == KV_I8) return launch_stage1_tc_t<KV_I8>(fused, tmk, tmv, p, grid, stream);
  if (kind == KV_I4) return launch_stage1_tc_t<KV_I4>(fused, tmk, tmv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fd
