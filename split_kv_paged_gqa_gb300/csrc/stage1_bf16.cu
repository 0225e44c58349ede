// stage1_bf16.cu - stage-1 instantiations for one KV cache format (KV_BF16).
#include "stage1.cuh"

namespace fd {

cudaError_t stage1_prepare_bf16(int head_dim) {
  if (head_dim == 128) return stage1_prepare_t<KV_BF16, 128>();
  if (head_dim == 64) return stage1_prepare_t<KV_BF16, 64>();
  return cudaErrorInvalidValue;
}

cudaError_t launch_stage1_bf16(int head_dim, bool fused, bool deep, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const Stage1Params &p, dim3 grid, cudaStream_t stream) {
  if (head_dim == 128) return launch_stage1_t<KV_BF16, 128>(fused, deep, tmk, tmv, p, grid, stream);
  if (head_dim == 64) return launch_stage1_t<KV_BF16, 64>(fused, deep, tmk, tmv, p, grid, stream);
  return cudaErrorInvalidValue;
}

}  // namespace fd
