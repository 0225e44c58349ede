// graph_metadata.cu - the decode metadata of a batch, rebuilt on the device
// in one launch (sm_103a).
//
// "sglang PR 29843" (section 功能与动机) rebuilds cache_seqlens, cu_seqlens_k /
// cu_seqlens_q and page_table on every CUDA-graph replay with about 25 small
// host-dispatched operations, 0.7-1.0 ms of host time on some CPUs; its fix
// (section 实现拆解, item 1) computes all of them in one kernel with one
// program per batch row, three q modes (preset / cumsum / strided) and a -1
// sentinel guard. This is that step, ahead of the decode path, as a CUDA
// kernel: CTA b builds row b.
//
//  * cache_seqlens[b] = seq_lens[b]; 0 for a padding row (pool index < 0).
//  * page_table[b, j] = req_to_token[r, j * P] / P for j < ceil(L_b / P) (a
//    request's pages start on page boundaries), -1 past the last page, for an
//    unallocated slot (< 0) and on a padding row.
//  * cu_seqlens_k[b] = sum of cache_seqlens over rows < b (b = 0 .. B).
//  * cu_seqlens_q: preset (copied), cumsum (exclusive prefix sum of per-row
//    query tokens, 0 on a padding row) or strided (b * q_stride).
// Warp 0 of CTA b forms its two prefix sums over rows < b from the inputs
// directly (B is at most a few hundred rows), so no second pass is needed.
// Pool rows past the pool and pages past the pool row's columns are recorded
// in the status word and read as padding / -1.
#include <cuda_runtime.h>
#include <stdint.h>

#include "fd.h"
#include "kernels.h"

namespace fd {

namespace {

constexpr int kMetaThreads = 512;

__device__ __forceinline__ int64_t load_index(const void *p, int is64, int64_t i) {
  return is64 ? static_cast<const int64_t *>(p)[i] : static_cast<const int *>(p)[i];
}

__global__ void __launch_bounds__(kMetaThreads) fd_graph_metadata_kernel(const MetaParams p) {
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int64_t r_raw = load_index(p.pool_idx, p.idx64, b * p.idx_s);
  const bool pad = r_raw < 0;
  const bool out_of_pool = r_raw >= p.pool_rows;
  if (out_of_pool && tid == 0 && p.status) atomicOr(p.status, FD_DEVSTAT_BAD_PAGE);
  const bool live = !pad && !out_of_pool;
  int L = live ? p.seq_lens[b * p.sl_s] : 0;
  if (L < 0) L = 0;

  if (tid < 32) {
    // exclusive prefix sums over rows < b (and, for the last row, through b)
    long long sk = 0, sq = 0;
    for (int i = lane; i < b; i += 32) {
      const int64_t ri = load_index(p.pool_idx, p.idx64, i * p.idx_s);
      const bool li = ri >= 0 && ri < p.pool_rows;
      const int Li = li ? max(p.seq_lens[i * p.sl_s], 0) : 0;
      sk += Li;
      if (p.q_mode == FD_QMODE_CUMSUM) sq += li ? p.q_in[i * p.q_s] : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      sk += __shfl_xor_sync(0xffffffffu, sk, o);
      sq += __shfl_xor_sync(0xffffffffu, sq, o);
    }
    if (lane == 0) {
      p.cu_k[b] = static_cast<int>(sk);
      if (p.q_mode == FD_QMODE_CUMSUM) p.cu_q[b] = static_cast<int>(sq);
      else if (p.q_mode == FD_QMODE_STRIDED) p.cu_q[b] = b * p.q_stride;
      else p.cu_q[b] = p.q_in[b * p.q_s];
      p.cache_seqlens[b] = L;
      if (b == p.B - 1) {  // the closing entries
        p.cu_k[p.B] = static_cast<int>(sk + L);
        if (p.q_mode == FD_QMODE_CUMSUM) p.cu_q[p.B] = static_cast<int>(sq + (live ? p.q_in[b * p.q_s] : 0));
        else if (p.q_mode == FD_QMODE_STRIDED) p.cu_q[p.B] = p.B * p.q_stride;
        else p.cu_q[p.B] = p.q_in[p.B * p.q_s];
      }
    }
  }

  // page-table row b
  const int n_pages = live ? (L + p.P - 1) / p.P : 0;
  if (live && n_pages > p.W && tid == 0 && p.status) atomicOr(p.status, FD_DEVSTAT_SEQLEN_OVERFLOW);
  const int *row = live ? p.req_to_token + r_raw * p.rt_sr : nullptr;
  bool past_cols = false;
  for (int j = tid; j < p.W; j += kMetaThreads) {
    int v = -1;
    if (j < n_pages) {
      const int64_t pos = static_cast<int64_t>(j) * p.P;
      if (pos < p.pool_cols) {
        const int slot = row[pos * p.rt_sc];
        v = slot >= 0 ? slot / p.P : -1;
      } else {
        past_cols = true;
      }
    }
    p.page_table[b * p.pt_sb + j] = v;
  }
  if (__syncthreads_or(past_cols) && tid == 0 && p.status) atomicOr(p.status, FD_DEVSTAT_BAD_PAGE);
}

}  // namespace

cudaError_t launch_graph_metadata(const MetaParams &p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  fd_graph_metadata_kernel<<<p.B, kMetaThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace fd
