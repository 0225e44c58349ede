// kernels.h - host/device interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fd {

enum KvKind : int { KV_BF16 = 0, KV_I8 = 1, KV_I4 = 2 };

// Keys per split of a request with L keys: equal page-aligned chunks
// P * ceil(ceil(L / S) / P), but never fewer than chunk_min keys. With
// chunk_min derived from the batch's max length, every non-empty split of
// every request holds about the same number of keys (load balance across a
// mixed-length batch); requests shorter than the max use fewer splits.
__host__ __device__ inline int split_chunk(int L, int S, int log2_page, int chunk_min) {
  const int per = (L + S - 1) / S;
  const int c = ((per + (1 << log2_page) - 1) >> log2_page) << log2_page;
  return c > chunk_min ? c : chunk_min;
}

// Non-empty splits of a request with L keys.
__host__ __device__ inline int split_count(int L, int S, int log2_page, int chunk_min) {
  if (L <= 0) return 0;
  const int c = split_chunk(L, S, log2_page, chunk_min);
  const int n = (L + c - 1) / c;
  return n < S ? n : S;
}

// Stage 1: one CTA per (row tile, split, KV head, request).
struct Stage1Params {
  const __nv_bfloat16 *q;          // [B, Tq, Hq, D]
  int64_t q_sb, q_st, q_sh;        // element strides of q (d stride is 1)
  const float *kv_scales;          // [2, N, P, Hkv, n_g] or null
  int64_t sc_sk, sc_sp, sc_ss, sc_sh;  // element strides (group stride is 1)
  const int *page_table;           // [B, W]
  int64_t pt_sb;
  const int *seqlens;              // [B]
  int64_t sl_s;
  int num_pages;                   // N
  int page_size;                   // P
  int log2_page;                   // log2(P)
  int max_pages;                   // W
  int Tq, Hq, Hkv, G, R, row_tiles;
  int num_splits;                  // S
  int chunk_min;                   // minimum keys per split (0: equal splits per request)
  float scale_log2;                // softmax_scale * log2(e)
  // split outputs (num_splits > 1): workspace rows [B, Tq, Hq, S] of D floats
  float *o_part;
  float *lse_part;
  // fused outputs (num_splits == 1)
  void *out;
  int out_f32;
  int64_t o_sb, o_st, o_sh;
  float *lse;
  int64_t l_sb, l_st, l_sh;
  unsigned *status;
  // Fused merge (num_splits > 1): one counter per (request, KV head, row
  // tile); the last split CTA to finish merges the tile. Null: stage 2 merges.
  unsigned *counters;
};

// Stage 2: one warp per (request, query token, query head).
struct Stage2Params {
  const float *o_part;
  const float *lse_part;
  int B, Tq, Hq, D, num_splits;
  // the split geometry of stage 1: only the non-empty splits of a request are read
  const int *seqlens;
  int64_t sl_s;
  int log2_page, max_pages, chunk_min;
  void *out;
  int out_f32;
  int64_t o_sb, o_st, o_sh;
  float *lse;
  int64_t l_sb, l_st, l_sh;
};

// Slots per TMA box of the stage-1 kernel: a box holds min(page_size, this)
// rows of one page and head.
int stage1_block_n(int kind, int head_dim);

// Raise the dynamic shared-memory limit of every stage-1 variant of (kind, D).
cudaError_t stage1_prepare(int kind, int head_dim);

// deep: the one-CTA-per-SM deep-ring variant (bf16 cache; ignored otherwise).
cudaError_t launch_stage1(int kind, int head_dim, bool fused, bool deep, const CUtensorMap &tmk,
                          const CUtensorMap &tmv, const Stage1Params &p, dim3 grid,
                          cudaStream_t stream);

cudaError_t launch_stage2(const Stage2Params &p, cudaStream_t stream, bool pdl);

// Per-kind entry points (one translation unit each).
cudaError_t stage1_prepare_bf16(int head_dim);
cudaError_t stage1_prepare_i8(int head_dim);
cudaError_t stage1_prepare_i4(int head_dim);
cudaError_t launch_stage1_bf16(int head_dim, bool fused, bool deep, const CUtensorMap &tmk,
                               const CUtensorMap &tmv, const Stage1Params &p, dim3 grid,
                               cudaStream_t stream);
cudaError_t launch_stage1_i8(int head_dim, bool fused, bool deep, const CUtensorMap &tmk,
                             const CUtensorMap &tmv, const Stage1Params &p, dim3 grid,
                             cudaStream_t stream);
cudaError_t launch_stage1_i4(int head_dim, bool fused, bool deep, const CUtensorMap &tmk,
                             const CUtensorMap &tmv, const Stage1Params &p, dim3 grid,
                             cudaStream_t stream);

}  // namespace fd
