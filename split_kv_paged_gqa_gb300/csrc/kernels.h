// kernels.h - host/device interface between the C ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fd {

enum KvKind : int { KV_BF16 = 0, KV_I8 = 1, KV_I4 = 2 };

// Keys per split of a request with L keys: equal page-aligned chunks
// P * ceil(ceil(L / S) / P), but never fewer than chunk_min keys.
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

// Balanced split policy. A call asking for S splits per request cuts the
// batch's n_total pages (sum over requests of ceil(L_b / P)) into chunks of
//   cp = ceil(n_total / (B * S)) pages,
// and a request of n pages gets ceil(n / cp) splits (at least 1, at most
// s_cap), which then cut it into equal page-aligned chunks as split_chunk
// does. Every split of the batch holds about cp pages, whatever the length
// mix. With equal lengths, every request gets split_count(L, S) splits of
// split_chunk(L, S) keys: the same splits as the equal policy.
__host__ __device__ inline int balanced_chunk_pages(long long n_total, int B, int S) {
  const long long units = static_cast<long long>(B) * S;
  const long long cp = (n_total + units - 1) / units;
  return cp < 1 ? 1 : (cp > 0x7fffffffLL ? 0x7fffffff : static_cast<int>(cp));
}

// The split budget of a request with n pages (the S that split_chunk and
// split_count take for it).
__host__ __device__ inline int balanced_budget(int n_pages, int cp, int s_cap) {
  if (n_pages <= 0) return 1;
  const int s = static_cast<int>((static_cast<long long>(n_pages) + cp - 1) / cp);
  return s < s_cap ? s : s_cap;
}

// Stage 1: one CTA per (row tile, split, KV head, request).
// Equal policy: grid (row_tiles * S, Hkv, B). Balanced policy: a flat grid
// over (split unit, KV head, row tile), x = (u * Hkv + h) * row_tiles + rt,
// where units number the splits of the batch request by request; CTAs past
// the batch's last unit exit at once.
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
  int num_splits;                  // S (balanced policy: splits per request on average)
  int chunk_min;                   // minimum keys per split (0: none)
  int balanced;                    // 1: balanced split policy (see balanced_chunk_pages)
  int batch;                       // B
  int s_cap;                       // partial rows per output row in the workspace (>= splits of any request)
  float scale_log2;                // softmax_scale * log2(e)
  // split outputs: workspace rows [B, Tq, Hq, s_cap] of D floats (a request
  // with one non-empty split writes its final outputs directly instead)
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
  int balanced, s_cap;
  // the split geometry of stage 1: only the non-empty splits of a request are
  // read; a request with exactly one was written by stage 1 and is skipped
  const int *seqlens;
  int64_t sl_s;
  int log2_page, max_pages, chunk_min;
  void *out;
  int out_f32;
  int64_t o_sb, o_st, o_sh;
  float *lse;
  int64_t l_sb, l_st, l_sh;
};

// Decode metadata of a batch from a request-to-token pool (graph_metadata.cu).
struct MetaParams {
  const int *req_to_token;  // [pool_rows, pool_cols]
  int64_t rt_sr, rt_sc;     // element strides
  int64_t pool_rows, pool_cols;
  const void *pool_idx;     // [B] int32 or int64
  int idx64;
  int64_t idx_s;
  const int *seq_lens;      // [B]
  int64_t sl_s;
  int B, P, W;              // batch, page size, page-table width
  int q_mode;               // an fd_q_mode
  const int *q_in;          // preset: [B + 1] cu_seqlens_q; cumsum: [B] query tokens; strided: unused
  int64_t q_s;
  int q_stride;
  int *page_table;          // [B, W]
  int64_t pt_sb;
  int *cache_seqlens;       // [B]
  int *cu_k, *cu_q;         // [B + 1]
  unsigned *status;         // or null
};

cudaError_t launch_graph_metadata(const MetaParams &p, cudaStream_t stream);

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

// Stage 1 on the tcgen05 tensor cores for INT8 / INT4 caches with head_dim
// 128 (one row tile of up to 16 query rows per CTA, no fused merge).
cudaError_t stage1_tc_prepare(int kind);
cudaError_t launch_stage1_tc(int kind, bool fused, const CUtensorMap &tmk, const CUtensorMap &tmv,
                             const Stage1Params &p, dim3 grid, cudaStream_t stream);

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
