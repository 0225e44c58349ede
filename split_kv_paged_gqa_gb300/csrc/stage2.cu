// stage2.cu - merge of the KV splits by log-sum-exp (sm_103a).
//
// The stage-2 kernel of "feat(autotune): separate general and decode attention
// warmup" (LightLLM PR 1549), section "Covered decode kernels" (MTP attention
// stages 1 and 2; section "Validation": stage-2 inputs reused). For one output
// row (request, query token, query head) with split partials (o_s, lse_s):
//   M = max_s lse_s,  w_s = exp(lse_s - M),  out = sum_s w_s o_s / sum_s w_s,
//   lse = M + ln(sum_s w_s).
// Only the non-empty splits of the row's request (split_count of its length
// and split budget) are read; a request with exactly one was written by
// stage 1 directly and is skipped here. Splits with lse_s = -inf (a row with
// no visible key in them) carry weight 0 (their partial is a finite 0); a row
// whose splits are all empty gets out = 0, lse = -inf. One warp per row; the
// split partials of a row are contiguous (nv x D fp32, at a stride of s_cap
// rows per output row) and read coalesced.
// Launched with programmatic dependent launch: the grid may start while stage 1
// drains and waits on griddepcontrol before touching the workspace.
#include <cuda_bf16.h>
#include <math.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitmap.cuh"

namespace fd {

// Rows per CTA: small CTAs spread a short merge over more SMs. A batch-1 ×
// 32K call (64 rows of 16 partials) measured 24.0 us with 8-warp CTAs, 23.75
// with 4, 23.4 with 2 and 23.45 with 1 (same process; batch 64 and the
// mixed-length batch unchanged within 0.2 %).
constexpr int kS2Warps = 2;

template <int D>
__global__ void __launch_bounds__(kS2Warps * 32) fd_stage2_kernel(const __grid_constant__ Stage2Params p) {
  // The next kernel may be scheduled at once: a programmatic dependent waits
  // for this grid to complete (after its own wait below) before it reads
  // anything this grid writes.
  griddep_launch_dependents();
  constexpr int VPL = D / 32;  // values per lane
  const int row = blockIdx.x * kS2Warps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= p.B * p.Tq * p.Hq) return;
  const int b_row = row / (p.Hq * p.Tq);
  const int cap = p.max_pages << p.log2_page;
  // The length is read before the wait: stage 1 triggers this grid only after
  // its own dependency wait, so whatever wrote the lengths before stage 1 has
  // completed by now, and stage 1 does not write them. It comes from L2, not
  // from a line this SM's L1 may still hold from an earlier kernel.
  // The balanced split map is rebuilt from all the lengths, before the wait too.
  const int L = load_len<false>(p.seqlens, p.sl_s, b_row, cap);  // clamped as stage 1 clamps it
  int S_req = p.num_splits;
  if (p.balanced) {
    const int cp = balanced_chunk_pages(batch_pages<false>(p.seqlens, p.sl_s, p.B, cap, p.log2_page, lane), p.B,
                                        p.num_splits);
    S_req = balanced_budget((L + (1 << p.log2_page) - 1) >> p.log2_page, cp, p.s_cap);
  }
  const int nv = split_count(L, S_req, p.log2_page, p.chunk_min);  // splits stage 1 wrote
  if (nv == 1) return;  // stage 1 wrote this row's outputs
  griddep_wait();
  const float *lp = p.lse_part + static_cast<int64_t>(row) * p.s_cap;
  const float *op = p.o_part + static_cast<int64_t>(row) * p.s_cap * D + lane * VPL;
  // The LSEs and the first 16 partials are requested together (one round
  // trip for up to 16 splits); the weights are applied once both are in.
  constexpr int U = 16;
  float v[U][VPL];
#pragma unroll
  for (int u = 0; u < U; ++u) {
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[u][i] = 0.f;
    if (u < nv) {
      if constexpr (VPL == 4) {
        const float4 t = *reinterpret_cast<const float4 *>(op + u * D);
        v[u][0] = t.x;
        v[u][1] = t.y;
        v[u][2] = t.z;
        v[u][3] = t.w;
      } else {
        const float2 t = *reinterpret_cast<const float2 *>(op + u * D);
        v[u][0] = t.x;
        v[u][1] = t.y;
      }
    }
  }
  const float l0 = lane < nv ? lp[lane] : -INFINITY;
  const float l1 = lane + 32 < nv ? lp[lane + 32] : -INFINITY;
  float M = fmaxf(l0, l1);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  const float w0 = (l0 == -INFINITY) ? 0.f : expf(l0 - M);
  const float w1 = (l1 == -INFINITY) ? 0.f : expf(l1 - M);
  float Z = w0 + w1;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);

  float acc[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) acc[i] = 0.f;
  for (int s0 = 0; s0 < nv; s0 += U) {
    if (s0 > 0) {  // later groups of splits (more than 16)
#pragma unroll
      for (int u = 0; u < U; ++u) {
#pragma unroll
        for (int i = 0; i < VPL; ++i) v[u][i] = 0.f;
        if (s0 + u < nv) {
          if constexpr (VPL == 4) {
            const float4 t = *reinterpret_cast<const float4 *>(op + (s0 + u) * D);
            v[u][0] = t.x;
            v[u][1] = t.y;
            v[u][2] = t.z;
            v[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2 *>(op + (s0 + u) * D);
            v[u][0] = t.x;
            v[u][1] = t.y;
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int sp = s0 + u;
      const float wa = __shfl_sync(0xffffffffu, w0, sp & 31);
      const float wb = __shfl_sync(0xffffffffu, w1, sp & 31);
      const float w = sp < nv ? (sp < 32 ? wa : wb) : 0.f;  // empty splits carry weight 0
#pragma unroll
      for (int i = 0; i < VPL; ++i) acc[i] = fmaf(w, v[u][i], acc[i]);
    }
  }
  const float inv = Z > 0.f ? 1.f / Z : 0.f;
  const int hq = row % p.Hq;
  const int t = (row / p.Hq) % p.Tq;
  const int b = row / (p.Hq * p.Tq);
  const int64_t base = b * p.o_sb + t * p.o_st + hq * p.o_sh + lane * VPL;
  if (p.out_f32) {
    float *dst = reinterpret_cast<float *>(p.out) + base;
#pragma unroll
    for (int i = 0; i < VPL; ++i) dst[i] = acc[i] * inv;
  } else {
    __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + base;
#pragma unroll
    for (int i = 0; i < VPL; i += 2)
      *reinterpret_cast<uint32_t *>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
  }
  if (lane == 0 && p.lse) p.lse[b * p.l_sb + t * p.l_st + hq * p.l_sh] = Z > 0.f ? M + logf(Z) : -INFINITY;
}

cudaError_t launch_stage2(const Stage2Params &p, cudaStream_t stream, bool pdl) {
  const int rows = p.B * p.Tq * p.Hq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((rows + kS2Warps - 1) / kS2Warps);
  cfg.blockDim = dim3(kS2Warps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  if (p.D == 128) return cudaLaunchKernelEx(&cfg, fd_stage2_kernel<128>, p);
  if (p.D == 64) return cudaLaunchKernelEx(&cfg, fd_stage2_kernel<64>, p);
  return cudaErrorInvalidValue;
}

int stage1_block_n(int, int) { return 64; }

cudaError_t stage1_prepare(int kind, int head_dim) {
  cudaError_t e = cudaErrorInvalidValue;
  switch (kind) {
    case KV_BF16: return stage1_prepare_bf16(head_dim);
    case KV_I8: e = stage1_prepare_i8(head_dim); break;
    case KV_I4: e = stage1_prepare_i4(head_dim); break;
  }
  if (e == cudaSuccess && head_dim == 128) e = stage1_tc_prepare(kind);
  return e;
}

cudaError_t launch_stage1(int kind, int head_dim, bool fused, bool deep, const CUtensorMap &tmk,
                          const CUtensorMap &tmv, const Stage1Params &p, dim3 grid,
                          cudaStream_t stream) {
  switch (kind) {
    case KV_BF16: return launch_stage1_bf16(head_dim, fused, deep, tmk, tmv, p, grid, stream);
    case KV_I8: return launch_stage1_i8(head_dim, fused, deep, tmk, tmv, p, grid, stream);
    case KV_I4: return launch_stage1_i4(head_dim, fused, deep, tmk, tmv, p, grid, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace fd
