// splitmap.cuh - the balanced split map, derived on the device from cache_seqlens.
//
// Balanced policy (see balanced_chunk_pages in kernels.h): every split of the
// batch holds about cp = ceil(n_total / (B * S)) pages, so a long request gets
// more splits than a short one and a mixed-length batch keeps its CTAs
// evenly loaded. Nothing is precomputed on the host: each CTA (and each merge
// warp) reads the B lengths and rebuilds the map, so a captured call stays
// valid for any lengths at replay. These are warp-collective helpers: all 32
// lanes must call them with the same arguments.
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace fd {

template <bool RELAXED>
__device__ __forceinline__ int load_len_raw(const int *seqlens, int64_t sl_s, int i) {
  return RELAXED ? ld_relaxed_gpu(seqlens + i * sl_s) : ld_cg(seqlens + i * sl_s);
}

__device__ __forceinline__ int clamp_len(int L, int cap) { return L < 0 ? 0 : (L > cap ? cap : L); }

template <bool RELAXED>
__device__ __forceinline__ int load_len(const int *seqlens, int64_t sl_s, int i, int cap) {
  return clamp_len(load_len_raw<RELAXED>(seqlens, sl_s, i), cap);
}

// Sum over the batch of ceil(L_b / P), lengths clamped to [0, cap].
// RELAXED: loads that are well defined while another kernel may still write
// the lengths (the result then only steers prefetches).
template <bool RELAXED>
__device__ __noinline__ long long batch_pages(const int *seqlens, int64_t sl_s, int B, int cap, int log2_page,
                                                 int lane) {
  long long n = 0;
  for (int i = lane; i < B; i += 32) {
    const int L = load_len<RELAXED>(seqlens, sl_s, i, cap);
    n += (L + (1 << log2_page) - 1) >> log2_page;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  return n;
}

struct SplitUnit {
  int b;   // request (-1: the unit index is past the batch's last split)
  int s;   // split index within the request
  int sb;  // the request's split budget (the S of split_chunk / split_count)
  int L;   // the request's length as stored (not clamped)
};

// The u-th non-empty split of the batch, numbering the splits request by
// request (request 0's splits first).
template <bool RELAXED>
__device__ __noinline__ SplitUnit locate_unit(const int *seqlens, int64_t sl_s, int B, int cap, int log2_page,
                                                 int cp, int s_cap, int chunk_min, int u, int lane) {
  int base = 0;
  for (int i0 = 0; i0 < B; i0 += 32) {
    const int i = i0 + lane;
    const int raw = i < B ? load_len_raw<RELAXED>(seqlens, sl_s, i) : 0;
    const int L = clamp_len(raw, cap);
    const int sb = balanced_budget((L + (1 << log2_page) - 1) >> log2_page, cp, s_cap);
    const int nv = split_count(L, sb, log2_page, chunk_min);
    int incl = nv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += t;
    }
    const int tot = __shfl_sync(0xffffffffu, incl, 31);
    if (u < base + tot) {
      const unsigned m = __ballot_sync(0xffffffffu, base + incl > u);
      const int src = __ffs(m) - 1;
      SplitUnit r;
      r.b = i0 + src;
      r.s = u - base - __shfl_sync(0xffffffffu, incl - nv, src);
      r.sb = __shfl_sync(0xffffffffu, sb, src);
      r.L = __shfl_sync(0xffffffffu, raw, src);
      return r;
    }
    base += tot;
  }
  SplitUnit none;
  none.b = -1;
  none.s = 0;
  none.sb = 1;
  none.L = 0;
  return none;
}

// The u-th split of the balanced map (chunk of about cp pages; see
// balanced_chunk_pages) with its request's stored length. A batch of at most
// 32 requests is read once, one length per lane: the page total and the
// search share that load, one round trip instead of two.
template <bool RELAXED>
__device__ __forceinline__ SplitUnit locate_balanced(const int *seqlens, int64_t sl_s, int B, int cap, int log2_page,
                                                     int S, int s_cap, int chunk_min, int u, int lane) {
  if (B > 32) {
    const int cp = balanced_chunk_pages(batch_pages<RELAXED>(seqlens, sl_s, B, cap, log2_page, lane), B, S);
    return locate_unit<RELAXED>(seqlens, sl_s, B, cap, log2_page, cp, s_cap, chunk_min, u, lane);
  }
  const int raw = lane < B ? load_len_raw<RELAXED>(seqlens, sl_s, lane) : 0;
  const int L = clamp_len(raw, cap);
  long long n = (L + (1 << log2_page) - 1) >> log2_page;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  const int cp = balanced_chunk_pages(n, B, S);
  const int sb = balanced_budget((L + (1 << log2_page) - 1) >> log2_page, cp, s_cap);
  const int nv = lane < B ? split_count(L, sb, log2_page, chunk_min) : 0;
  int incl = nv;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  SplitUnit r;
  const unsigned m = __ballot_sync(0xffffffffu, incl > u);
  if (m == 0u) {
    r.b = -1;
    r.s = 0;
    r.sb = 1;
    r.L = 0;
    return r;
  }
  const int src = __ffs(m) - 1;
  r.b = src;
  r.s = u - __shfl_sync(0xffffffffu, incl - nv, src);
  r.sb = __shfl_sync(0xffffffffu, sb, src);
  r.L = __shfl_sync(0xffffffffu, raw, src);
  return r;
}

}  // namespace fd
