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
__device__ __forceinline__ int load_len(const int *seqlens, int64_t sl_s, int i, int cap) {
  int L = RELAXED ? ld_relaxed_gpu(seqlens + i * sl_s) : ld_cg(seqlens + i * sl_s);
  return L < 0 ? 0 : (L > cap ? cap : L);
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
};

// The u-th non-empty split of the batch, numbering the splits request by
// request (request 0's splits first).
template <bool RELAXED>
__device__ __noinline__ SplitUnit locate_unit(const int *seqlens, int64_t sl_s, int B, int cap, int log2_page,
                                                 int cp, int s_cap, int chunk_min, int u, int lane) {
  int base = 0;
  for (int i0 = 0; i0 < B; i0 += 32) {
    const int i = i0 + lane;
    const int L = i < B ? load_len<RELAXED>(seqlens, sl_s, i, cap) : 0;
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
      return r;
    }
    base += tot;
  }
  SplitUnit none;
  none.b = -1;
  none.s = 0;
  none.sb = 1;
  return none;
}

}  // namespace fd
