// stage1_tc.cuh - stage 1 of split-KV paged GQA flash decode for INT8 / INT4
// KV caches on the tcgen05 tensor cores (sm_103a, head_dim 128).
//
// Computes what fd_stage1_kernel computes for the quantised caches ("Triton
// GQA flash decode stage 1" with INT8 / INT4 KV in "feat(autotune): separate
// general and decode attention warmup", section "Covered decode kernels"):
// per (request, KV head, split, tile of 16 query rows) the partial output and
// log-sum-exp over the split's keys. The work is laid out for tcgen05:
//
//  * one CTA = 8 compute warps (two warpgroups), a TMA producer warp and an
//    MMA warp. Keys go in blocks of 128; thread t of a warpgroup owns key t of
//    the block, which is TMEM lane t of the score accumulator.
//  * the producer streams the raw code tiles (and fp32 scales) of each block
//    into a shared-memory ring with TMA, as fd_stage1_kernel does.
//  * the compute warps convert the codes once per block into fp16 operand
//    tiles (K-major, 128-byte swizzle): K as [key][dim] and V^T as
//    [dim][key]. Codes become exact fp16 biased integers (1024 + code + bias,
//    one LOP3 or PRMT per pair); int4 V takes its per-group scale in fp16 as
//    the register path does.
//  * the MMA warp issues S^T = K Q'^T (M = 128 keys, N = 16 query rows; int4:
//    one 32-channel group per accumulator, so each group's K scale can be
//    applied) and O^T += V^T P^T (M = 128 dims, N = 16 rows), accumulating in
//    TMEM.
//  * softmax runs per thread on its key's 8 rows (warpgroup 0: rows 0-7,
//    warpgroup 1: rows 8-15) with a lazily updated row max: only when a score
//    exceeds the running max by more than 2^8 does the warpgroup reduce the
//    block's row max and rescale its running sums and O columns. The common
//    block needs no cross-thread reduction at all; row sums stay per thread
//    and are reduced once at the end.
//
// Numerics match the register path: K codes are exact in fp16 and Q is scaled
// per row by a power of two into exact fp16 (odd int4 channels by 1/16 more);
// the code bias is taken out of the fp32 scores with per-(row, group)
// constants; V codes are debiased exactly in fp16; int8 folds its per-key V
// scale into P (fp16), int4 multiplies the V codes by the fp16 group scale. Keys at or past a row's limit are masked by
// selection, and V columns of keys past the split end are zero, so poisoned
// cache slots never reach a result.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitmap.cuh"
#include "tc.cuh"

namespace fd {

template <int KIND>
struct TcCfg {
  static constexpr int D = 128;
  static constexpr int BLOCK_N = 128;              // keys per block (M of the score MMA)
  static constexpr int NCW = 8;                    // compute warps: two warpgroups
  static constexpr int PRODUCER = NCW;             // warp index of the TMA producer
  static constexpr int MMA_WARP = NCW + 1;         // warp index of the MMA issuer (owns TMEM)
  static constexpr int THREADS = (NCW + 2) * 32;
  static constexpr int RB = KIND == KV_I8 ? D : D / 2;   // code bytes per cache row
  static constexpr int SW = RB;                    // TMA swizzle span of a code tile (box = whole rows)
  static constexpr int NG = KIND == KV_I4 ? D / 32 : 1;  // scale groups per row
  static constexpr int WPK = RB / 4;               // 32-bit code words per key
  static constexpr int CPW = KIND == KV_I8 ? 4 : 8;      // channels per code word
  static constexpr int SEG_MAX = 64;               // slots per TMA box at most
  static constexpr int STAGES = KIND == KV_I8 ? 3 : 4;
  static constexpr int TILE = BLOCK_N * RB;        // code bytes of K (or V) per stage
  static constexpr int SC = BLOCK_N * NG * 4;      // scale bytes of K (or V) per stage
  static constexpr int STAGE = (2 * TILE + 2 * SC + 1023) / 1024 * 1024;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int OFF_KH = RING;              // K  fp16 [128 keys][128 dims]
  static constexpr int OFF_VH = OFF_KH + 32768;    // 2 x V^T fp16 [128 rows][128 key slots]
  static constexpr int OFF_Q = OFF_VH + 2 * 32768; // Q' fp16 [16 rows][128 dims]
  static constexpr int OFF_P = OFF_Q + 4096;       // 2 x P fp16 [16 rows][128 key slots]
  static constexpr int OFF_QI = OFF_P + 2 * 4096;  // per row 2^e, then NG bias constants per row (fp32)
  static constexpr int QI = 16 * (1 + NG) * 4;
  static constexpr int OFF_RED = OFF_QI + QI;      // row reductions: [NCW][8] pairs of floats
  static constexpr int RED = NCW * 8 * 2 * 4;
  static constexpr int OFF_BAR = (OFF_RED + RED + 7) / 8 * 8;
  static constexpr int NBAR = 2 * STAGES + 6;      // full[], empty[], kfull, sfull, pfull[2], ofull[2]
  static constexpr int OFF_TSLOT = OFF_BAR + NBAR * 8;
  static constexpr int SMEM = OFF_TSLOT + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;   // slack to align the base to 1024
  static constexpr uint32_t TMEM_COLS = 256;
  static constexpr uint32_t TM_S = 0;              // 2 x score accumulators (NG x 16 columns) at 0 and 64
  static constexpr uint32_t TM_O = 128;            // O^T accumulator: 16 columns
  static constexpr uint32_t IDESC = umma_idesc_f16(128, 16);
  static_assert(SMEM_ALLOC <= 227 * 1024, "shared memory");
  static_assert(STAGE % 1024 == 0 && TILE % 1024 == 0, "swizzle atoms");
};

// V^T row of channel d = CPW * w + j (channel j of code word w): rows are
// ordered so that the lanes of a warp, which hold different words, store to
// rows of different swizzle phases. O^T lanes come out in this order.
template <int CPW>
__device__ __forceinline__ int tc_vrow(int d) {
  return (128 / CPW) * (d % CPW) + d / CPW;
}
template <int CPW>
__device__ __forceinline__ int tc_dim_of_vrow(int r) {
  return CPW * (r % (128 / CPW)) + r / (128 / CPW);
}

// Slot of key k of a block in the PV operands (columns of V^T and of P):
// 8-key chunks in order, the keys of odd chunks in reverse. (The V converters
// of odd chunks load their keys in reverse, which keeps their shared-memory
// loads free of bank conflicts.)
__device__ __forceinline__ int tc_key_slot(int k) {
  const int c = k >> 3, j = k & 7;
  return (c << 3) | ((c & 1) ? 7 - j : j);
}

// Byte offset of fp16 element (row, col) of a K-major, 128-byte-swizzled tile
// of `rows` rows: 64-column blocks of rows x 128 bytes, the 16-byte chunk
// index XORed with row % 8.
__device__ __forceinline__ uint32_t tc_sw128(int row, int col, int rows) {
  return (col >> 6) * rows * 128 + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + ((col & 7) << 1);
}

__device__ __forceinline__ uint32_t lop_or(uint32_t x, uint32_t mask, uint32_t ormask) {
  return (x & mask) | ormask;
}

// K tile: thread t of warpgroup h converts the codes of key t, channels
// [64h, 64h + 64), into row t of column block h (eight 16-byte chunks).
//  int8: code c -> fp16 1024 + (c + 128), channels in order.
//  int4: code c -> fp16 1024 + (c + 8) for the even channel of a byte and
//        1024 + 16 (c + 8) for the odd one (Q' divides those by 16); the 8
//        channels of a code word land in the order 0 4 1 5 2 6 3 7.
template <int KIND>
__device__ __forceinline__ void tc_convert_k(const uint8_t *kt, uint8_t *kh, int t, int h) {
  using C = TcCfg<KIND>;
  uint8_t *row = kh + h * (128 * 128) + t * 128;
#pragma unroll
  for (int q = 0; q < C::RB / 32; ++q) {  // 16-byte pieces of this half of the code row
    const uint4 v = *reinterpret_cast<const uint4 *>(kt + swz<C::SW>(t * C::RB + (C::RB / 2) * h + 16 * q));
    const uint32_t wd[4] = {v.x, v.y, v.z, v.w};
    if constexpr (KIND == KV_I4) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // one code word -> one 16-byte chunk
        const uint32_t x = wd[k] ^ 0x88888888u, y = x >> 8;
        uint4 o;
        o.x = lop_or(x, 0x000F000Fu, 0x64006400u);
        o.y = lop_or(x, 0x00F000F0u, 0x64006400u);
        o.z = lop_or(y, 0x000F000Fu, 0x64006400u);
        o.w = lop_or(y, 0x00F000F0u, 0x64006400u);
        const int chunk = 4 * q + k;
        *reinterpret_cast<uint4 *>(row + ((chunk ^ (t & 7)) << 4)) = o;
      }
    } else {
#pragma unroll
      for (int k = 0; k < 2; ++k) {  // two code words -> one 16-byte chunk
        const uint32_t x0 = wd[2 * k] ^ 0x80808080u, x1 = wd[2 * k + 1] ^ 0x80808080u;
        uint4 o;
        o.x = __byte_perm(x0, 0x64646464u, 0x5140);
        o.y = __byte_perm(x0, 0x64646464u, 0x7362);
        o.z = __byte_perm(x1, 0x64646464u, 0x5140);
        o.w = __byte_perm(x1, 0x64646464u, 0x7362);
        const int chunk = 2 * q + k;
        *reinterpret_cast<uint4 *>(row + ((chunk ^ (t & 7)) << 4)) = o;
      }
    }
  }
}

// V^T tile: converter thread (compute warp w, lane l) takes key chunk
// c = 2w + l / 16 of the block and code word wi of each of its 8 keys
// (int4: wi = l % 16; int8: also l % 16 + 16), and writes, for every channel
// of the word, the 16-byte chunk (8 key slots) of that channel's V^T row.
// Half-warps of odd chunks load their keys in reverse (their slots run
// backwards), so the two half-warps always read rows of opposite parity.
// Keys at or past nvalid (past the split end) read as code 0 with scale 0.
template <int KIND>
__device__ __forceinline__ void tc_convert_v(const uint8_t *vt, const float *vsc, uint8_t *vh, int w, int lane,
                                             int nvalid) {
  using C = TcCfg<KIND>;
  const int hh = lane >> 4, c = 2 * w + hh;
  int key[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) key[i] = 8 * c + (hh ? 7 - i : i);
#pragma unroll
  for (int u = 0; u < C::WPK / 16; ++u) {
    const int wi = (lane & 15) + 16 * u;
    uint32_t x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
      x[i] = key[i] < nvalid ? *reinterpret_cast<const uint32_t *>(vt + swz<C::SW>(key[i] * C::RB + 4 * wi)) : 0u;
    if constexpr (KIND == KV_I4) {
      const int grp = wi / 4;  // 32-channel scale group of this word
      uint32_t sp[4];
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const float s0 = key[2 * pp] < nvalid ? vsc[key[2 * pp] * C::NG + grp] : 0.f;
        const float s1 = key[2 * pp + 1] < nvalid ? vsc[key[2 * pp + 1] * C::NG + grp] : 0.f;
        sp[pp] = pack_f16x2(s0, s1);
      }
      uint32_t o[8][4];  // [channel of the word][key pair]
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const uint32_t a = x[2 * pp] ^ 0x88888888u, bb = x[2 * pp + 1] ^ 0x88888888u;
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {  // bytes 0-1, then 2-3, of both keys' words
          const uint32_t t0 = __byte_perm(a, bb, hb ? 0x7632u : 0x5410u);
          const uint32_t t8 = t0 >> 8;
          const uint32_t e0 = hsub2_u32(lop_or(t0, 0x000F000Fu, 0x64006400u), 1032.0f);
          const uint32_t e1 = hfma2_u32(lop_or(t0, 0x00F000F0u, 0x64006400u), 1.0f / 16.0f, -72.0f);
          const uint32_t e2 = hsub2_u32(lop_or(t8, 0x000F000Fu, 0x64006400u), 1032.0f);
          const uint32_t e3 = hfma2_u32(lop_or(t8, 0x00F000F0u, 0x64006400u), 1.0f / 16.0f, -72.0f);
          o[4 * hb + 0][pp] = hmul2_u32(e0, sp[pp]);
          o[4 * hb + 1][pp] = hmul2_u32(e1, sp[pp]);
          o[4 * hb + 2][pp] = hmul2_u32(e2, sp[pp]);
          o[4 * hb + 3][pp] = hmul2_u32(e3, sp[pp]);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        *reinterpret_cast<uint4 *>(vh + tc_sw128(tc_vrow<8>(8 * wi + j), 8 * c, 128)) =
            make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
    } else {
      uint32_t o[4][4];  // [byte (channel) of the word][key pair]
#pragma unroll
      for (int pp = 0; pp < 4; ++pp) {
        const uint32_t a = x[2 * pp] ^ 0x80808080u, bb = x[2 * pp + 1] ^ 0x80808080u;
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
          const uint32_t sel = bi | (bi << 4) | ((4u + bi) << 8) | ((4u + bi) << 12);
          o[bi][pp] = hsub2_u32(lop_or(__byte_perm(a, bb, sel), 0x00FF00FFu, 0x64006400u), 1152.0f);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j)
        *reinterpret_cast<uint4 *>(vh + tc_sw128(tc_vrow<4>(4 * wi + j), 8 * c, 128)) =
            make_uint4(o[j][0], o[j][1], o[j][2], o[j][3]);
    }
  }
}

// Q' tile (B operand of the score MMA) and the per-row constants, by the 256
// compute threads: thread i takes row i / 16, channels 8 (i % 16) .. +7.
// Each row is scaled by 2^(15 - e), e the exponent of its max |q|, so every
// bf16 value becomes an exact fp16 value; int4 channels are permuted like the
// K codes (0 4 1 5 2 6 3 7 within a word) and odd channels divided by 16.
// qinfo[r] = 2^(e - 15); qinfo[16 + r * NG + g] = the code bias of group g:
//   int8: 1152 * sum q',   int4: 1032 * sum_even q' + 72 * sum_odd q'.
template <int KIND>
__device__ __forceinline__ void tc_prepare_q(const Stage1Params &p, int b, int h, int rt, uint8_t *qtile,
                                             float *qinfo, int tid) {
  using C = TcCfg<KIND>;
  const int r = tid >> 4, cc = tid & 15;
  const int rg = rt * 16 + r;
  float v[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = 0.f;
  if (rg < p.R) {
    const int t = rg / p.G, gq = rg - t * p.G;
    const uint4 raw =
        *reinterpret_cast<const uint4 *>(p.q + b * p.q_sb + t * p.q_st + (h * p.G + gq) * p.q_sh + cc * 8);
    const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      v[2 * i] = __uint_as_float(rw[i] << 16);
      v[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
    }
  }
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  int E = 0;
  if (mx > 0.f && mx <= 3.0e38f) frexpf(mx, &E);
  E = max(E, -100);  // keep 2^(15 - E) finite for rows of tiny values
  const float down = ldexpf(1.0f, 15 - E);  // exact power of two
  float q[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) q[i] = v[i] * down;
  uint4 o;
  float c;
  if constexpr (KIND == KV_I4) {
    const float k16 = 1.0f / 16.0f;
    o.x = pack_f16x2(q[0], q[4]);
    o.y = pack_f16x2(q[1] * k16, q[5] * k16);
    o.z = pack_f16x2(q[2], q[6]);
    o.w = pack_f16x2(q[3] * k16, q[7] * k16);
    c = 1032.0f * (q[0] + q[2] + q[4] + q[6]) + 72.0f * (q[1] + q[3] + q[5] + q[7]);
    c += __shfl_xor_sync(0xffffffffu, c, 1);  // the 4 words of a 32-channel group
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    if ((cc & 3) == 0) qinfo[16 + r * C::NG + cc / 4] = c;
  } else {
    o.x = pack_f16x2(q[0], q[1]);
    o.y = pack_f16x2(q[2], q[3]);
    o.z = pack_f16x2(q[4], q[5]);
    o.w = pack_f16x2(q[6], q[7]);
    c = 1152.0f * (q[0] + q[1] + q[2] + q[3] + q[4] + q[5] + q[6] + q[7]);
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) c += __shfl_xor_sync(0xffffffffu, c, m);
    if (cc == 0) qinfo[16 + r] = c;
  }
  *reinterpret_cast<uint4 *>(qtile + tc_sw128(r, 8 * cc, 16)) = o;
  if (cc == 0) qinfo[r] = ldexpf(1.0f, E - 15);
}

// Bounded mbarrier wait that also gives up at once when another warp of the
// CTA has given up (the abort word in shared memory): after a timeout every
// warp runs to the end without waiting, so no named barrier is left waiting.
__device__ __forceinline__ bool tc_wait(uint64_t *bar, unsigned parity, unsigned *status, volatile int *abort) {
  if (mbar_try_wait(bar, parity)) return true;
  if (*abort) return false;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      atomicOr(status, FD_DEVSTAT_WAIT_TIMEOUT);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ bool tc_wait_warp(uint64_t *bar, unsigned parity, unsigned *status,
                                             volatile int *abort) {
  return __all_sync(0xffffffffu, tc_wait(bar, parity, status, abort)) != 0;
}

// One output element (row rg of the tile's request rows, channel d): the
// final output when the request has a single split, else the fp32 partial.
__device__ __forceinline__ void tc_write(const Stage1Params &p, bool direct, int b, int h, int s, int rg, int d,
                                         float val, float lse_nat) {
  const int t = rg / p.G, hq = h * p.G + (rg - t * p.G);
  if (direct) {
    const int64_t o = b * p.o_sb + t * p.o_st + hq * p.o_sh + d;
    if (p.out_f32) reinterpret_cast<float *>(p.out)[o] = val;
    else reinterpret_cast<__nv_bfloat16 *>(p.out)[o] = __float2bfloat16_rn(val);
    if (d == 0 && p.lse) p.lse[b * p.l_sb + t * p.l_st + hq * p.l_sh] = lse_nat;
  } else {
    const int64_t rowi = ((static_cast<int64_t>(b) * p.Tq + t) * p.Hq + hq) * p.s_cap + s;
    p.o_part[rowi * 128 + d] = val;
    if (d == 0) p.lse_part[rowi] = lse_nat;
  }
}

template <int KIND, bool FUSED>
__global__ void __launch_bounds__(TcCfg<KIND>::THREADS, 1)
    fd_stage1_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                        const __grid_constant__ Stage1Params p) {
  using C = TcCfg<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::STAGES;
  // Block j: K(j) converted -> kfull; score MMAs done -> sfull; V^T(j) and P(j)
  // written (buffer j % 2) and O rescaled -> pfull[j % 2]; PV MMAs done ->
  // ofull[j % 2]. Per-buffer barriers keep every waiter within one phase of
  // its barrier (a parity wait cannot tell phase j from phase j + 2).
  uint64_t *kfull = empty + C::STAGES;  // count: compute warps
  uint64_t *sfull = kfull + 1;          // tcgen05.commit
  uint64_t *pfull = kfull + 2;          // [2], count: compute warps
  uint64_t *ofull = kfull + 4;          // [2], tcgen05.commit
  uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_TSLOT + 8);
  float *qinfo = reinterpret_cast<float *>(smem + C::OFF_QI);
  float *red = reinterpret_cast<float *>(smem + C::OFF_RED);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int rt, h, u = 0, b, s;
  if (p.balanced) {
    rt = blockIdx.x % p.row_tiles;
    h = (blockIdx.x / p.row_tiles) % p.Hkv;
    u = blockIdx.x / (p.row_tiles * p.Hkv);
    b = -1;
    s = 0;
  } else {
    rt = blockIdx.x % p.row_tiles;
    s = blockIdx.x / p.row_tiles;
    h = blockIdx.y;
    b = blockIdx.z;
  }
  int S_req = p.num_splits;
  const int cap = p.max_pages * p.page_size;
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], 1 + 32);
      mbar_init(&empty[i], C::NCW);
    }
    mbar_init(kfull, C::NCW);
    mbar_init(sfull, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&pfull[i], C::NCW);
      mbar_init(&ofull[i], 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();  // inputs written by the previous kernel are visible from here on

  int L_bal = 0;
  if (p.balanced) {
    const SplitUnit su = locate_balanced<false>(p.seqlens, p.sl_s, p.batch, cap, p.log2_page, p.num_splits,
                                                p.s_cap, p.chunk_min, u, lane);
    if (su.b < 0) {
      griddep_launch_dependents();
      return;
    }
    b = su.b;
    s = su.s;
    S_req = su.sb;
    L_bal = su.L;
  }
  int L = p.balanced ? L_bal : p.seqlens[b * p.sl_s];
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0) atomicOr(p.status, FD_DEVSTAT_SEQLEN_OVERFLOW);
    L = L < 0 ? 0 : cap;
  }
  const int chunk = split_chunk(L, S_req, p.log2_page, p.chunk_min);
  const int c0 = s * chunk;
  const int c1 = min(L, c0 + chunk);
  const bool direct = FUSED || split_count(L, S_req, p.log2_page, p.chunk_min) == 1;
  if (c0 >= c1) {
    // Only an unsplit call reaches here with rows to write: a request with no
    // keys gets out = 0, lse = -inf. (A split call's empty splits write
    // nothing; the merge reads non-empty splits only.)
    if (FUSED) {
      const int ntile_rows = min(16, p.R - rt * 16);
      for (int i = threadIdx.x; i < ntile_rows * 128; i += C::THREADS)
        tc_write(p, true, b, h, s, rt * 16 + i / 128, i % 128, 0.f, -INFINITY);
    }
    griddep_launch_dependents();
    return;
  }
  const int n_iters = (c1 - c0 + C::BLOCK_N - 1) / C::BLOCK_N;

  // ---- set-up: TMEM, the Q' tile and its row constants, an all-zero P tile
  if (warp == C::MMA_WARP) tmem_alloc(tslot, C::TMEM_COLS);
  if (warp < C::NCW) {
    tc_prepare_q<KIND>(p, b, h, rt, smem + C::OFF_Q, qinfo, threadIdx.x);
    for (int i = threadIdx.x; i < 2 * 4096 / 16; i += C::NCW * 32)
      reinterpret_cast<uint4 *>(smem + C::OFF_P)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();  // Q' and P are read by the tensor cores
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;

  if (warp == C::PRODUCER) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    const uint64_t pol = l2_policy_evict_first();
    const int P = p.page_size;
    const int *pt = p.page_table + b * p.pt_sb;
    const int SEG = P < C::SEG_MAX ? P : C::SEG_MAX;  // slots per TMA box (within one page)
    const int log2_seg = P < C::SEG_MAX ? p.log2_page : 6;
    const unsigned seg_bytes = static_cast<unsigned>(SEG * C::RB);
    // Page ids of the split, relative to its first page fp0, in 32-page
    // windows held one per lane: wa = pages [32 win, 32 win + 32), wb = the
    // next 32, wc = the 32 after. A block reads only wa and wb (it spans at
    // most 17 pages); when it starts past wa the windows shift and the load of
    // a new wc is issued, two windows before any block reads it.
    const int fp0 = c0 >> p.log2_page;
    const int npg = ((c1 - 1) >> p.log2_page) - fp0 + 1;
    auto ld_pid = [&](int pi) { return pi < npg ? pt[fp0 + pi] : 0; };
    int win = 0;
    int wa = ld_pid(lane), wb = ld_pid(32 + lane), wc = ld_pid(64 + lane);
    auto pid_of = [&](int pi) {  // page id of relative page pi (pi in the two windows); all lanes call
      const int r = pi - 32 * win;
      const int a = __shfl_sync(0xffffffffu, wa, r & 31);
      const int bq = __shfl_sync(0xffffffffu, wb, r & 31);
      return r < 32 ? a : bq;
    };
    int issued = 0;
    for (int it = 0; it < n_iters; ++it) {
      const int tok0 = c0 + it * C::BLOCK_N;
      const int tend = min(tok0 + C::BLOCK_N, c1);
      const int first = (tok0 >> p.log2_page) - fp0;  // relative page of the block's first key
      if (first >= 32 * (win + 1)) {
        wa = wb;
        wb = wc;
        ++win;
        wc = ld_pid(32 * (win + 2) + lane);
      }
      const int stage = it % C::STAGES;
      const unsigned ph = (it / C::STAGES) & 1;
      if (!tc_wait_warp(&empty[stage], ph ^ 1, p.status, abort_flag)) break;
      uint8_t *kt = smem + stage * C::STAGE;
      uint8_t *vt = kt + C::TILE;
      const int nseg = (tend - tok0 + SEG - 1) >> log2_seg;
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<unsigned>(nseg) * seg_bytes * 2u);
      {  // lane i issues segment i (a block holds at most 128 / 8 = 16 segments)
        const int i = lane;
        const int ts = tok0 + (min(i, nseg - 1) << log2_seg);
        int pid = pid_of((ts >> p.log2_page) - fp0);
        const bool bad = i < nseg && (pid < 0 || pid >= p.num_pages);
        if (bad) pid = p.num_pages;  // outside the pool: record, and let TMA zero-fill
        if (__any_sync(0xffffffffu, bad) && lane == 0) atomicOr(p.status, FD_DEVSTAT_BAD_PAGE);
        if (i < nseg) {
          const int off = (i << log2_seg) * C::RB;
          tma_load_4d(kt + off, &tmk, 0, h, ts & (P - 1), pid, &full[stage], pol);
          tma_load_4d(vt + off, &tmv, 0, h, ts & (P - 1), pid, &full[stage], pol);
        }
      }
      float *ksc = reinterpret_cast<float *>(vt + C::TILE);
      float *vsc = ksc + C::BLOCK_N * C::NG;
#pragma unroll
      for (int i = lane; i < C::BLOCK_N; i += 32) {
        const int tok = tok0 + i;
        const int pid = pid_of((min(tok, tend - 1) >> p.log2_page) - fp0);
        if (tok < tend) {
          // a page id outside the pool takes page 0's scales (its codes read as 0)
          const int ps = (pid >= 0 && pid < p.num_pages) ? pid : 0;
          const float *src = p.kv_scales + static_cast<int64_t>(ps) * p.sc_sp +
                             static_cast<int64_t>(tok & (P - 1)) * p.sc_ss + static_cast<int64_t>(h) * p.sc_sh;
          cp_async_ca<C::NG * 4>(ksc + i * C::NG, src);
          cp_async_ca<C::NG * 4>(vsc + i * C::NG, src + p.sc_sk);
        }
      }
      cp_async_mbar_arrive_noinc(&full[stage]);
      issued = it + 1;
    }
    // drain: the most recent phase of every stage this warp filled has landed
    if (lane == 0) {
      for (int k = issued > C::STAGES ? issued - C::STAGES : 0; k < issued; ++k)
        mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1, p.status);
    }
  } else if (warp == C::MMA_WARP) {
    // ======================= MMA issuer =======================
    // Order: S(0); then per block j: S(j + 1) as soon as K(j + 1) is in, PV(j)
    // once P(j) is in. The scores of block j + 1 are computed while block j's
    // softmax runs.
    if (lane == 0) {
      const uint32_t kh = smem_u32(smem + C::OFF_KH), vh = smem_u32(smem + C::OFF_VH);
      const uint32_t qd = smem_u32(smem + C::OFF_Q), pd = smem_u32(smem + C::OFF_P);
      constexpr int KS_PER_G = 8 / C::NG;  // 16-channel K steps per scale group
      auto issue_s = [&](int j) {          // S^T(j) = K Q'^T into accumulator j % 2
        const uint32_t dst = tmem + C::TM_S + 64 * (j & 1);
#pragma unroll
        for (int g = 0; g < C::NG; ++g)
#pragma unroll
          for (int kk = 0; kk < KS_PER_G; ++kk) {
            const int ks = g * KS_PER_G + kk;
            const uint32_t oa = (ks >> 2) * (128 * 128) + (ks & 3) * 32;  // K tile, 128 rows
            const uint32_t ob = (ks >> 2) * (16 * 128) + (ks & 3) * 32;   // Q' tile, 16 rows
            umma_f16_ss(dst + 16 * g, umma_desc_sw128(kh + oa), umma_desc_sw128(qd + ob), C::IDESC,
                        kk > 0 ? 1u : 0u);
          }
        umma_commit(sfull);
      };
      auto issue_pv = [&](int j) {  // O^T += V^T(j) P(j)^T
        const uint32_t vb = vh + (j & 1) * 32768, pb = pd + (j & 1) * 4096;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t oa = (kk >> 2) * (128 * 128) + (kk & 3) * 32;  // V^T tile, 128 rows
          const uint32_t ob = (kk >> 2) * (16 * 128) + (kk & 3) * 32;   // P tile, 16 rows
          umma_f16_ss(tmem + C::TM_O, umma_desc_sw128(vb + oa), umma_desc_sw128(pb + ob), C::IDESC,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&ofull[j & 1]);
      };
      uint64_t *last_bar = nullptr;  // the barrier and phase of the last commit
      unsigned last_par = 0;
      if (tc_wait(kfull, 0, p.status, abort_flag)) {
        tc_fence_after();
        issue_s(0);
        last_bar = sfull;
        last_par = 0;
        for (int j = 0; j < n_iters; ++j) {
          if (j + 1 < n_iters) {
            if (!tc_wait(kfull, (j + 1) & 1, p.status, abort_flag)) break;
            tc_fence_after();
            issue_s(j + 1);
            last_bar = sfull;
            last_par = (j + 1) & 1;
          }
          if (!tc_wait(&pfull[j & 1], (j >> 1) & 1, p.status, abort_flag)) break;
          tc_fence_after();
          issue_pv(j);
          last_bar = &ofull[j & 1];
          last_par = (j >> 1) & 1;
        }
      }
      // every MMA issued has completed before TMEM is released (a commit
      // tracks all earlier MMAs of this thread)
      if (last_bar) mbar_wait(last_bar, last_par, p.status);
    }
    __syncwarp();
  } else {
    // ======================= compute warpgroups =======================
    const int wg = warp >> 2;           // rows 8 wg .. 8 wg + 7 of the tile
    const int t = threadIdx.x & 127;    // this thread's key of a block = its TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    float rs[8], qc[C::NG][8], m[8], l[8];
    int lim[8];
    int limmin = 0x7fffffff;
    bool any_row = false;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int r = 8 * wg + i, rg = rt * 16 + r;
      rs[i] = qinfo[r] * p.scale_log2;
#pragma unroll
      for (int g = 0; g < C::NG; ++g) qc[g][i] = qinfo[16 + r * C::NG + g];
      m[i] = -INFINITY;
      l[i] = 0.f;
      if (rg < p.R) {
        lim[i] = min(c1, L - (p.Tq - 1) + rg / p.G);
        limmin = min(limmin, lim[i]);
        any_row = true;
      } else {
        lim[i] = c0;  // padding row: no key is visible
      }
    }
    const int bar_id = 2 + wg;
    // Block j: V(j) -> V^T buffer j % 2 (after PV(j - 2)); release the stage;
    // wait S(j); K(j + 1) -> K tile (S(j) has read it); softmax(j) -> P buffer
    // j % 2. K(0) goes first.
    tc_wait_warp(&full[0], 0, p.status, abort_flag);
    tc_convert_k<KIND>(smem, smem + C::OFF_KH, t, wg);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(kfull);
    for (int it = 0; it < n_iters; ++it) {
      const int stage = it % C::STAGES;
      const int tok0 = c0 + it * C::BLOCK_N;
      const uint8_t *kt = smem + stage * C::STAGE;
      const uint8_t *vt = kt + C::TILE;
      const float *ksc = reinterpret_cast<const float *>(vt + C::TILE);
      const float *vsc = ksc + C::BLOCK_N * C::NG;
      const int nvalid = c1 - tok0;  // keys of this block inside the split
      float ks[C::NG];
      if constexpr (C::NG == 4) {
        const float4 k4 = *reinterpret_cast<const float4 *>(ksc + t * 4);
        ks[0] = k4.x;
        ks[1] = k4.y;
        ks[2] = k4.z;
        ks[3] = k4.w;
      } else {
        ks[0] = ksc[t];
      }
      float vs_key = 0.f;  // int8: this key's V scale, folded into P
      if constexpr (KIND == KV_I8) vs_key = t < nvalid ? vsc[t] : 0.f;

      // V codes -> V^T buffer it % 2, once PV(it - 2) has released it
      if (it >= 2) tc_wait_warp(&ofull[it & 1], ((it - 2) >> 1) & 1, p.status, abort_flag);
      tc_convert_v<KIND>(vt, vsc, smem + C::OFF_VH + (it & 1) * 32768, warp, lane, nvalid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);  // the stage's codes and scales are consumed

      tc_wait_warp(sfull, it & 1, p.status, abort_flag);
      tc_fence_after();
      // K codes of the next block -> K tile (S(it) has read it)
      if (it + 1 < n_iters) {
        const int st1 = (it + 1) % C::STAGES;
        tc_wait_warp(&full[st1], ((it + 1) / C::STAGES) & 1, p.status, abort_flag);
        tc_convert_k<KIND>(smem + st1 * C::STAGE, smem + C::OFF_KH, t, wg);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(kfull);
      }
      if (any_row) {
        float a[C::NG][8];
#pragma unroll
        for (int g = 0; g < C::NG; ++g) tmem_ld8(tl + C::TM_S + 64 * (it & 1) + 16 * g + 8 * wg, a[g]);
        tmem_wait_ld();
        float sv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          float acc = 0.f;
#pragma unroll
          for (int g = 0; g < C::NG; ++g) acc = fmaf(ks[g], a[g][i] - qc[g][i], acc);
          sv[i] = acc * rs[i];
        }
        const int kidx = tok0 + t;
        if (tok0 + C::BLOCK_N > limmin) {  // some key of the block is past some row's limit
#pragma unroll
          for (int i = 0; i < 8; ++i) sv[i] = kidx < lim[i] ? sv[i] : -INFINITY;
        }
        bool need = false;
#pragma unroll
        for (int i = 0; i < 8; ++i) need |= sv[i] > m[i] + 8.0f;
        if (bar_red_or(bar_id, 128, need)) {
          // a score exceeds its row's running max by more than 2^8: reduce the
          // block's row maxima over the warpgroup and rescale
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float x = sv[i];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
            if (lane == 0) red[(warp * 8 + i) * 2] = x;
          }
          named_barrier(bar_id, 128);
          float alpha[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            float bm = red[((4 * wg) * 8 + i) * 2];
#pragma unroll
            for (int ww = 1; ww < 4; ++ww) bm = fmaxf(bm, red[((4 * wg + ww) * 8 + i) * 2]);
            const float mn = fmaxf(m[i], bm);
            alpha[i] = mn == -INFINITY ? 1.f : fast_exp2(m[i] - mn);  // m = -inf: nothing to keep
            m[i] = mn;
            l[i] *= alpha[i];
          }
          if (it > 0) {  // the O^T columns of these rows, once PV(it - 1) has completed
            tc_wait_warp(&ofull[(it - 1) & 1], ((it - 1) >> 1) & 1, p.status, abort_flag);
            tc_fence_after();
            float o8[8];
            tmem_ld8(tl + C::TM_O + 8 * wg, o8);
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) o8[i] *= alpha[i];
            tmem_st8(tl + C::TM_O + 8 * wg, o8);
            tmem_wait_st();
          }
        }
        float pv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float e = fast_exp2(sv[i] - (m[i] == -INFINITY ? 0.f : m[i]));
          l[i] += e;
          if constexpr (KIND == KV_I8) pv[i] = e == 0.f ? 0.f : e * vs_key;
          else pv[i] = e;
        }
        // P[row][slot]: lanes 2q, 2q+1 hold neighbouring slots; the even lane
        // stores rows 0-3 of this warpgroup's 8, the odd lane rows 4-7
        const bool odd = (lane & 1) != 0;
        const bool self_lo = (((t >> 3) & 1) == 0) == !odd;
        const int pslot = tc_key_slot(t) & ~1;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float mine = odd ? pv[4 + k] : pv[k];
          const float theirs = __shfl_xor_sync(0xffffffffu, odd ? pv[k] : pv[4 + k], 1);
          const uint32_t v = self_lo ? pack_f16x2(mine, theirs) : pack_f16x2(theirs, mine);
          const int row = 8 * wg + (odd ? 4 : 0) + k;
          *reinterpret_cast<uint32_t *>(smem + C::OFF_P + (it & 1) * 4096 + tc_sw128(row, pslot, 16)) = v;
        }
      }
      fence_proxy_async_smem();  // P and V^T are read by the tensor cores
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&pfull[it & 1]);
    }

    // ---- epilogue: normalise the O^T columns of this warpgroup's rows
    tc_wait_warp(&ofull[(n_iters - 1) & 1], ((n_iters - 1) >> 1) & 1, p.status, abort_flag);
    tc_fence_after();
    named_barrier(bar_id, 128);  // red[] is free: every slow path of the loop has read it
    if (any_row) {
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        float x = l[i];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
        if (lane == 0) red[(warp * 8 + i) * 2 + 1] = x;
      }
      named_barrier(bar_id, 128);
      float o8[8];
      tmem_ld8(tl + C::TM_O + 8 * wg, o8);
      tmem_wait_ld();
      const int d = tc_dim_of_vrow<C::CPW>((warp & 3) * 32 + lane);
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        const int rg = rt * 16 + 8 * wg + i;
        if (rg >= p.R) continue;
        float Ls = 0.f;
#pragma unroll
        for (int ww = 0; ww < 4; ++ww) Ls += red[((4 * wg + ww) * 8 + i) * 2 + 1];
        const float val = Ls > 0.f ? o8[i] / Ls : 0.f;
        const float lse_nat = Ls > 0.f ? (m[i] + log2f(Ls)) * 0.69314718055994531f : -INFINITY;
        tc_write(p, direct, b, h, s, rg, d, val, lse_nat);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == C::MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
  griddep_launch_dependents();
}

template <int KIND>
cudaError_t stage1_tc_prepare_t() {
  cudaError_t e = cudaFuncSetAttribute(fd_stage1_tc_kernel<KIND, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, TcCfg<KIND>::SMEM_ALLOC);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fd_stage1_tc_kernel<KIND, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<KIND>::SMEM_ALLOC);
  return e;
}

template <int KIND>
cudaError_t launch_stage1_tc_t(bool fused, const CUtensorMap &tmk, const CUtensorMap &tmv, const Stage1Params &p,
                               dim3 grid, cudaStream_t stream) {
  using C = TcCfg<KIND>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = C::SMEM_ALLOC;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (fused) return cudaLaunchKernelEx(&cfg, fd_stage1_tc_kernel<KIND, true>, tmk, tmv, p);
  return cudaLaunchKernelEx(&cfg, fd_stage1_tc_kernel<KIND, false>, tmk, tmv, p);
}

}  // namespace fd
