// stage1.cuh - split-KV paged GQA flash decode, stage 1 (sm_103a).
//
// Computes, for one (request b, KV head h, KV split s, tile of 16 query rows),
// the softmax-normalised partial output and log-sum-exp of the tile's rows
// over the split's keys: "Triton GQA flash decode stage 1" and its INT8 /
// INT4 KV variants in "feat(autotune): separate general and decode attention
// warmup" (LightLLM PR 1549), section "Covered decode kernels". The query rows
// of a tile are the G query heads of KV head h times the Tq query tokens
// (row r = t * G + g), so K and V are read once per group ("GQA").
//
// Structure of one CTA (NUM_CW consumer warps + 1 producer warp):
//  * split range: chunk = split_chunk(L_b, S, ...) (equal page-aligned chunks,
//    at least chunk_min keys); split s owns keys [s * chunk, min(L_b, (s + 1) *
//    chunk)), derived here from cache_seqlens.
//  * producer warp: reads page ids from the page table one stage ahead, and
//    lane i issues the 4-D TMA loads (d, head, slot, page) of page segment i
//    of K and V into a STAGES-deep shared-memory ring, 128-byte swizzled,
//    completing on a per-stage mbarrier. Quantised caches also copy their
//    per-row fp32 scales with cp.async (one arrival per lane on the barrier).
//  * consumer warps: warp w takes keys [KPW w, KPW w + KPW) of each stage of
//    4 KPW keys (KPW = 16; 32 for the 16-row int4 and the narrow int8
//    variants, as two 16-key sub-blocks that share one softmax step).
//    QK^T and PV run on mma.sync m16n8k16 (fp32 accumulate) with the 16 query
//    rows as M; the online softmax keeps a running max / sum per row in the
//    log2 domain with quad shuffles. bf16 caches feed ldmatrix fragments
//    straight from the TMA tile. Quantised caches are converted in registers
//    from the raw tile, no staging copy:
//      - K: ldmatrix of the raw rows as 16-bit elements hands each thread 4
//        (int8) or 8 (int4) consecutive codes of one key; they become exact
//        (biased) fp16 B fragments, and the Q A fragments are built once per CTA with
//        the matching channel order (a dot product does not care about the
//        order of its terms). K scales multiply the fp32 scores (per
//        32-channel group for int4, from one accumulator per group).
//      - V, int8: ldmatrix.trans of 8 keys x 16 channels pairs two keys'
//        codes at a channel in one register (bytes 0, 2 and 1, 3), so each
//        fp16 fragment takes one LOP3 and one subtract; the per-key V scale
//        is folded into the probabilities (fp16).
//      - V, int4: ldmatrix.trans of 8 keys x one scale group's 16 bytes hands
//        each thread the 4 nibbles of two keys at 4 channels of the group, so
//        every PV n-tile lies inside one 32-channel group; the group's V
//        scale multiplies the probabilities (one P operand per group) and the
//        codes need only their bias removed. O stays in tensor memory between
//        blocks.
//        PV output columns come out permuted and are put back in order by the
//        epilogue.
//    Quantised tiles of at most 8 rows ("narrow", warp_block_km) swap the
//    roles: keys and channels are the M dimension, the rows the 8-wide N
//    dimension, so the MMAs and the softmax carry no empty rows.
//  * epilogue: the consumer warps merge their (max, sum, O) through shared
//    memory and write either fp32 partial O + LSE to the split workspace, or
//    (num_splits == 1) the final bf16/fp32 output and LSE.
//
// Keys at or past a row's limit are masked by selection (-inf score, zero
// probability), and V rows past the split end are zeroed in shared memory
// before PV, so stale or poisoned cache slots (NaN, huge values) never reach
// a result.
#pragma once

#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "splitmap.cuh"
#include "tc.cuh"

namespace fd {

template <int KIND, int D_, bool DEEP = false, bool NARROW = false>
struct S1Cfg {
  static constexpr int D = D_;
  static constexpr bool QUANT = KIND != KV_BF16;
  // NARROW (quantised caches, tiles of at most 8 query rows): the keys are the
  // M dimension of the MMAs and the rows the 8-wide N dimension (warp_block_km)
  static_assert(!NARROW || QUANT, "the narrow variant serves quantised caches");
  static_assert(!(NARROW && DEEP), "one variant at a time");
  static constexpr int OT = NARROW ? D / 16 : D / 8;     // O fragments (4 fp32 each) per thread
  static constexpr int ROW_BYTES = KIND == KV_BF16 ? 2 * D : (KIND == KV_I8 ? D : D / 2);
  static constexpr int BOX_BYTES = ROW_BYTES < 128 ? ROW_BYTES : 128;  // TMA box inner extent
  static constexpr int N_BOX = ROW_BYTES / BOX_BYTES;
  static constexpr int BOX_ELEMS = KIND == KV_BF16 ? BOX_BYTES / 2 : BOX_BYTES;
  static constexpr int NG = KIND == KV_I4 ? D / 32 : 1;  // fp32 scales per cache row
  static constexpr int NT = D / 8;                       // PV n-tiles (channels per thread, quantised V)
  // consumer warps; the deep (one CTA per SM) variant doubles them so a lone
  // CTA has more blocks in flight
  static constexpr int NUM_CW = DEEP ? 8 : 4;
  // keys per consumer warp and stage: 16, or 32 for the 16-row int4 and the
  // narrow int8 variants (two 16-key sub-blocks share one softmax step, one
  // reload of the Q fragments and, int4, one round trip of O through tensor
  // memory, and their MMA chains interleave)
  static constexpr int KPW = (KIND == KV_I4 && !NARROW && !DEEP) || (KIND == KV_I8 && NARROW) ? 32 : 16;
  static constexpr int BLOCK_N = NUM_CW * KPW;           // keys per pipeline stage
  static constexpr int SEG_MAX = 64;                     // slots per TMA box at most
  static constexpr int THREADS = (NUM_CW + 1) * 32;
  // DEEP: one CTA per SM with 8 consumer warps and 64 KB stages, for grids
  // that fit in one wave (small batches), where a single CTA must keep enough
  // bytes and blocks in flight.
  // Quantised kinds are bound by the consumer warps' latency, not by bytes in
  // flight: the 16-row variants and the narrow int8 one (its 128-key stages)
  // run three CTAs per SM (128 registers), the narrow int4 one four (96
  // registers), on rings that fit (FOUR asks for four where they fit).
  static constexpr bool FOUR = NARROW;
  static constexpr int STAGES = KIND == KV_BF16 ? 3 : (KIND == KV_I8 ? (FOUR ? 2 : 3) : (FOUR ? 4 : 6) * 16 / KPW);
  // Quantised kinds park the (identical) Q fragments of the consumer warps in
  // shared memory and reload them per block, so they do not hold 32 (narrow:
  // 16) registers through the PV half of the loop.
  static constexpr bool QA_SMEM = QUANT && !NARROW;
  static constexpr bool QB_SMEM = NARROW;
  static constexpr int TILE = BLOCK_N * ROW_BYTES;       // K (or V) bytes of one stage
  static constexpr int SC = QUANT ? BLOCK_N * NG * 4 : 0;
  static constexpr int STAGE = ((2 * TILE + 2 * SC) + 1023) / 1024 * 1024;
  static constexpr int RING = STAGES * STAGE;
  static constexpr int QROW = D * 2 + 16;                // padded bf16 row of the Q tile
  static constexpr int QB = 16 * QROW;
  static constexpr int CROW = D + 8;                     // padded fp32 row of the combine tile
  static constexpr int TR = NARROW ? 8 : 16;              // combine-tile rows per warp
  static constexpr int CMB_O = NUM_CW * TR * CROW * 4;
  static constexpr int CMB = CMB_O + NUM_CW * TR * 2 * 4;
  static constexpr int OFF_Q = RING;
  static constexpr int OFF_QI = OFF_Q + QB;              // per row: 2^e, then NG bias constants
  static constexpr int QI = QUANT ? 16 * (1 + NG) * 4 : 0;
  static constexpr int OFF_QA = (OFF_QI + QI + 15) / 16 * 16;  // [D/16][32 lanes] uint4
  static constexpr int QAB = QA_SMEM ? (D / 16) * 32 * 16 : (QB_SMEM ? (D / 16) * 32 * 8 : 0);
  static constexpr int OFF_BAR = (OFF_QA + QAB + 7) / 8 * 8;
  static constexpr int OFF_FLAG = OFF_BAR + 2 * STAGES * 8;  // "this CTA merges" flag
  // the epilogue's (request, split, length, budget | direct << 16), parked
  // here through the main loop so they hold no registers there
  static constexpr int OFF_META = OFF_FLAG + 16;
  // int4 keeps O in tensor memory between blocks: D/2 fp32 columns
  // per thread (its lane), allocated by consumer warp 0; the address lands here
  // (int8 measured faster with O in registers; narrow O is half the size)
  static constexpr bool O_TMEM = KIND == KV_I4 && !NARROW;
  static constexpr int TMEM_COLS = D / 2;
  // int8 V codes enter PV as subnormals (kU8Sub): one fragment of bias row sums
  static constexpr bool V_SUB = KIND == KV_I8;
  static constexpr int NR = 1;
  static constexpr int OFF_TMEM = OFF_META + 16;
  static constexpr int SMEM = OFF_TMEM + 16;
  static constexpr int SMEM_ALLOC = SMEM + 1024;         // slack to align the base to 1024
  // CTAs per SM the shared memory allows (228 KB per SM, 1 KB reserved per CTA)
  static constexpr int MIN_BLOCKS = FOUR && 4 * (SMEM_ALLOC + 1024) <= 228 * 1024 ? 4
                                    : 3 * (SMEM_ALLOC + 1024) <= 228 * 1024   ? 3
                                    : 2 * (SMEM_ALLOC + 1024) <= 228 * 1024 ? 2
                                                                             : 1;
  static_assert(CMB <= RING, "combine tile must fit in the ring");
  static_assert(TILE % 1024 == 0, "tiles must keep the 1024-byte swizzle alignment");
  static_assert(D == 64 || D == 128, "head_dim");
};

// ----------------------------------------------------------------------------
// In-register conversions of cache codes to fp16 (exact: |code| <= 128).

// int4 codes are stored as two's-complement nibbles n = code & 15, and
// n ^ 8 = code + 8 = u in [0, 15]. From the nibbles at bits 0-3 and 16-19:
// f16x2 (1024 + u, 1024 + u'); from those at bits 4-7 and 20-23:
// f16x2 (1024 + 16u, 1024 + 16u'). Mask, bias and exponent in one LOP3 each
// (the XOR constant is a register: kNibLo / kNibHi).
constexpr uint32_t kNibLo = 0x64086408u, kNibHi = 0x64806480u;
__device__ __forceinline__ uint32_t nib_lo_f16_biased(uint32_t t, uint32_t c) {
  return and_xor<0x000F000Fu>(t, c);
}
__device__ __forceinline__ uint32_t nib_hi_f16_biased(uint32_t t, uint32_t c) {
  return and_xor<0x00F000F0u>(t, c);
}

// int8 V codes enter PV as fp16 subnormals: a half whose bits are u < 1024
// has the value u * 2^-24 exactly, so one LOP3 (mask, and flip the code's
// sign bit: u = code + 128) gives the operand pair, with no fp16
// subtraction. The bias left in the products is 128 times the row sum R of
// the probability operand over the keys; one more MMA against ones per
// 16-key sub-block accumulates R beside O, and the epilogue takes
// O = 2^24 O_raw - 128 R (remove_v_bias). Products and R are exact in fp32
// before accumulation, and for codes of either sign the bias term is of the
// order of the result, so the cancellation costs a bit or two of the sum.
// (int4 keeps exact biased fp16 codes: with its per-group V scales the bias
// sums it would need measured no faster.)
constexpr uint32_t kU8Sub = 0x00800080u;     // bytes 0 and 2: u = code ^ 0x80
constexpr uint32_t kOnesF16 = 0x3C003C00u;   // f16x2 (1, 1)
__device__ __forceinline__ uint32_t i8pair_to_f16_sub(uint32_t t, uint32_t c) { return and_xor<0x00FF00FFu>(t, c); }

// ----------------------------------------------------------------------------
// One 16-key block of one warp, bf16 cache: scores, online softmax, PV.
//
// kbase / vbase: shared addresses of the stage's K / V tiles, laid out as
// 64-element halves (half stride `half`) of 128-byte swizzled rows; the
// warp's keys are rows row0..row0+15.
template <class C>
__device__ __forceinline__ void warp_block(uint32_t kbase, uint32_t vbase, uint32_t half, int row0,
                                           const uint32_t (&qa)[C::D / 16][4],
                                           float (&o)[C::D / 8][4], float (&m)[2], float (&l)[2],
                                           int tok_row0, int lim0, int lim1, float scale_log2,
                                           int lane) {
  constexpr int D = C::D;
  constexpr int NG = 1;
  const int c = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;

  // ---- S = Q K^T (16 rows x 16 keys), one accumulator per scale group
  float acc[NG][2][4];
#pragma unroll
  for (int gi = 0; gi < NG; ++gi)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[gi][nt][e] = 0.f;

  const int krow = row0 + ((mi >> 1) << 3) + ri;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks) {
    const int d = ks * 16 + ((mi & 1) << 3);
    uint32_t bk[4];
    ldsm_x4(bk, kbase + (d >> 6) * half + swz<128>(krow * 128 + (d & 63) * 2));
    const int gi = NG == 1 ? 0 : ks / 2;
    mma_bf16_16816(acc[gi][0], qa[ks], bk[0], bk[1]);
    mma_bf16_16816(acc[gi][1], qa[ks], bk[2], bk[3]);
  }

  // ---- scale, mask (by selection), running max
  float s[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int key = nt * 8 + 2 * c + (e & 1);
      const float v = acc[0][nt][e];
      const int lim = (e < 2) ? lim0 : lim1;
      s[nt][e] = (tok_row0 + key < lim) ? v * scale_log2 : -INFINITY;
    }
  }
  float mx0 = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
  float mx1 = fmaxf(fmaxf(s[0][2], s[0][3]), fmaxf(s[1][2], s[1][3]));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const float b0 = mn0 == -INFINITY ? 0.f : mn0;
  const float b1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = fast_exp2(m[0] - b0), al1 = fast_exp2(m[1] - b1);
  m[0] = mn0;
  m[1] = mn1;

  float p[2][4];
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    p[nt][0] = fast_exp2(s[nt][0] - b0);
    p[nt][1] = fast_exp2(s[nt][1] - b0);
    p[nt][2] = fast_exp2(s[nt][2] - b1);
    p[nt][3] = fast_exp2(s[nt][3] - b1);
  }
  l[0] = l[0] * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
  l[1] = l[1] * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);

  if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int j = 0; j < D / 8; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al0;
      o[j][2] *= al1;
      o[j][3] *= al1;
    }
  }

  // ---- P (bf16) as the A operand of PV
  uint32_t pa[4];
  pa[0] = pack_bf16x2(p[0][0], p[0][1]);
  pa[1] = pack_bf16x2(p[0][2], p[0][3]);
  pa[2] = pack_bf16x2(p[1][0], p[1][1]);
  pa[3] = pack_bf16x2(p[1][2], p[1][3]);

  // ---- O += P V
  const int vrow = row0 + ((mi & 1) << 3) + ri;
#pragma unroll
  for (int dp = 0; dp < D / 16; ++dp) {
    const int d = dp * 16 + ((mi >> 1) << 3);
    uint32_t bv[4];
    ldsm_x4_t(bv, vbase + (d >> 6) * half + swz<128>(vrow * 128 + (d & 63) * 2));
    mma_bf16_16816(o[2 * dp], pa, bv[0], bv[1]);
    mma_bf16_16816(o[2 * dp + 1], pa, bv[2], bv[3]);
  }
}

// ----------------------------------------------------------------------------
// Online-softmax update in the log2 domain for a thread's two rows (g, g+8)
// over KB 16-key sub-blocks that share one row max (scores s[kb][nt][e], row
// g for e < 2, g + 8 for e >= 2): row max over the quad, alpha = 2^(m_old -
// m_new), p = 2^(s - m_new), running sum rescaled by alpha. Rows that have
// seen no key keep m = -inf and p = 0. Returns whether O must be rescaled by
// al (warp-uniform).
// LAZY: the rows keep their running max m until some row of the warp sees a
// score above its m + kLazyMax (log2 units); until then p = 2^(s - m) may
// reach 2^kLazyMax, and al = 1. The result is the same up to rounding (l, O
// and the LSE all use the same m), and the 64-multiply rescale of O runs
// about once per split instead of on a third of its blocks.
constexpr float kLazyMax = 8.f;
template <int KB, bool LAZY>
__device__ __forceinline__ bool softmax_update_kb(const float (&s)[KB][2][4], float (&p)[KB][2][4],
                                                  float (&m)[2], float (&l)[2], float (&al)[2]) {
  float mx0 = fmaxf(fmaxf(s[0][0][0], s[0][0][1]), fmaxf(s[0][1][0], s[0][1][1]));
  float mx1 = fmaxf(fmaxf(s[0][0][2], s[0][0][3]), fmaxf(s[0][1][2], s[0][1][3]));
#pragma unroll
  for (int kb = 1; kb < KB; ++kb) {
    mx0 = fmaxf(mx0, fmaxf(fmaxf(s[kb][0][0], s[kb][0][1]), fmaxf(s[kb][1][0], s[kb][1][1])));
    mx1 = fmaxf(mx1, fmaxf(fmaxf(s[kb][0][2], s[kb][0][3]), fmaxf(s[kb][1][2], s[kb][1][3])));
  }
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
  mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
  mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
  float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  bool rescale;
  if constexpr (LAZY) {
    // (a row's first finite score always moves it: -inf + kLazyMax = -inf)
    rescale = __any_sync(0xffffffffu, mn0 > m[0] + kLazyMax || mn1 > m[1] + kLazyMax);
    if (!rescale) {
      mn0 = m[0];
      mn1 = m[1];
    }
  }
  const float b0 = mn0 == -INFINITY ? 0.f : mn0;
  const float b1 = mn1 == -INFINITY ? 0.f : mn1;
  al[0] = fast_exp2(m[0] - b0);
  al[1] = fast_exp2(m[1] - b1);
  m[0] = mn0;
  m[1] = mn1;
  if constexpr (!LAZY) rescale = __any_sync(0xffffffffu, al[0] != 1.f || al[1] != 1.f);
  float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      p[kb][nt][0] = fast_exp2(s[kb][nt][0] - b0);
      p[kb][nt][1] = fast_exp2(s[kb][nt][1] - b0);
      p[kb][nt][2] = fast_exp2(s[kb][nt][2] - b1);
      p[kb][nt][3] = fast_exp2(s[kb][nt][3] - b1);
    }
    sum0 += p[kb][0][0] + p[kb][0][1] + p[kb][1][0] + p[kb][1][1];
    sum1 += p[kb][0][2] + p[kb][0][3] + p[kb][1][2] + p[kb][1][3];
  }
  l[0] = l[0] * al[0] + sum0;
  l[1] = l[1] * al[1] + sum1;
  return rescale;
}

// ----------------------------------------------------------------------------
// One block of C::KPW keys (KB = KPW / 16 sub-blocks of 16 sharing one
// softmax step) of one warp, quantised cache, straight from the raw tile.
//
// kt / vt: the stage's raw K / V tiles (rows of ROW_BYTES, TMA-swizzled with
// span BOX_BYTES); ksc / vsc: the stage's per-row fp32 scales (NG per row).
// qa: Q fragments in the channel order the K codes arrive in (see
// build_q_fragments). O columns come out permuted: n-tile j, d-slot n holds
// channel n * NT + j.
template <class C, int KIND>
__device__ __forceinline__ void warp_block_q(const uint8_t *kt, const uint8_t *vt, const float *ksc,
                                             const float *vsc, int row0,
                                             const uint32_t (&qa)[C::D / 16][4],
                                             const uint4 *qa_s, const float (&qc)[2][C::NG], const float *qcs,
                                             const float (&rs)[2],
                                             float (&o)[C::NT][4], float (&ra)[C::NR][4], uint32_t tm_o,
                                             float (&m)[2], float (&l)[2], int tok_row0, int c1, int lim0,
                                             int lim1, int lane) {
  constexpr int NG = C::NG, RB = C::ROW_BYTES, SW = C::BOX_BYTES, NT = C::NT;
  constexpr int KB = C::KPW / 16;  // 16-key sub-blocks
  constexpr int CH = RB / 16;      // 16-byte chunks per cache row
  const int g = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t kbase = smem_u32(kt);
  const uint32_t nib_lo = kNibLo, nib_hi = kNibHi;

  // ---- S = Q K^T in fp16 with biased K codes. Each 16-byte chunk of a K row
  // is one scale group for int4 (32 channels); its accumulator is folded into
  // the scores as soon as its products are done: sv = sum_g ks_g (acc_g - c_g).
  // int4 reads the constants c_g of its rows g, g + 8 from shared memory
  // (qcs: prepare_q_rows' table at row g; row g + 8 at + 8 NG) rather than
  // holding them in registers through the block.
  // The sub-blocks' products are independent: their MMA chains interleave.
  float sv[KB][2][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) sv[kb][nt][e] = 0.f;
  float acc8[KB][2][4];  // int8: one accumulator over all chunks, starting at -bias
#pragma unroll
  for (int kb = 0; kb < KB; ++kb)
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc8[kb][nt][e] = KIND == KV_I8 ? -qc[e >> 1][0] : 0.f;
  const int krow = row0 + ((mi >> 1) << 3) + ri;
#pragma unroll
  for (int kc = 0; kc < CH; kc += 2) {
    uint32_t r[KB][4];  // (n-tile 0, chunk kc), (n-tile 0, kc+1), (n-tile 1, kc), (n-tile 1, kc+1)
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) ldsm_x4(r[kb], kbase + swz<SW>((krow + 16 * kb) * RB + (kc + (mi & 1)) * 16));
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int ch = kc + hh;
      if constexpr (KIND == KV_I8) {
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const uint32_t x = r[kb][nt * 2 + hh] ^ 0x80808080u;  // bytes u = code + 128
            mma_f16_16816(acc8[kb][nt], qa[ch], __byte_perm(x, 0x64646464u, 0x5140),
                          __byte_perm(x, 0x64646464u, 0x7362));
          }
      } else {
        float acc[KB][2][4];  // this group's products, starting at -bias
        // the group's two Q fragments (k-steps 2 ch, 2 ch + 1), from shared memory
        const uint4 va = qa_s[(2 * ch) * 32 + lane], vb = qa_s[(2 * ch + 1) * 32 + lane];
        const uint32_t qlo[4] = {va.x, va.y, va.z, va.w}, qhi[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[kb][nt][e] = -qcs[(e >> 1) * 8 * NG + ch];
            // raw nibble k (= code & 15) is channel 32ch + 8c + k; masking it
            // and XOR-ing in 8 and the exponent of 1024 is one LOP3 per pair
            const uint32_t x = r[kb][nt * 2 + hh];
            const uint32_t y = x >> 8;
            mma_f16_16816(acc[kb][nt], qlo, nib_lo_f16_biased(x, nib_lo), nib_lo_f16_biased(y, nib_lo));
            mma_f16_16816(acc[kb][nt], qhi, nib_hi_f16_biased(x, nib_hi),
                          nib_hi_f16_biased(y, nib_hi));
          }
#pragma unroll
        for (int kb = 0; kb < KB; ++kb)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int key = 16 * kb + nt * 8 + 2 * c + (e & 1);
              sv[kb][nt][e] = fmaf(acc[kb][nt][e], ksc[(row0 + key) * NG + ch], sv[kb][nt][e]);
            }
      }
    }
  }
  if constexpr (KIND == KV_I8) {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 16 * kb + nt * 8 + 2 * c + (e & 1);
          sv[kb][nt][e] = acc8[kb][nt][e] * ksc[row0 + key];
        }
  }

  // ---- row scale, mask by selection (a block whose keys every row of the
  // warp sees, which is every block but a split's last, needs no selection)
  const bool full = __all_sync(0xffffffffu, tok_row0 + C::KPW <= min(lim0, lim1));
  float s[KB][2][4];
  if (full) {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
          const float2 r2 = __fmul2_rn(make_float2(sv[kb][nt][2 * hr], sv[kb][nt][2 * hr + 1]),
                                       make_float2(rs[hr], rs[hr]));
          s[kb][nt][2 * hr] = r2.x;
          s[kb][nt][2 * hr + 1] = r2.y;
        }
  } else {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int key = 16 * kb + nt * 8 + 2 * c + (e & 1);
          const int hr = e >> 1;
          const int lim = hr ? lim1 : lim0;
          s[kb][nt][e] = (tok_row0 + key < lim) ? sv[kb][nt][e] * rs[hr] : -INFINITY;
        }
      }
  }
  float p[KB][2][4], al[2];
  // int4 may let p reach 2^kLazyMax (fp16 P; its V scale stays with V); int8
  // folds the V scale into P, so it keeps the exact running max
  const bool rescale = softmax_update_kb<KB, KIND == KV_I4>(s, p, m, l, al);
  // alpha-rescale of O if the max moved
  auto rescale_o = [&](auto &oo) {  // O fragments and the V-bias row sums alike
    if (rescale) {
#pragma unroll
      for (int j = 0; j < static_cast<int>(sizeof(oo) / sizeof(oo[0])); ++j) {
        oo[j][0] *= al[0];
        oo[j][1] *= al[0];
        oo[j][2] *= al[1];
        oo[j][3] *= al[1];
      }
    }
  };
  if constexpr (!C::O_TMEM) rescale_o(o);  // (O in tensor memory is rescaled once loaded)
  if constexpr (C::V_SUB) rescale_o(ra);

  // ---- P as the fp16 A operand (int8: the per-key V scale folded in)
  uint32_t pa[KB][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    if constexpr (KIND == KV_I8) {
      float pv[2][4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float vs = vsc[row0 + 16 * kb + nt * 8 + 2 * c + (e & 1)];
          pv[nt][e] = p[kb][nt][e] * vs;
        }
      pa[kb][0] = pack_f16x2(pv[0][0], pv[0][1]);
      pa[kb][1] = pack_f16x2(pv[0][2], pv[0][3]);
      pa[kb][2] = pack_f16x2(pv[1][0], pv[1][1]);
      pa[kb][3] = pack_f16x2(pv[1][2], pv[1][3]);
    } else {
      pa[kb][0] = pack_f16x2(p[kb][0][0], p[kb][0][1]);
      pa[kb][1] = pack_f16x2(p[kb][0][2], p[kb][0][3]);
      pa[kb][2] = pack_f16x2(p[kb][1][0], p[kb][1][1]);
      pa[kb][3] = pack_f16x2(p[kb][1][2], p[kb][1][3]);
    }
  }

  // ---- V fragments: keys (2c, 2c+1) -> b0, (2c+8, 2c+9) -> b1 of each
  // sub-block (keys at or past c1 meet a zero probability; their codes and
  // scales are finite)
  int vrows[KB][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    const int kA = row0 + 16 * kb + 2 * c, kB = kA + 8;
    vrows[kb][0] = kA;
    vrows[kb][1] = kA + 1;
    vrows[kb][2] = kB;
    vrows[kb][3] = kB + 1;
  }
  if constexpr (KIND == KV_I8) {
    static_assert(NT % 4 == 0, "int8 V words");
    static_assert(!C::O_TMEM, "int8 keeps O in registers");
    // ldmatrix.trans of 8 keys x 16 channels (16 bytes) gives thread (g, c)
    // the codes of channels 16 s + 2 g and + 1 of keys 2c, 2c + 1 (bytes 0, 2
    // and 1, 3 of the register): n-tile 2 s + e holds channel 16 s + 2 n + e
    // at MMA column n. Keys at or past c1 meet a zero probability (their codes
    // are finite). Codes as subnormals; ra accumulates the row sums of P.
    const uint32_t vbase = smem_u32(vt);
    const uint32_t u8_sub = kU8Sub, ones = kOnesF16;
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      mma_f16_16816(ra[0], pa[kb], ones, ones);
      const int key = row0 + 16 * kb + 8 * ((lane >> 3) & 1) + (lane & 7);
#pragma unroll
      for (int sp = 0; sp < C::D / 16; sp += 2) {
        uint32_t R[4];  // (keys 0-7, slice sp), (keys 8-15, sp), (keys 0-7, sp + 1), (keys 8-15, sp + 1)
        ldsm_x4_t(R, vbase + swz<SW>(key * RB + 16 * (sp + (lane >> 4))));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int sl = sp + h2;
          const uint32_t lo = R[2 * h2], hi = R[2 * h2 + 1];
          mma_f16_16816(o[2 * sl], pa[kb], i8pair_to_f16_sub(lo, u8_sub), i8pair_to_f16_sub(hi, u8_sub));
          mma_f16_16816(o[2 * sl + 1], pa[kb], i8pair_to_f16_sub(lo >> 8, u8_sub),
                        i8pair_to_f16_sub(hi >> 8, u8_sub));
        }
      }
    }
  } else {
    static_assert(NT == 4 * NG, "int4: four n-tiles per 32-channel scale group");
    static_assert(C::O_TMEM, "int4 keeps O in tensor memory");
    // O from tensor memory: it waits there through the score half of the
    // block, which then runs with D/2 fewer live registers (the previous
    // block's store has long landed; the wait only orders it before the load)
    float ot[NT][4];
    tmem_wait_st();
#pragma unroll
    for (int i = 0; i < NT / 8; ++i) tmem_ld32(tm_o + 32 * i, &ot[8 * i][0]);
    tmem_wait_ld();
    rescale_o(ot);
    // V codes paired by ldmatrix.trans: matrix (keys 8h .. 8h + 7 of the
    // sub-block, 16 bytes of group gi) gives thread (g, c) the 4 nibbles
    // (channels 32 gi + 4 g .. + 3) of keys 8h + 2c and 8h + 2c + 1; n-tile
    // 4 gi + q holds channel 32 gi + 4 n + q at MMA column n. Each group's V
    // scale multiplies the probabilities (the A operand) instead of V.
    const uint32_t vbase = smem_u32(vt);
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      // V-scale pairs per group of the thread's keys (2c, 2c + 1) and
      // (2c + 8, 2c + 9) of this sub-block
      uint32_t sp0[NG], sp1[NG];
      {
        float sk[4][NG];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
#pragma unroll
          for (int gi = 0; gi < NG; ++gi) sk[i][gi] = vsc[vrows[kb][i] * NG + gi];
        }
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) {
          sp0[gi] = pack_f16x2(sk[0][gi], sk[1][gi]);
          sp1[gi] = pack_f16x2(sk[2][gi], sk[3][gi]);
        }
      }
#pragma unroll
      for (int gp = 0; gp < NG; gp += 2) {  // two groups per ldmatrix.x4
        uint32_t R[4];  // (keys 0-7, gp), (keys 8-15, gp), (keys 0-7, gp + 1), (keys 8-15, gp + 1)
        const int key = row0 + 16 * kb + 8 * ((lane >> 3) & 1) + (lane & 7);
        ldsm_x4_t(R, vbase + swz<SW>(key * RB + 16 * (gp + (lane >> 4))));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int gi = gp + h2;
          const uint32_t aw[4] = {hmul2_u32(pa[kb][0], sp0[gi]), hmul2_u32(pa[kb][1], sp0[gi]),
                                  hmul2_u32(pa[kb][2], sp1[gi]), hmul2_u32(pa[kb][3], sp1[gi])};
          const uint32_t lo = R[2 * h2], hi = R[2 * h2 + 1];
          const uint32_t lo8 = lo >> 8, hi8 = hi >> 8;
          mma_f16_16816(ot[4 * gi + 0], aw, hsub2_u32(nib_lo_f16_biased(lo, nib_lo), 1032.0f),
                        hsub2_u32(nib_lo_f16_biased(hi, nib_lo), 1032.0f));
          mma_f16_16816(ot[4 * gi + 1], aw, hfma2_u32(nib_hi_f16_biased(lo, nib_hi), 1.0f / 16.0f, -72.0f),
                        hfma2_u32(nib_hi_f16_biased(hi, nib_hi), 1.0f / 16.0f, -72.0f));
          mma_f16_16816(ot[4 * gi + 2], aw, hsub2_u32(nib_lo_f16_biased(lo8, nib_lo), 1032.0f),
                        hsub2_u32(nib_lo_f16_biased(hi8, nib_lo), 1032.0f));
          mma_f16_16816(ot[4 * gi + 3], aw, hfma2_u32(nib_hi_f16_biased(lo8, nib_hi), 1.0f / 16.0f, -72.0f),
                        hfma2_u32(nib_hi_f16_biased(hi8, nib_hi), 1.0f / 16.0f, -72.0f));
        }
      }
    }
#pragma unroll
    for (int i = 0; i < NT / 8; ++i) tmem_st32(tm_o + 32 * i, &ot[8 * i][0]);
  }
}

// ----------------------------------------------------------------------------
// One block of C::KPW keys (KB = KPW / 16 sub-blocks of 16 sharing one
// softmax step) of one warp, quantised cache, for tiles of at most 8 query
// rows ("narrow"). The 16 keys of a sub-block are the M dimension of the MMAs
// and the rows the 8-wide N dimension, so no tile is mostly padding:
//   S^T (16 keys x 8 rows)  = K (keys x channels) Q^T,
//   O^T (16 channels x 8 rows) += V^T (channels x keys) P^T.
// The K codes become A fragments straight from ldmatrix, in the channel order
// of warp_block_q's B fragments (qb[ks] = that order's row-g Q fragment).
// S^T's fragment holds keys (g, g + 8) x rows (2c, 2c + 1): a row's max
// reduces over the 8 lanes of one c. P^T reaches the B-fragment layout of PV
// through two 8x8 transposes (movmatrix). V codes become A fragments from
// ldmatrix.trans (see the V^T step below for the channel of each m-tile
// slot); o[j][0,1] / o[j][2,3] hold the m-tile's slot g / g + 8 channel for
// rows (2c, 2c + 1).
// l holds the thread's partial row sums over its keys (reduced across the 8
// lanes of a row by the caller); m is the full row max.
template <class C, int KIND>
__device__ __forceinline__ void warp_block_km(const uint8_t *kt, const uint8_t *vt, const float *ksc,
                                              const float *vsc, int row0, const uint32_t (&qb)[C::D / 16][2],
                                              const float (&qc)[2][C::NG], const float (&rs)[2],
                                              float (&o)[C::OT][4], float (&ra)[C::NR][4], float (&m)[2],
                                              float (&l)[2], int tok_row0, int c1, int lim0, int lim1, int lane) {
  constexpr int NG = C::NG, RB = C::ROW_BYTES, SW = C::BOX_BYTES, NT = C::NT;
  constexpr int KB = C::KPW / 16;  // 16-key sub-blocks
  constexpr int CH = RB / 16;      // 16-byte chunks per cache row
  const int g = lane >> 2, c = lane & 3;
  const int mi = lane >> 3, ri = lane & 7;
  const uint32_t kbase = smem_u32(kt);
  const uint32_t nib_lo = kNibLo, nib_hi = kNibHi;

  // ---- S^T = K Q^T: sv[kb] = (key g, row 2c), (g, 2c+1), (g+8, 2c), (g+8, 2c+1)
  float sv[KB][4];
  float acc8[KB][4];  // int8: from -bias
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    sv[kb][0] = sv[kb][1] = sv[kb][2] = sv[kb][3] = 0.f;
    acc8[kb][0] = acc8[kb][2] = -qc[0][0];
    acc8[kb][1] = acc8[kb][3] = -qc[1][0];
  }
  const int krow = row0 + ((mi >> 1) << 3) + ri;
#pragma unroll
  for (int kc = 0; kc < CH; kc += 2) {
    uint32_t r[KB][4];  // (key g, chunk kc), (key g, kc + 1), (key g + 8, kc), (key g + 8, kc + 1)
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) ldsm_x4(r[kb], kbase + swz<SW>((krow + 16 * kb) * RB + (kc + (mi & 1)) * 16));
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int ch = kc + hh;
#pragma unroll
      for (int kb = 0; kb < KB; ++kb) {
        if constexpr (KIND == KV_I8) {
          const uint32_t xg = r[kb][hh] ^ 0x80808080u, x8 = r[kb][2 + hh] ^ 0x80808080u;  // bytes u = code + 128
          const uint32_t a[4] = {__byte_perm(xg, 0x64646464u, 0x5140), __byte_perm(x8, 0x64646464u, 0x5140),
                                 __byte_perm(xg, 0x64646464u, 0x7362), __byte_perm(x8, 0x64646464u, 0x7362)};
          mma_f16_16816(acc8[kb], a, qb[ch][0], qb[ch][1]);
        } else {
          float acc[4] = {-qc[0][ch], -qc[1][ch], -qc[0][ch], -qc[1][ch]};
          const uint32_t xg = r[kb][hh], x8 = r[kb][2 + hh];
          const uint32_t yg = xg >> 8, y8 = x8 >> 8;
          const uint32_t alo[4] = {nib_lo_f16_biased(xg, nib_lo), nib_lo_f16_biased(x8, nib_lo),
                                   nib_lo_f16_biased(yg, nib_lo), nib_lo_f16_biased(y8, nib_lo)};
          const uint32_t ahi[4] = {nib_hi_f16_biased(xg, nib_hi), nib_hi_f16_biased(x8, nib_hi),
                                   nib_hi_f16_biased(yg, nib_hi), nib_hi_f16_biased(y8, nib_hi)};
          mma_f16_16816(acc, alo, qb[2 * ch][0], qb[2 * ch][1]);
          mma_f16_16816(acc, ahi, qb[2 * ch + 1][0], qb[2 * ch + 1][1]);
          const float kg = ksc[(row0 + 16 * kb + g) * NG + ch], k8 = ksc[(row0 + 16 * kb + g + 8) * NG + ch];
          sv[kb][0] = fmaf(acc[0], kg, sv[kb][0]);
          sv[kb][1] = fmaf(acc[1], kg, sv[kb][1]);
          sv[kb][2] = fmaf(acc[2], k8, sv[kb][2]);
          sv[kb][3] = fmaf(acc[3], k8, sv[kb][3]);
        }
      }
    }
  }
  if constexpr (KIND == KV_I8) {
#pragma unroll
    for (int kb = 0; kb < KB; ++kb) {
      const float kg = ksc[row0 + 16 * kb + g], k8 = ksc[row0 + 16 * kb + g + 8];
      sv[kb][0] = acc8[kb][0] * kg;
      sv[kb][1] = acc8[kb][1] * kg;
      sv[kb][2] = acc8[kb][2] * k8;
      sv[kb][3] = acc8[kb][3] * k8;
    }
  }

  // ---- row scale, mask by selection, online softmax (rows 2c, 2c + 1)
  const bool full = __all_sync(0xffffffffu, tok_row0 + C::KPW <= min(lim0, lim1));
  float s[KB][4];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    s[kb][0] = sv[kb][0] * rs[0];
    s[kb][1] = sv[kb][1] * rs[1];
    s[kb][2] = sv[kb][2] * rs[0];
    s[kb][3] = sv[kb][3] * rs[1];
    if (!full) {
      const int kg = tok_row0 + 16 * kb + g, k8 = kg + 8;
      if (kg >= lim0) s[kb][0] = -INFINITY;
      if (kg >= lim1) s[kb][1] = -INFINITY;
      if (k8 >= lim0) s[kb][2] = -INFINITY;
      if (k8 >= lim1) s[kb][3] = -INFINITY;
    }
  }
  float mx0 = fmaxf(s[0][0], s[0][2]), mx1 = fmaxf(s[0][1], s[0][3]);
#pragma unroll
  for (int kb = 1; kb < KB; ++kb) {
    mx0 = fmaxf(mx0, fmaxf(s[kb][0], s[kb][2]));
    mx1 = fmaxf(mx1, fmaxf(s[kb][1], s[kb][3]));
  }
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
  }
  const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
  const float b0 = mn0 == -INFINITY ? 0.f : mn0;  // a row with no key yet keeps m = -inf
  const float b1 = mn1 == -INFINITY ? 0.f : mn1;
  const float al0 = fast_exp2(m[0] - b0), al1 = fast_exp2(m[1] - b1);
  m[0] = mn0;
  m[1] = mn1;
  float p[KB][4];
  float ps0 = 0.f, ps1 = 0.f;
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    p[kb][0] = fast_exp2(s[kb][0] - b0);
    p[kb][1] = fast_exp2(s[kb][1] - b1);
    p[kb][2] = fast_exp2(s[kb][2] - b0);
    p[kb][3] = fast_exp2(s[kb][3] - b1);
    ps0 += p[kb][0] + p[kb][2];
    ps1 += p[kb][1] + p[kb][3];
  }
  l[0] = fmaf(l[0], al0, ps0);
  l[1] = fmaf(l[1], al1, ps1);
  if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
    for (int j = 0; j < C::OT; ++j) {
      o[j][0] *= al0;
      o[j][1] *= al1;
      o[j][2] *= al0;
      o[j][3] *= al1;
    }
    if constexpr (C::V_SUB) {
      ra[0][0] *= al0;
      ra[0][1] *= al1;
      ra[0][2] *= al0;
      ra[0][3] *= al1;
    }
  }

  // ---- P^T -> the B fragments of PV (int8: the per-key V scale folded in)
  uint32_t pb0[KB], pb1[KB];
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    if constexpr (KIND == KV_I8) {
      const float vg = vsc[row0 + 16 * kb + g], v8 = vsc[row0 + 16 * kb + g + 8];
      p[kb][0] *= vg;
      p[kb][1] *= vg;
      p[kb][2] *= v8;
      p[kb][3] *= v8;
    }
    // (keys g | g + 8) x (rows 2c, 2c + 1) -> row g x (keys 2c, 2c + 1 | 2c + 8, 2c + 9)
    pb0[kb] = movmatrix_trans(pack_f16x2(p[kb][0], p[kb][1]));
    pb1[kb] = movmatrix_trans(pack_f16x2(p[kb][2], p[kb][3]));
  }

  // ---- V^T as A fragments, from ldmatrix.trans of 8 keys x 16 bytes: thread
  // (g, c) gets the 16-bit element g of keys 2c and 2c + 1 (and of 2c + 8,
  // 2c + 9 from the next matrix), so each register pairs two keys' codes as
  // the MMA wants them, with no byte permutes. Keys at or past c1 meet a zero
  // probability (their codes and scales are finite).
  //   int8: m-tile j = channels 16 j ..: row g = channel 16 j + 2 g (bytes 0
  //         and 2 of the register), row g + 8 = 16 j + 2 g + 1 (bytes 1, 3).
  //   int4: m-tile j = 2 gi + qq inside scale group gi: row g = channel
  //         32 gi + 4 g + 2 qq, row g + 8 = the next channel; the group's V
  //         scale multiplies the probabilities (the B operand).
  // int8 codes enter as subnormals, and ra sums the B operand over the keys
  // (an MMA with an A operand of ones).
  const uint32_t vbase = smem_u32(vt);
  const uint32_t ones = kOnesF16;
  const uint32_t ones4[4] = {ones, ones, ones, ones};
#pragma unroll
  for (int kb = 0; kb < KB; ++kb) {
    const int key = row0 + 16 * kb + 8 * ((lane >> 3) & 1) + (lane & 7);
    if constexpr (KIND == KV_I8) {
      static_assert(C::OT % 2 == 0, "int8: 16-channel slices in pairs");
      const uint32_t u8_sub = kU8Sub;
      mma_f16_16816(ra[0], ones4, pb0[kb], pb1[kb]);
#pragma unroll
      for (int sp = 0; sp < C::OT; sp += 2) {
        uint32_t R[4];  // (keys 0-7, slice sp), (keys 8-15, sp), (keys 0-7, sp + 1), (keys 8-15, sp + 1)
        ldsm_x4_t(R, vbase + swz<SW>(key * RB + 16 * (sp + (lane >> 4))));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const uint32_t lo = R[2 * h2], hi = R[2 * h2 + 1];
          const uint32_t a[4] = {i8pair_to_f16_sub(lo, u8_sub), i8pair_to_f16_sub(lo >> 8, u8_sub),
                                 i8pair_to_f16_sub(hi, u8_sub), i8pair_to_f16_sub(hi >> 8, u8_sub)};
          mma_f16_16816(o[sp + h2], a, pb0[kb], pb1[kb]);
        }
      }
    } else {
      static_assert(C::OT == 2 * NG && NG % 2 == 0, "int4: two m-tiles per 32-channel scale group");
      const int kA = row0 + 16 * kb + 2 * c, kB = kA + 8;
      const int vrows[4] = {kA, kA + 1, kB, kB + 1};
      float sk[4][NG];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int gi = 0; gi < NG; ++gi) sk[i][gi] = vsc[vrows[i] * NG + gi];
      }
      auto code = [&](uint32_t t, int q) {  // nibble q of two keys -> exact f16x2 codes
        return (q & 1) ? hfma2_u32(nib_hi_f16_biased(t >> (4 * (q - 1)), nib_hi), 1.0f / 16.0f, -72.0f)
                       : hsub2_u32(nib_lo_f16_biased(t >> (4 * q), nib_lo), 1032.0f);
      };
#pragma unroll
      for (int gp = 0; gp < NG; gp += 2) {
        uint32_t R[4];  // (keys 0-7, group gp), (keys 8-15, gp), (keys 0-7, gp + 1), (keys 8-15, gp + 1)
        ldsm_x4_t(R, vbase + swz<SW>(key * RB + 16 * (gp + (lane >> 4))));
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
          const int gi = gp + h2;
          const uint32_t b0 = hmul2_u32(pb0[kb], pack_f16x2(sk[0][gi], sk[1][gi]));
          const uint32_t b1 = hmul2_u32(pb1[kb], pack_f16x2(sk[2][gi], sk[3][gi]));
          const uint32_t lo = R[2 * h2], hi = R[2 * h2 + 1];
#pragma unroll
          for (int qq = 0; qq < 2; ++qq) {
            const uint32_t a[4] = {code(lo, 2 * qq), code(lo, 2 * qq + 1), code(hi, 2 * qq), code(hi, 2 * qq + 1)};
            mma_f16_16816(o[2 * gi + qq], a, b0, b1);
          }
        }
      }
    }
  }
}

// The int8 V codes entered PV as subnormals (see kU8Sub): O = 2^24 O_raw -
// 128 R, with R the row sums in ra[0], whose entries line up with those of
// every O fragment (16-row: rows g, g + 8; narrow: rows 2c, 2c + 1).
template <class C>
__device__ __forceinline__ void remove_v_bias(float (&o)[C::OT][4], const float (&ra)[C::NR][4]) {
#pragma unroll
  for (int j = 0; j < C::OT; ++j) {
#pragma unroll
    for (int e = 0; e < 4; ++e) o[j][e] = fmaf(o[j][e], 16777216.0f, -128.0f * ra[0][e]);
  }
}

// Quantised caches run Q K^T in fp16. Each query row is scaled by an exact
// power of two, 2^-e, so that its largest |q| lies in [2^14, 2^15): every bf16
// value then converts to fp16 exactly (8 significant bits fit 11; values below
// 2^-28 of the row max, which round, cannot move an fp32 dot product). The
// K codes enter the product biased (see warp_block_q), and the bias is taken
// back out of the fp32 scores with per-(row, group) constants:
//   int8: K = 1024 + u, u = code + 128       -> c = 1152 * sum_d q'_d
//   int4: even channels K = 1024 + u, odd channels K = 1024 + 16u with Q/16
//         (u = code + 8)                      -> c_g = 1032 * sum_even q' + 72 * sum_odd q'
// qinfo[r] = 2^e, qinfo[16 + r * NG + g] = c_g (fp32). 128 consumer threads,
// 8 per row.
template <class C, int KIND>
__device__ __forceinline__ void prepare_q_rows(const uint8_t *qs, float *qinfo, int tid) {
  constexpr int D = C::D, NG = C::NG, PER = D / 8;  // channels per thread
  const int row = tid >> 3, k = tid & 7;
  const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(qs + row * C::QROW) + k * PER;
  float v[PER];
  float mx = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    v[i] = __bfloat162float(q[i]);
    mx = fmaxf(mx, fabsf(v[i]));
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  int E = 0;
  if (mx > 0.f && mx <= 3.0e38f) frexpf(mx, &E);
  E = max(E, -100);  // keep 2^(15-E) finite for rows of tiny values
  const float down = ldexpf(1.0f, 15 - E);  // exact power of two
  float se = 0.f, so = 0.f;
#pragma unroll
  for (int i = 0; i < PER; ++i) {
    if (i & 1) so += v[i] * down;
    else se += v[i] * down;
  }
  if constexpr (KIND == KV_I8) {
    float c = 1152.0f * (se + so);
    c += __shfl_xor_sync(0xffffffffu, c, 1);
    c += __shfl_xor_sync(0xffffffffu, c, 2);
    c += __shfl_xor_sync(0xffffffffu, c, 4);
    if (k == 0) qinfo[16 + row] = c;
  } else {
    constexpr int TPG = 32 / PER;  // threads per 32-channel group
    float c = 1032.0f * se + 72.0f * so;
#pragma unroll
    for (int o = 1; o < TPG; o <<= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (k % TPG == 0) qinfo[16 + row * NG + k / TPG] = c;
  }
  if (k == 0) qinfo[row] = ldexpf(1.0f, E - 15);
}

// Q A fragments (fp16, prescaled) in the channel order warp_block_q feeds K in.
//  int8, k-step ks (16-byte chunk of 16 codes): slots (2c, 2c+1) are channels
//    16ks+4c+{0,1}, slots (2c+8, 2c+9) are 16ks+4c+{2,3}.
//  int4, chunk ch of 32 codes, base = 32ch+8c: k-step 2ch has slots
//    (2c, 2c+1) = base+{0,4}, (2c+8, 2c+9) = base+{2,6}; k-step 2ch+1 has
//    base+{1,5} and base+{3,7}, divided by 16.
template <class C, int KIND>
__device__ __forceinline__ void build_q_fragments(const uint8_t *qs, const float *qinfo,
                                                  uint32_t (&qa)[C::D / 16][4], int lane) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    const int row = g + 8 * half;
    const __nv_bfloat16 *q = reinterpret_cast<const __nv_bfloat16 *>(qs + row * C::QROW);
    const float down = 1.0f / qinfo[row];  // exact: qinfo[row] is a power of two
    auto qv = [&](int d) { return __bfloat162float(q[d]) * down; };
    if constexpr (KIND == KV_I8) {
#pragma unroll
      for (int ks = 0; ks < C::D / 16; ++ks) {
        const int d = 16 * ks + 4 * c;
        qa[ks][half] = pack_f16x2(qv(d), qv(d + 1));
        qa[ks][2 + half] = pack_f16x2(qv(d + 2), qv(d + 3));
      }
    } else {
#pragma unroll
      for (int ch = 0; ch < C::D / 32; ++ch) {
        const int d = 32 * ch + 8 * c;
        qa[2 * ch][half] = pack_f16x2(qv(d), qv(d + 4));
        qa[2 * ch][2 + half] = pack_f16x2(qv(d + 2), qv(d + 6));
        qa[2 * ch + 1][half] = pack_f16x2(qv(d + 1) * 0.0625f, qv(d + 5) * 0.0625f);
        qa[2 * ch + 1][2 + half] = pack_f16x2(qv(d + 3) * 0.0625f, qv(d + 7) * 0.0625f);
      }
    }
  }
}

// ----------------------------------------------------------------------------

template <class C>
__device__ __forceinline__ void write_row_outputs(const Stage1Params &p, bool fused, int b, int h,
                                                  int s, int row_glob, int d0, const float *vals,
                                                  int nvals, float lse_nat, bool write_lse) {
  const int t = row_glob / p.G, g = row_glob - t * p.G;
  const int hq = h * p.G + g;
  if (fused) {
    if (p.out_f32) {
      float *dst = reinterpret_cast<float *>(p.out) + b * p.o_sb + t * p.o_st + hq * p.o_sh + d0;
      for (int i = 0; i < nvals; i += 4)
        *reinterpret_cast<float4 *>(dst + i) = make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
    } else {
      __nv_bfloat16 *dst =
          reinterpret_cast<__nv_bfloat16 *>(p.out) + b * p.o_sb + t * p.o_st + hq * p.o_sh + d0;
      for (int i = 0; i < nvals; i += 8) {
        uint4 v;
        v.x = pack_bf16x2(vals[i + 0], vals[i + 1]);
        v.y = pack_bf16x2(vals[i + 2], vals[i + 3]);
        v.z = pack_bf16x2(vals[i + 4], vals[i + 5]);
        v.w = pack_bf16x2(vals[i + 6], vals[i + 7]);
        *reinterpret_cast<uint4 *>(dst + i) = v;
      }
    }
    if (write_lse && p.lse) p.lse[b * p.l_sb + t * p.l_st + hq * p.l_sh] = lse_nat;
  } else {
    const int64_t rowi = ((static_cast<int64_t>(b) * p.Tq + t) * p.Hq + hq) * p.s_cap + s;
    float *dst = p.o_part + rowi * C::D + d0;
    for (int i = 0; i < nvals; i += 4)
      *reinterpret_cast<float4 *>(dst + i) = make_float4(vals[i], vals[i + 1], vals[i + 2], vals[i + 3]);
    if (write_lse) p.lse_part[rowi] = lse_nat;
  }
}

// One output row from a warp: lane l holds columns 2l + 64k and 2l + 64k + 1
// in vals[k]; lane 0 writes the LSE. Destinations as in write_row_outputs.
template <class C>
__device__ __forceinline__ void write_row_pairs(const Stage1Params &p, bool fused, int b, int h, int s,
                                                int row_glob, int lane, const float2 (&vals)[C::D / 64],
                                                float lse_nat) {
  const int t = row_glob / p.G, g = row_glob - t * p.G;
  const int hq = h * p.G + g;
  if (fused) {
    if (p.out_f32) {
      float *dst = reinterpret_cast<float *>(p.out) + b * p.o_sb + t * p.o_st + hq * p.o_sh + 2 * lane;
#pragma unroll
      for (int k = 0; k < C::D / 64; ++k) *reinterpret_cast<float2 *>(dst + 64 * k) = vals[k];
    } else {
      __nv_bfloat16 *dst =
          reinterpret_cast<__nv_bfloat16 *>(p.out) + b * p.o_sb + t * p.o_st + hq * p.o_sh + 2 * lane;
#pragma unroll
      for (int k = 0; k < C::D / 64; ++k)
        *reinterpret_cast<uint32_t *>(dst + 64 * k) = pack_bf16x2(vals[k].x, vals[k].y);
    }
    if (lane == 0 && p.lse) p.lse[b * p.l_sb + t * p.l_st + hq * p.l_sh] = lse_nat;
  } else {
    const int64_t rowi = ((static_cast<int64_t>(b) * p.Tq + t) * p.Hq + hq) * p.s_cap + s;
    float *dst = p.o_part + rowi * C::D + 2 * lane;
#pragma unroll
    for (int k = 0; k < C::D / 64; ++k) *reinterpret_cast<float2 *>(dst + 64 * k) = vals[k];
    if (lane == 0) p.lse_part[rowi] = lse_nat;
  }
}

// The merge of the last split CTA of a tile: for each of the tile's rows, the
// nv non-empty split partials (o_s, lse_s) combine as
//   M = max_s lse_s, w_s = exp(lse_s - M), out = sum w_s o_s / sum w_s,
//   lse = M + ln(sum w_s)
// (the stage-2 merge). One warp per row, lanes over the D columns, eight
// partial loads in flight; partials written by other CTAs are read through L2.
template <class C>
__device__ __forceinline__ void merge_tile(const Stage1Params &p, int b, int h, int rt, int nv, int warp,
                                           int nwarps, int lane) {
  constexpr int D = C::D, VPL = D / 32;
  const int nrows = min(16, p.R - rt * 16);
  for (int r = warp; r < nrows; r += nwarps) {
    const int rg = rt * 16 + r;
    const int t = rg / p.G, hq = h * p.G + (rg - t * p.G);
    const int64_t base = ((static_cast<int64_t>(b) * p.Tq + t) * p.Hq + hq) * p.s_cap;
    const float l0 = lane < nv ? __ldcg(p.lse_part + base + lane) : -INFINITY;
    const float l1 = lane + 32 < nv ? __ldcg(p.lse_part + base + lane + 32) : -INFINITY;
    float M = fmaxf(l0, l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float w0 = (l0 == -INFINITY) ? 0.f : expf(l0 - M);
    const float w1 = (l1 == -INFINITY) ? 0.f : expf(l1 - M);
    float Z = w0 + w1;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Z += __shfl_xor_sync(0xffffffffu, Z, o);
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float *op = p.o_part + base * D + lane * VPL;
    for (int s0 = 0; s0 < nv; s0 += 8) {
      float w[8];
      float v[8][VPL];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int sp = s0 + u;
        const float wa = __shfl_sync(0xffffffffu, w0, sp & 31);
        const float wb = __shfl_sync(0xffffffffu, w1, sp & 31);
        w[u] = sp < nv ? (sp < 32 ? wa : wb) : 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i) v[u][i] = 0.f;
        if (w[u] > 0.f) {
          if constexpr (VPL == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4 *>(op + sp * D));
            v[u][0] = x.x;
            v[u][1] = x.y;
            v[u][2] = x.z;
            v[u][3] = x.w;
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2 *>(op + sp * D));
            v[u][0] = x.x;
            v[u][1] = x.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
#pragma unroll
        for (int i = 0; i < VPL; ++i) acc[i] = fmaf(w[u], v[u][i], acc[i]);
    }
    const float inv = Z > 0.f ? 1.f / Z : 0.f;
    const int64_t ob = b * p.o_sb + t * p.o_st + hq * p.o_sh + lane * VPL;
    if (p.out_f32) {
      float *dst = reinterpret_cast<float *>(p.out) + ob;
#pragma unroll
      for (int i = 0; i < VPL; ++i) dst[i] = acc[i] * inv;
    } else {
      __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + ob;
#pragma unroll
      for (int i = 0; i < VPL; i += 2)
        *reinterpret_cast<uint32_t *>(dst + i) = pack_bf16x2(acc[i] * inv, acc[i + 1] * inv);
    }
    if (lane == 0 && p.lse) p.lse[b * p.l_sb + t * p.l_st + hq * p.l_sh] = Z > 0.f ? M + logf(Z) : -INFINITY;
  }
}

// L2 prefetch of a CTA's first STAGES blocks of K and V, issued before the
// dependency wait by the producer warp. The length and page ids are read with
// relaxed loads while the previous kernel may still be writing them: they
// only choose which boxes to prefetch (a stale page id costs bandwidth; an id
// outside the pool is skipped), and the kernel reads both again after the
// wait. TMA drops boxes that fall outside the tensor.
// Returns the (clamped) length the prefetch used.
template <class C>
__device__ __forceinline__ int prefetch_first_blocks(const CUtensorMap *tmk, const CUtensorMap *tmv,
                                                     const Stage1Params &p, int b, int h, int s,
                                                     int S_req, int lane) {
  if (lane == 0) {
    tma_prefetch_desc(tmk);
    tma_prefetch_desc(tmv);
  }
  const int P = p.page_size;
  const int cap = p.max_pages * P;
  int L = ld_relaxed_gpu(p.seqlens + b * p.sl_s);
  L = L < 0 ? 0 : (L > cap ? cap : L);
  const int chunk = split_chunk(L, S_req, p.log2_page, p.chunk_min);
  const int c0 = s * chunk;
  const int c1 = min(L, c0 + chunk);
  if (c0 >= c1) return L;
  const int t1 = min(c1, c0 + C::STAGES * C::BLOCK_N);
  const int log2_seg = P < C::SEG_MAX ? p.log2_page : 6;
  const int nseg = (t1 - c0 + (1 << log2_seg) - 1) >> log2_seg;
  const int *pt = p.page_table + b * p.pt_sb;
  for (int i = lane; i < nseg; i += 32) {
    const int ts = c0 + (i << log2_seg);
    const int pid = ld_relaxed_gpu(pt + (ts >> p.log2_page));
    if (pid < 0 || pid >= p.num_pages) continue;
#pragma unroll
    for (int bx = 0; bx < C::N_BOX; ++bx) {
      tma_prefetch_4d(tmk, bx * C::BOX_ELEMS, h, ts & (P - 1), pid);
      tma_prefetch_4d(tmv, bx * C::BOX_ELEMS, h, ts & (P - 1), pid);
    }
  }
  return L;
}

template <int KIND, int D, bool FUSED, bool DEEP, bool NARROW>
__global__ void __launch_bounds__(S1Cfg<KIND, D, DEEP, NARROW>::THREADS, S1Cfg<KIND, D, DEEP, NARROW>::MIN_BLOCKS)
    fd_stage1_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                     const __grid_constant__ Stage1Params p) {
  using C = S1Cfg<KIND, D, DEEP, NARROW>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *empty = full + C::STAGES;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // Which (request b, split s of its S_req, KV head h, row tile rt) this CTA
  // computes. Balanced policy: unit u of the batch, located after the wait.
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
  // The pipeline barriers read no input: set them up before the wait below.
  if (threadIdx.x == 0) {
    for (int i = 0; i < C::STAGES; ++i) {
      mbar_init(&full[i], C::QUANT ? 1 + 32 : 1);
      mbar_init(&empty[i], C::NUM_CW);
    }
    fence_mbar_init();
  }
  if constexpr (C::QUANT) {
    // The scale slots start at zero. The producer fills only the slots of
    // keys before the split end, so a slot past it holds zero or a scale of
    // an earlier block of this split: always a finite value (for finite
    // inputs), which meets a zero probability without a selection.
    constexpr int N16 = 2 * C::SC / 16;
    for (int i = threadIdx.x; i < C::STAGES * N16; i += C::THREADS)
      *reinterpret_cast<uint4 *>(smem + (i / N16) * C::STAGE + 2 * C::TILE + (i % N16) * 16) =
          make_uint4(0u, 0u, 0u, 0u);
  }
  __syncthreads();

  // Launched as a programmatic dependent of the previous kernel in the stream:
  // everything that kernel wrote is visible after this wait, before any input
  // is read for its value. The one-wave variant's CTAs are often resident
  // while that kernel drains; they spend the wait pulling their first blocks
  // into L2 (from values that only steer prefetches).
  int hint_L = -1;  // deep producer warp: the length its prefetch used
  int hint_b = b, hint_s = s, hint_S = S_req;
  if constexpr (DEEP) {
    if (warp == C::NUM_CW) {
      if (p.balanced) {
        const SplitUnit su = locate_balanced<true>(p.seqlens, p.sl_s, p.batch, cap, p.log2_page, p.num_splits,
                                                   p.s_cap, p.chunk_min, u, lane);
        hint_b = su.b;
        hint_s = su.s;
        hint_S = su.sb;
      }
      if (hint_b >= 0) hint_L = prefetch_first_blocks<C>(&tmk, &tmv, p, hint_b, h, hint_s, hint_S, lane);
    }
  }
  griddep_wait();
  // Every trigger of this kernel comes after its wait: the merge kernel relies
  // on that to read the lengths before its own wait.
  // The one-wave grid lets the merge kernel be scheduled from here on (every
  // CTA of this grid is resident by then), so it is waiting, not launching,
  // when this grid completes; it reads the workspace only after that. The
  // multi-wave variants trigger as they finish: an early merge grid would sit
  // on the resources their last wave uses.
  if constexpr (DEEP) griddep_launch_dependents();

  // The deep producer loads its first page ids now, at the hinted split range,
  // in the same round trip as the lengths; they are used only if the length
  // read after the wait equals the hint (then the range is the same).
  int pn0 = 0, pn1 = 0;
  if constexpr (DEEP) {
    if (warp == C::NUM_CW && hint_L > 0) {
      const int hc = split_chunk(hint_L, hint_S, p.log2_page, p.chunk_min);
      const int h0 = hint_s * hc, h1 = min(hint_L, h0 + hc);
      if (h0 < h1) {
        const int *pt = p.page_table + hint_b * p.pt_sb;
        const int first = h0 >> p.log2_page;
        const int np = ((min(h0 + C::BLOCK_N, h1) - 1) >> p.log2_page) - first + 1;
        pn0 = lane < np ? ld_cg(pt + first + lane) : 0;
        pn1 = lane + 32 < np ? ld_cg(pt + first + 32 + lane) : 0;
      }
    }
  }

  int L_bal = 0;  // balanced: the located request's stored length
  if (p.balanced) {  // every warp locates the unit (same loads, same answer)
    const SplitUnit su = locate_balanced<false>(p.seqlens, p.sl_s, p.batch, cap, p.log2_page, p.num_splits,
                                                p.s_cap, p.chunk_min, u, lane);
    if (su.b < 0) {  // past the batch's last split
      if constexpr (!DEEP) griddep_launch_dependents();
      return;
    }
    b = su.b;
    s = su.s;
    S_req = su.sb;
    L_bal = su.L;
  }

  // Consumers issue their query-tile loads now, so their latency overlaps the
  // length load below (the tile is written to shared memory later).
  constexpr int Q_JOBS = 16 * (D / 8);  // 16-byte pieces of the 16-row Q tile
  constexpr int Q_PER = (Q_JOBS + C::NUM_CW * 32 - 1) / (C::NUM_CW * 32);
  uint4 qv[Q_PER];
  if (warp < C::NUM_CW) {
#pragma unroll
    for (int k = 0; k < Q_PER; ++k) {
      const int i = threadIdx.x + k * C::NUM_CW * 32;
      qv[k] = make_uint4(0u, 0u, 0u, 0u);
      const int r = i / (D / 8), cc = i % (D / 8);
      const int rg = rt * 16 + r;
      if (i < Q_JOBS && rg < p.R) {
        const int t = rg / p.G, gq = rg - t * p.G;
        qv[k] = *reinterpret_cast<const uint4 *>(p.q + b * p.q_sb + t * p.q_st + (h * p.G + gq) * p.q_sh +
                                                 cc * 8);
      }
    }
  }
  const int P = p.page_size;

  // ---- split range from cache_seqlens (on the device; no host metadata)
  // (the balanced map read it already; the deep variant read these words
  // before the wait: take them from L2)
  int L = p.balanced ? L_bal : (DEEP ? ld_cg(p.seqlens + b * p.sl_s) : p.seqlens[b * p.sl_s]);
  if (L < 0 || L > cap) {
    if (threadIdx.x == 0) atomicOr(p.status, FD_DEVSTAT_SEQLEN_OVERFLOW);
    L = L < 0 ? 0 : cap;
  }
  const int chunk = split_chunk(L, S_req, p.log2_page, p.chunk_min);
  const int c0 = s * chunk;
  const int c1 = min(L, c0 + chunk);
  // A request with a single non-empty split gets its final outputs from this
  // CTA; the merge skips it.
  const bool direct = FUSED || split_count(L, S_req, p.log2_page, p.chunk_min) == 1;

  if (c0 >= c1) {
    // An empty split of a split call writes nothing: the merge reads only the
    // split_count() non-empty splits. A request with no keys in an unsplit
    // call gets out = 0, lse = -inf here.
    // With the fused merge, a request with no keys has no split to merge
    // it: its split-0 CTA writes the empty rows (out = 0, lse = -inf).
    if (!FUSED && !(p.counters && L == 0 && s == 0)) {
      if constexpr (!DEEP) griddep_launch_dependents();
      return;
    }
    const int ntile_rows = min(16, p.R - rt * 16);
    for (int i = threadIdx.x; i < ntile_rows * (D / 8); i += C::THREADS) {
      const int r = i / (D / 8), d0 = (i % (D / 8)) * 8;
      const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      write_row_outputs<C>(p, true, b, h, s, rt * 16 + r, d0, z, 8, -INFINITY, d0 == 0);
    }
    if constexpr (!DEEP) griddep_launch_dependents();
    return;
  }

  const int n_iters = (c1 - c0 + C::BLOCK_N - 1) / C::BLOCK_N;

  if (warp == C::NUM_CW) {
    // ======================= producer warp =======================
    if (lane == 0) {
      tma_prefetch_desc(&tmk);
      tma_prefetch_desc(&tmv);
    }
    const uint64_t pol = l2_policy_evict_first();
    const int *pt = p.page_table + b * p.pt_sb;
    const int SEG = P < C::SEG_MAX ? P : C::SEG_MAX;  // slots per TMA box (within one page)
    const int log2_seg = P < C::SEG_MAX ? p.log2_page : 6;
    const unsigned seg_bytes = static_cast<unsigned>(SEG * C::ROW_BYTES);

    auto load_pids = [&](int it, int &q0, int &q1) {
      const int tok0 = c0 + it * C::BLOCK_N;
      const int first = tok0 >> p.log2_page;
      const int np = ((min(tok0 + C::BLOCK_N, c1) - 1) >> p.log2_page) - first + 1;
      q0 = lane < np ? (DEEP ? ld_cg(pt + first + lane) : pt[first + lane]) : 0;
      q1 = lane + 32 < np ? (DEEP ? ld_cg(pt + first + 32 + lane) : pt[first + 32 + lane]) : 0;
    };
    if (!DEEP || L != hint_L || b != hint_b || s != hint_s || S_req != hint_S) load_pids(0, pn0, pn1);
    int issued = 0;
    for (int it = 0; it < n_iters; ++it) {
      int p0 = pn0, p1 = pn1;
      if (it + 1 < n_iters) load_pids(it + 1, pn0, pn1);
      const int tok0 = c0 + it * C::BLOCK_N;
      const int tend = min(tok0 + C::BLOCK_N, c1);
      const int first = tok0 >> p.log2_page;
      const int np = ((tend - 1) >> p.log2_page) - first + 1;
      // page ids outside the pool: record and redirect past the end (TMA zero-fills)
      const bool bad0 = lane < np && (p0 < 0 || p0 >= p.num_pages);
      const bool bad1 = lane + 32 < np && (p1 < 0 || p1 >= p.num_pages);
      if (__any_sync(0xffffffffu, bad0 || bad1) && lane == 0) atomicOr(p.status, FD_DEVSTAT_BAD_PAGE);
      if (bad0) p0 = p.num_pages;
      if (bad1) p1 = p.num_pages;
      const int stage = it % C::STAGES;
      const unsigned ph = (it / C::STAGES) & 1;
      if (!mbar_wait_warp(&empty[stage], ph ^ 1, p.status)) break;
      uint8_t *kt = smem + stage * C::STAGE;
      uint8_t *vt = kt + C::TILE;
      // segments of SEG slots starting at token tok0 + i * SEG, each inside one page
      const int nseg = (tend - tok0 + SEG - 1) >> log2_seg;
      if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<unsigned>(nseg) * seg_bytes * 2u);
      {  // lane i issues segment i (a stage holds at most BLOCK_N / 8 <= 16 segments)
        const int i = lane;
        const int ts = tok0 + (min(i, nseg - 1) << log2_seg);
        const int pi = (ts >> p.log2_page) - first;
        const int a0 = __shfl_sync(0xffffffffu, p0, pi & 31);
        const int a1 = __shfl_sync(0xffffffffu, p1, pi & 31);
        if (i < nseg) {
          const int pid = pi < 32 ? a0 : a1;
          const int slot0 = ts & (P - 1);
          const int row0 = i << log2_seg;
#pragma unroll
          for (int bx = 0; bx < C::N_BOX; ++bx) {
            const int off = bx * C::BLOCK_N * C::BOX_BYTES + row0 * C::BOX_BYTES;
            tma_load_4d(kt + off, &tmk, bx * C::BOX_ELEMS, h, slot0, pid, &full[stage], pol);
            tma_load_4d(vt + off, &tmv, bx * C::BOX_ELEMS, h, slot0, pid, &full[stage], pol);
          }
        }
      }
      if constexpr (C::QUANT) {
        float *ksc = reinterpret_cast<float *>(vt + C::TILE);
        float *vsc = ksc + C::BLOCK_N * C::NG;
#pragma unroll
        for (int i = lane; i < C::BLOCK_N; i += 32) {
          const int tok = tok0 + i;
          const int pi = (tok >> p.log2_page) - first;
          const int a0 = __shfl_sync(0xffffffffu, p0, pi & 31);
          const int a1 = __shfl_sync(0xffffffffu, p1, pi & 31);
          const int pid = pi < 32 ? a0 : a1;
          if (tok < tend) {
            // a page id outside the pool (reported above; its codes read as
            // 0) takes page 0's scales, so the result stays finite
            const int ps = pid < p.num_pages ? pid : 0;
            const float *src = p.kv_scales + static_cast<int64_t>(ps) * p.sc_sp +
                               static_cast<int64_t>(tok & (P - 1)) * p.sc_ss +
                               static_cast<int64_t>(h) * p.sc_sh;
            cp_async_ca<C::NG * 4>(ksc + i * C::NG, src);
            cp_async_ca<C::NG * 4>(vsc + i * C::NG, src + p.sc_sk);
          }
        }
        cp_async_mbar_arrive_noinc(&full[stage]);
      }
      issued = it + 1;
    }
    // drain: the most recent phase of every stage this warp filled has landed
    if (lane == 0) {
      for (int k = issued > C::STAGES ? issued - C::STAGES : 0; k < issued; ++k)
        mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1, p.status);
    }
  } else {
    // ======================= consumer warps =======================
    const int g = lane >> 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_TMEM);
    if constexpr (C::O_TMEM) {
      if (warp == 0) tmem_alloc(tmem_slot, C::TMEM_COLS);
      tc_fence_before();  // the address is read after the barrier below
    }
    // Q tile (16 rows; rows past R are zero) -> shared -> A fragments
    uint8_t *qs = smem + C::OFF_Q;
#pragma unroll
    for (int k = 0; k < Q_PER; ++k) {
      const int i = threadIdx.x + k * C::NUM_CW * 32;
      if (i < Q_JOBS) *reinterpret_cast<uint4 *>(qs + (i / (D / 8)) * C::QROW + (i % (D / 8)) * 16) = qv[k];
    }
    if (threadIdx.x == 0)
      *reinterpret_cast<int4 *>(smem + C::OFF_META) = make_int4(b, s, L, S_req | (direct ? 1 << 16 : 0));
    named_barrier(1, C::NUM_CW * 32);
    if constexpr (C::O_TMEM) tc_fence_after();
    uint32_t qa[D / 16][4];
    uint32_t qb[D / 16][2];  // narrow: the row-g Q fragments as B operands
    // the thread's two query rows: g and g + 8, or (narrow) 2c and 2c + 1
    const int qrow0 = NARROW ? 2 * (lane & 3) : g, qrow_step = NARROW ? 1 : 8;
    float qc[2][C::NG], rs[2];
    if constexpr (C::QUANT) {
      float *qinfo = reinterpret_cast<float *>(smem + C::OFF_QI);
      if (threadIdx.x < 128) prepare_q_rows<C, KIND>(qs, qinfo, threadIdx.x);  // 8 threads per row
      named_barrier(1, C::NUM_CW * 32);
      build_q_fragments<C, KIND>(qs, qinfo, qa, lane);
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        qb[ks][0] = qa[ks][0];
        qb[ks][1] = qa[ks][2];
      }
      if constexpr (C::QB_SMEM) {
        if (warp == 0) {
          uint2 *qb_s = reinterpret_cast<uint2 *>(smem + C::OFF_QA);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks) qb_s[ks * 32 + lane] = make_uint2(qb[ks][0], qb[ks][1]);
        }
        named_barrier(1, C::NUM_CW * 32);
      }
      if constexpr (C::QA_SMEM) {
        if (warp == 0) {
          uint4 *qa_s = reinterpret_cast<uint4 *>(smem + C::OFF_QA);
#pragma unroll
          for (int ks = 0; ks < D / 16; ++ks)
            qa_s[ks * 32 + lane] = make_uint4(qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3]);
        }
        named_barrier(1, C::NUM_CW * 32);
      }
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int qr = qrow0 + qrow_step * hr;
        rs[hr] = qinfo[qr] * p.scale_log2;
#pragma unroll
        for (int gi = 0; gi < C::NG; ++gi) qc[hr][gi] = qinfo[16 + qr * C::NG + gi];
      }
    } else {
      const int mi = lane >> 3, ri = lane & 7;
      const int row = ((mi & 1) << 3) + ri;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int col = ks * 16 + ((mi >> 1) << 3);
        ldsm_x4(qa[ks], smem_u32(qs + row * C::QROW + col * 2));
      }
    }
    // causal limits of this thread's two rows
    int lim[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      const int rg = rt * 16 + qrow0 + qrow_step * k;
      if (rg < p.R) {
        const int t = rg / p.G;
        lim[k] = min(c1, L - (p.Tq - 1) + t);
      } else {
        lim[k] = c1;
      }
    }

    float o[C::OT][4];
    float ra[C::NR][4];  // quantised V: the bias row sums (registers unless O is in tensor memory)
#pragma unroll
    for (int j = 0; j < C::OT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
#pragma unroll
    for (int j = 0; j < C::NR; ++j) ra[j][0] = ra[j][1] = ra[j][2] = ra[j][3] = 0.f;
    // warp w's threads own TMEM lanes 32w .. 32w + 31
    const uint32_t tm_o = C::O_TMEM ? *tmem_slot + ((static_cast<uint32_t>(warp) * 32u) << 16) : 0u;
    if constexpr (C::O_TMEM) {
#pragma unroll
      for (int i = 0; i < D / 64; ++i) tmem_st32(tm_o + 32 * i, &o[8 * i][0]);
    }
    float m[2] = {-INFINITY, -INFINITY};
    float l[2] = {0.f, 0.f};
    const int row0 = warp * C::KPW;  // the warp's first key in each stage

    for (int it = 0; it < n_iters; ++it) {
      const int stage = it % C::STAGES;
      const unsigned ph = (it / C::STAGES) & 1;
      if (!mbar_wait_warp(&full[stage], ph, p.status)) break;
      const int tok0 = c0 + it * C::BLOCK_N;
      const int tok_row0 = tok0 + row0;
      uint8_t *kt = smem + stage * C::STAGE;
      uint8_t *vt = kt + C::TILE;
      if (tok_row0 < c1) {
        if constexpr (C::QUANT) {
          const float *ksc = reinterpret_cast<const float *>(vt + C::TILE);
          const float *vsc = ksc + C::BLOCK_N * C::NG;
          if constexpr (NARROW) {
            static_assert(C::QB_SMEM, "the narrow block reloads its Q fragments from shared memory");
            uint32_t qr[D / 16][2];
            const uint2 *qb_s = reinterpret_cast<const uint2 *>(smem + C::OFF_QA);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks) {
              const uint2 v = qb_s[ks * 32 + lane];
              qr[ks][0] = v.x;
              qr[ks][1] = v.y;
            }
            warp_block_km<C, KIND>(kt, vt, ksc, vsc, row0, qr, qc, rs, o, ra, m, l, tok_row0, c1, lim[0],
                                   lim[1], lane);
          } else {
            static_assert(C::QA_SMEM, "the 16-row quantised block reads its Q fragments from shared memory");
            uint32_t qf[D / 16][4];  // int8: loaded here; int4 loads them group by group
            const uint4 *qa_s = reinterpret_cast<const uint4 *>(smem + C::OFF_QA);
            if constexpr (KIND != KV_I4) {
#pragma unroll
              for (int ks = 0; ks < D / 16; ++ks) {
                const uint4 v = qa_s[ks * 32 + lane];
                qf[ks][0] = v.x;
                qf[ks][1] = v.y;
                qf[ks][2] = v.z;
                qf[ks][3] = v.w;
              }
            }
            warp_block_q<C, KIND>(kt, vt, ksc, vsc, row0, qf, qa_s, qc,
                                  reinterpret_cast<const float *>(smem + C::OFF_QI) + 16 + (lane >> 2) * C::NG, rs,
                                  o, ra, tm_o, m, l, tok_row0, c1, lim[0], lim[1], lane);
          }
        } else {
          if (tok_row0 + 16 > c1) {  // zero V rows past the split end before PV
            constexpr int CH = C::N_BOX * (C::BOX_BYTES / 16);
            for (int job = lane; job < 16 * CH; job += 32) {
              const int r = job / CH, k = job % CH;
              if (tok_row0 + r >= c1) {
                const int bx = k / (C::BOX_BYTES / 16), cc = k % (C::BOX_BYTES / 16);
                *reinterpret_cast<uint4 *>(vt + bx * C::BLOCK_N * C::BOX_BYTES +
                                           swz<C::BOX_BYTES>((row0 + r) * C::BOX_BYTES + cc * 16)) =
                    make_uint4(0u, 0u, 0u, 0u);
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
          }
          warp_block<C>(smem_u32(kt), smem_u32(vt), C::BLOCK_N * 128, row0, qa, o, m, l, tok_row0,
                        lim[0], lim[1], p.scale_log2, lane);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
    }

    if constexpr (C::O_TMEM) {  // O back from tensor memory; the columns are freed below
      tmem_wait_st();
#pragma unroll
      for (int i = 0; i < D / 64; ++i) tmem_ld32(tm_o + 32 * i, &o[8 * i][0]);
      tmem_wait_ld();
      tc_fence_before();
    }
    if constexpr (C::V_SUB) remove_v_bias<C>(o, ra);

    // ---- merge the consumer warps' (max, sum, O) through shared memory
    // (a row's partial sums sit in the 4 lanes of a quad, or, narrow, in the
    // 8 lanes of one c)
#pragma unroll
    for (int x = NARROW ? 4 : 1; x < (NARROW ? 32 : 4); x <<= 1) {
      l[0] += __shfl_xor_sync(0xffffffffu, l[0], x);
      l[1] += __shfl_xor_sync(0xffffffffu, l[1], x);
    }
    named_barrier(1, C::NUM_CW * 32);  // every consumer is done with the ring
    if constexpr (C::O_TMEM) {
      if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, C::TMEM_COLS);
      }
    }
    const int4 meta = *reinterpret_cast<const int4 *>(smem + C::OFF_META);  // after the barrier above
    const int b_e = meta.x, s_e = meta.y, L_e = meta.z, S_e = meta.w & 0xffff;
    const bool direct_e = (meta.w >> 16) != 0;
    const int h_e = p.balanced ? (blockIdx.x / p.row_tiles) % p.Hkv : blockIdx.y;
    float *co = reinterpret_cast<float *>(smem);
    float *cm = reinterpret_cast<float *>(smem + C::CMB_O);
    float *cl = cm + C::NUM_CW * C::TR;
    if constexpr (NARROW) {
      // rows 2c, 2c + 1: o[j] = (channel ch: rows 2c, 2c+1), (ch + 1: rows 2c, 2c+1), ch below
      const int c = lane & 3;
      float *w0 = co + (warp * C::TR + 2 * c) * C::CROW;
      float *w1 = w0 + C::CROW;
#pragma unroll
      for (int j = 0; j < C::OT; ++j) {
        // m-tile j: channel pair (row g, row g + 8) of the m-tile (see warp_block_km)
        const int ch = KIND == KV_I8 ? 16 * j + 2 * g : 32 * (j / 2) + 4 * g + 2 * (j % 2);
        *reinterpret_cast<float2 *>(w0 + ch) = make_float2(o[j][0], o[j][2]);
        *reinterpret_cast<float2 *>(w1 + ch) = make_float2(o[j][1], o[j][3]);
      }
      if (g == 0) {
        cm[warp * C::TR + 2 * c] = m[0];
        cm[warp * C::TR + 2 * c + 1] = m[1];
        cl[warp * C::TR + 2 * c] = l[0];
        cl[warp * C::TR + 2 * c + 1] = l[1];
      }
    } else {
      const int c = lane & 3;
      float *w0 = co + (warp * 16 + g) * C::CROW;
      float *w1 = co + (warp * 16 + g + 8) * C::CROW;
      // rows g and g + 8 of the tile; the second half only if it holds queries
      auto put_rows = [&](float *w, int e) {
#pragma unroll
        for (int j = 0; j < D / 8; ++j) {
          if constexpr (KIND == KV_I4) {  // n-tile j = 4 gi + q, column n holds channel 32 gi + 4 n + q
            const int ch = 32 * (j / 4) + 8 * c + (j % 4);
            w[ch] = o[j][e];
            w[ch + 4] = o[j][e + 1];
          } else if constexpr (C::QUANT) {  // int8: n-tile j = 2 s + e, column n holds channel 16 s + 2 n + e
            const int ch = 16 * (j / 2) + 4 * c + (j % 2);
            w[ch] = o[j][e];
            w[ch + 2] = o[j][e + 1];
          } else {
            *reinterpret_cast<float2 *>(w + j * 8 + 2 * c) = make_float2(o[j][e], o[j][e + 1]);
          }
        }
      };
      put_rows(w0, 0);
      if (rt * 16 + 8 < p.R) put_rows(w1, 2);
      if (c == 0) {
        cm[warp * 16 + g] = m[0];
        cm[warp * 16 + g + 8] = m[1];
        cl[warp * 16 + g] = l[0];
        cl[warp * 16 + g + 8] = l[1];
      }
    }
    named_barrier(1, C::NUM_CW * 32);
    // Lane r of every consumer warp forms row r's weights (lanes past the
    // tile's rows repeat them); then each warp combines whole rows, lane l
    // taking the column pairs 2l + 64k, so every read of a partial row is 256
    // consecutive bytes (conflict-free) and every store coalesced. (Unrolling
    // a warp's rows measured the same for bf16 and cost the quantised
    // kernels registers in their main loop.)
    static_assert(C::TR % C::NUM_CW == 0, "rows per consumer warp");
    float wl[C::NUM_CW], inv_l, lse_l;
    {
      const int rr = lane % C::TR;
      float mw[C::NUM_CW];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < C::NUM_CW; ++w) {
        mw[w] = cm[w * C::TR + rr];
        M = fmaxf(M, mw[w]);
      }
      float Lsum = 0.f;
#pragma unroll
      for (int w = 0; w < C::NUM_CW; ++w) {
        wl[w] = mw[w] == -INFINITY ? 0.f : fast_exp2(mw[w] - M);
        Lsum = fmaf(wl[w], cl[w * C::TR + rr], Lsum);
      }
      inv_l = Lsum > 0.f ? 1.f / Lsum : 0.f;
      lse_l = Lsum > 0.f ? (M + log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
    }
    auto combine_row = [&](int i) {
      const int row = warp + i * C::NUM_CW;
      const int rg = rt * 16 + row;
      if (rg >= p.R) return;  // a padding row of the tile (its partials were not written)
      float wt[C::NUM_CW];
#pragma unroll
      for (int w = 0; w < C::NUM_CW; ++w) wt[w] = __shfl_sync(0xffffffffu, wl[w], row);
      const float inv = __shfl_sync(0xffffffffu, inv_l, row);
      const float lse_nat = __shfl_sync(0xffffffffu, lse_l, row);
      float2 vals[D / 64];
#pragma unroll
      for (int k = 0; k < D / 64; ++k) {
        float2 a = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < C::NUM_CW; ++w) {
          const float2 v = *reinterpret_cast<const float2 *>(co + (w * C::TR + row) * C::CROW + 2 * lane + 64 * k);
          a.x = fmaf(wt[w], v.x, a.x);
          a.y = fmaf(wt[w], v.y, a.y);
        }
        vals[k] = make_float2(a.x * inv, a.y * inv);
      }
      write_row_pairs<C>(p, direct_e, b_e, h_e, s_e, rg, lane, vals, lse_nat);
    };
#pragma unroll 1
    for (int i = 0; i < C::TR / C::NUM_CW; ++i) combine_row(i);
    if constexpr (!FUSED) {
      if (p.counters && !direct_e) {
        // Fused merge: publish this split's partials, count it, and let the
        // last split of the (request, KV head, row tile) merge them all.
        volatile unsigned *flag = reinterpret_cast<volatile unsigned *>(smem + C::OFF_FLAG);
        __threadfence();
        named_barrier(1, C::NUM_CW * 32);
        const int nv = split_count(L_e, S_e, p.log2_page, p.chunk_min);
        if (threadIdx.x == 0) {
          unsigned *ctr = p.counters + (static_cast<int64_t>(b_e) * p.Hkv + h_e) * p.row_tiles + rt;
          const unsigned done = atomicAdd(ctr, 1u) + 1u;
          const bool last = done == static_cast<unsigned>(nv);
          if (last) {
            *ctr = 0u;  // ready for the next call (and graph replay)
            __threadfence();
          }
          *flag = last ? 1u : 0u;
        }
        named_barrier(1, C::NUM_CW * 32);
        if (*flag) merge_tile<C>(p, b_e, h_e, rt, nv, warp, C::NUM_CW, lane);
      }
    }
  }
  if constexpr (!DEEP) griddep_launch_dependents();
}

template <int KIND, int D, bool FUSED, bool DEEP, bool NARROW>
cudaError_t set_smem_limit() {
  return cudaFuncSetAttribute(fd_stage1_kernel<KIND, D, FUSED, DEEP, NARROW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, S1Cfg<KIND, D, DEEP, NARROW>::SMEM_ALLOC);
}

template <int KIND, int D>
cudaError_t stage1_prepare_t() {
  cudaError_t e = set_smem_limit<KIND, D, false, false, false>();
  if (e == cudaSuccess) e = set_smem_limit<KIND, D, true, false, false>();
  if constexpr (KIND == KV_BF16) {
    if (e == cudaSuccess) e = set_smem_limit<KIND, D, false, true, false>();
    if (e == cudaSuccess) e = set_smem_limit<KIND, D, true, true, false>();
  } else {
    if (e == cudaSuccess) e = set_smem_limit<KIND, D, false, false, true>();
    if (e == cudaSuccess) e = set_smem_limit<KIND, D, true, false, true>();
  }
  return e;
}

// Stage 1 is launched with programmatic stream serialization: its CTAs may be
// scheduled while the previous kernel drains (a previous kernel that never
// triggers simply completes first), and griddepcontrol.wait at its start
// orders it after that kernel's memory operations.
template <int KIND, int D, bool DEEP, bool NARROW>
cudaError_t launch_variant(bool fused, const CUtensorMap &tmk, const CUtensorMap &tmv,
                           const Stage1Params &p, dim3 grid, cudaStream_t stream) {
  using C = S1Cfg<KIND, D, DEEP, NARROW>;
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
  if (fused) return cudaLaunchKernelEx(&cfg, fd_stage1_kernel<KIND, D, true, DEEP, NARROW>, tmk, tmv, p);
  return cudaLaunchKernelEx(&cfg, fd_stage1_kernel<KIND, D, false, DEEP, NARROW>, tmk, tmv, p);
}

// deep: one-wave grids of the bf16 cache use the deep-ring variant.
// Quantised caches with at most 8 query rows per KV head use the narrow one.
template <int KIND, int D>
cudaError_t launch_stage1_t(bool fused, bool deep, const CUtensorMap &tmk, const CUtensorMap &tmv,
                            const Stage1Params &p, dim3 grid, cudaStream_t stream) {
  if constexpr (KIND == KV_BF16) {
    if (deep) return launch_variant<KIND, D, true, false>(fused, tmk, tmv, p, grid, stream);
  } else {
    if (p.R <= 8) return launch_variant<KIND, D, false, true>(fused, tmk, tmv, p, grid, stream);
  }
  return launch_variant<KIND, D, false, false>(fused, tmk, tmv, p, grid, stream);
}

}  // namespace fd
