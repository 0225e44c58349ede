// fd_api.cu - the C ABI of libfd: plans, descriptor validation and launch.
//
// Everything here runs on the host. A decode call validates its descriptors
// in O(1) without touching device memory, encodes the two TMA descriptors of
// the K and V caches, and enqueues stage 1 (and stage 2 when num_splits > 1)
// on the caller's stream. It never synchronises or allocates, so it can be
// captured in a CUDA graph (sglang PR 29843 summary, sections "motivation" and
// "implementation": graph-replayed attention metadata must come from
// cache_seqlens / page_table on the device, with no .item()).
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "fd.h"
#include "kernels.h"
#include "plan.h"

namespace {

thread_local char g_err[512] = "";
thread_local fd_plan *g_plan = nullptr;

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int ilog2_exact(int v) {
  if (v <= 0 || (v & (v - 1))) return -1;
  int r = 0;
  while ((1 << r) < v) ++r;
  return r;
}

int elem_bytes(int dtype) {
  switch (dtype) {
    case FD_BF16: return 2;
    case FD_FP32: return 4;
    case FD_INT8: return 1;
    case FD_INT4X2: return 1;
    case FD_INT32: return 4;
    case FD_INT64: return 8;
  }
  return 0;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace

namespace fd {

fd_status fail(fd_status s, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

}  // namespace fd

using fd::fail;

#define FD_CUDA_TRY(call)                                                                 \
  do {                                                                                    \
    cudaError_t e_ = (call);                                                              \
    if (e_ != cudaSuccess)                                                                \
      return fail(FD_ERR_CUDA, "%s failed: %s (%d)", #call, cudaGetErrorString(e_), (int)e_); \
  } while (0)

extern "C" {

const char *fd_status_string(fd_status s) {
  switch (s) {
    case FD_OK: return "FD_OK";
    case FD_ERR_INVALID_ARG: return "FD_ERR_INVALID_ARG";
    case FD_ERR_UNSUPPORTED: return "FD_ERR_UNSUPPORTED";
    case FD_ERR_WORKSPACE: return "FD_ERR_WORKSPACE";
    case FD_ERR_CAPTURING: return "FD_ERR_CAPTURING";
    case FD_ERR_CUDA: return "FD_ERR_CUDA";
    case FD_ERR_DEVICE_STATUS: return "FD_ERR_DEVICE_STATUS";
    case FD_ERR_TIMEOUT: return "FD_ERR_TIMEOUT";
    case FD_ERR_NO_PLAN: return "FD_ERR_NO_PLAN";
    case FD_ERR_IO: return "FD_ERR_IO";
  }
  return "FD_ERR_UNKNOWN";
}

const char *fd_last_error(void) { return g_err; }

fd_status fd_plan_create(int device, int max_batch, int max_q_per_req, int num_q_heads,
                         int num_kv_heads, int head_dim, int page_size, fd_dtype kv_dtype,
                         int max_splits, float softmax_scale, fd_plan **plan) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan out-pointer is NULL");
  *plan = nullptr;
  if (max_batch < 1 || max_batch > 65535)
    return fail(FD_ERR_INVALID_ARG, "max_batch %d not in [1, 65535]", max_batch);
  if (max_q_per_req < 1 || max_q_per_req > 64)
    return fail(FD_ERR_INVALID_ARG, "max_q_per_req %d not in [1, 64]", max_q_per_req);
  if (num_q_heads < 1 || num_kv_heads < 1 || num_kv_heads > 65535 || num_q_heads % num_kv_heads)
    return fail(FD_ERR_INVALID_ARG, "heads: Hq=%d must be a positive multiple of Hkv=%d", num_q_heads,
                num_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(FD_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", head_dim);
  // A page's rows land in shared memory as whole TMA swizzle atoms (8 rows).
  const int lp = ilog2_exact(page_size);
  if (lp < 3 || page_size > 256)
    return fail(FD_ERR_UNSUPPORTED, "page_size %d must be a power of two in [8, 256]", page_size);
  int kind;
  switch (kv_dtype) {
    case FD_BF16: kind = fd::KV_BF16; break;
    case FD_INT8: kind = fd::KV_I8; break;
    case FD_INT4X2: kind = fd::KV_I4; break;
    default: return fail(FD_ERR_UNSUPPORTED, "kv_dtype %d not supported", (int)kv_dtype);
  }
  if (max_splits < 1 || max_splits > 64)
    return fail(FD_ERR_INVALID_ARG, "max_splits %d not in [1, 64]", max_splits);
  if (!(softmax_scale >= 0.f) || std::isinf(softmax_scale))
    return fail(FD_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");

  fd_plan *pl = new fd_plan();
  pl->device = device;
  pl->max_batch = max_batch;
  pl->max_q = max_q_per_req;
  pl->hq = num_q_heads;
  pl->hkv = num_kv_heads;
  pl->d = head_dim;
  pl->page = page_size;
  pl->log2_page = lp;
  pl->kv_dtype = kv_dtype;
  pl->kind = kind;
  pl->max_splits = max_splits;
  pl->scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
  if (const char *dir = std::getenv("FD_AUTOTUNE_CACHE_DIR")) pl->cache_dir = dir;
  // Split merge: the stage-2 kernel (default) or, with FD_MERGE=fused, the
  // last split CTA of each tile (measured slower on GB300: the tail merge
  // lengthens the critical path more than the second launch costs).
  const char *mg = std::getenv("FD_MERGE");
  pl->merge_kernel = !(mg && std::strcmp(mg, "fused") == 0);
  // Quantised caches run stage 1 on the register (mma.sync) kernel;
  // FD_QUANT_KERNEL=tc selects the tcgen05 kernel for head_dim 128 (measured
  // slower on GB300: its code conversions run on two warps per scheduler).
  const char *qk = std::getenv("FD_QUANT_KERNEL");
  pl->quant_tc = qk && std::strcmp(qk, "tc") == 0;

  if (device >= 0) {
    fd::DeviceGuard guard(device);
    cudaError_t e = guard.ok ? cudaSuccess : cudaErrorInvalidDevice;
    cudaDeviceProp prop;
    if (e == cudaSuccess) e = cudaGetDeviceProperties(&prop, device);
    if (e == cudaSuccess) {
      pl->num_sms = prop.multiProcessorCount;
      pl->gpu_name = prop.name;
      if (prop.major * 10 + prop.minor < 100) e = cudaErrorInvalidDevice;
    }
    pl->ws_rows = static_cast<size_t>(max_batch) * max_q_per_req * num_q_heads * max_splits;
    if (e == cudaSuccess && max_splits > 1)
      e = cudaMalloc(&pl->o_part, pl->ws_rows * head_dim * sizeof(float));
    if (e == cudaSuccess && max_splits > 1) e = cudaMalloc(&pl->lse_part, pl->ws_rows * sizeof(float));
    if (e == cudaSuccess) e = cudaMalloc(&pl->status, sizeof(unsigned));
    if (e == cudaSuccess) e = cudaMemset(pl->status, 0, sizeof(unsigned));
    pl->n_counters = static_cast<size_t>(max_batch) * num_kv_heads *
                     ((num_q_heads / num_kv_heads * max_q_per_req + 15) / 16);
    if (e == cudaSuccess && max_splits > 1) e = cudaMalloc(&pl->counters, pl->n_counters * sizeof(unsigned));
    if (e == cudaSuccess && max_splits > 1) e = cudaMemset(pl->counters, 0, pl->n_counters * sizeof(unsigned));
    if (e == cudaSuccess) e = fd::stage1_prepare(kind, head_dim);
    if (e == cudaSuccess && !encode_fn()) e = cudaErrorSymbolNotFound;
    if (e != cudaSuccess) {
      fd_plan_destroy(pl);
      return fail(FD_ERR_CUDA, "plan setup on device %d failed: %s (%d)", device,
                  cudaGetErrorString(e), (int)e);
    }
  }
  fd::autotune_load(pl);  // a missing or unreadable cache only means no tuned entries yet
  *plan = pl;
  return FD_OK;
}

fd_status fd_plan_destroy(fd_plan *plan) {
  if (!plan) return FD_OK;
  if (g_plan == plan) g_plan = nullptr;
  if (plan->device >= 0) {
    fd::DeviceGuard guard(plan->device);
    if (plan->o_part) cudaFree(plan->o_part);
    if (plan->lse_part) cudaFree(plan->lse_part);
    if (plan->status) cudaFree(plan->status);
    if (plan->counters) cudaFree(plan->counters);
  }
  delete plan;
  return FD_OK;
}

fd_status fd_set_plan(fd_plan *plan) {
  g_plan = plan;
  return FD_OK;
}

fd_plan *fd_get_plan(void) { return g_plan; }

fd_status fd_plan_workspace_bytes(fd_plan *plan, size_t *bytes) {
  if (!plan || !bytes) return fail(FD_ERR_INVALID_ARG, "NULL argument");
  *bytes = plan->o_part ? plan->ws_rows * (plan->d + 1) * sizeof(float) + plan->n_counters * sizeof(unsigned) : 0;
  return FD_OK;
}

fd_status fd_plan_set_split_policy(fd_plan *plan, int policy) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (policy != FD_SPLIT_BALANCED && policy != FD_SPLIT_EQUAL)
    return fail(FD_ERR_INVALID_ARG, "split policy %d unknown", policy);
  plan->split_policy = policy;
  return FD_OK;
}

fd_status fd_set_max_seqlen_hint(fd_plan *plan, int max_seqlen) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (max_seqlen < 0) return fail(FD_ERR_INVALID_ARG, "max_seqlen %d < 0", max_seqlen);
  plan->seqlen_hint = max_seqlen;
  return FD_OK;
}

fd_status fd_set_mean_seqlen_hint(fd_plan *plan, int mean_seqlen) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (mean_seqlen < 0) return fail(FD_ERR_INVALID_ARG, "mean_seqlen %d < 0", mean_seqlen);
  plan->mean_hint = mean_seqlen;
  return FD_OK;
}

fd_status fd_read_device_status(fd_plan *plan, int *code) {
  if (!plan || !code) return fail(FD_ERR_INVALID_ARG, "NULL argument");
  *code = 0;
  if (plan->device < 0 || !plan->status) return fail(FD_ERR_WORKSPACE, "host-only plan has no status word");
  fd::DeviceGuard guard(plan->device);
  unsigned v = 0;
  FD_CUDA_TRY(cudaDeviceSynchronize());
  FD_CUDA_TRY(cudaMemcpy(&v, plan->status, sizeof(v), cudaMemcpyDeviceToHost));
  FD_CUDA_TRY(cudaMemset(plan->status, 0, sizeof(unsigned)));
  // after an abandoned call the merge counters may be mid-count: start over
  if (v && plan->counters) FD_CUDA_TRY(cudaMemset(plan->counters, 0, plan->n_counters * sizeof(unsigned)));
  *code = static_cast<int>(v);
  if (v) return fail(FD_ERR_DEVICE_STATUS, "device status 0x%x", v);
  return FD_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// Descriptor validation

namespace {

fd_status check_tensor(const fd_tensor *t, const char *name, int ndim, bool unit_inner = true) {
  if (!t) return fail(FD_ERR_INVALID_ARG, "%s descriptor is NULL", name);
  if (!t->data) return fail(FD_ERR_INVALID_ARG, "%s data pointer is NULL", name);
  if (t->ndim != ndim) return fail(FD_ERR_INVALID_ARG, "%s has ndim %d, expected %d", name, t->ndim, ndim);
  for (int i = 0; i < ndim; ++i) {
    if (t->shape[i] < 0) return fail(FD_ERR_INVALID_ARG, "%s shape[%d] < 0", name, i);
    if (t->stride[i] < 0) return fail(FD_ERR_UNSUPPORTED, "%s stride[%d] < 0", name, i);
  }
  if (unit_inner && t->stride[ndim - 1] != 1 && t->shape[ndim - 1] > 1)
    return fail(FD_ERR_UNSUPPORTED, "%s innermost stride must be 1", name);
  return FD_OK;
}

#define FD_TRY(x)                   \
  do {                              \
    fd_status s_ = (x);             \
    if (s_ != FD_OK) return s_;     \
  } while (0)

fd_status encode_cache_map(CUtensorMap *map, const fd_tensor *c, const fd_plan *pl) {
  const int rowe = static_cast<int>(c->shape[3]);
  const int es = elem_bytes(c->dtype);
  const int row_bytes = rowe * es;
  const int box_bytes = row_bytes < 128 ? row_bytes : 128;
  const int bn = fd::stage1_block_n(pl->kind, pl->d);
  const int seg = pl->page < bn ? pl->page : bn;
  cuuint64_t dims[4] = {static_cast<cuuint64_t>(rowe), static_cast<cuuint64_t>(pl->hkv),
                        static_cast<cuuint64_t>(pl->page), static_cast<cuuint64_t>(c->shape[0])};
  cuuint64_t strides[3] = {static_cast<cuuint64_t>(c->stride[2] * es), static_cast<cuuint64_t>(c->stride[1] * es),
                           static_cast<cuuint64_t>(c->stride[0] * es)};
  cuuint32_t box[4] = {static_cast<cuuint32_t>(box_bytes / es), 1u, static_cast<cuuint32_t>(seg), 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMapSwizzle swz = box_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                           : box_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
  CUtensorMapDataType dt = c->dtype == FD_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(FD_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  // L2 promotion: whole 256-byte lines, except for 64-byte rows (int4, head
  // dim 128), where a 256-byte line spans four heads' rows of a slot and the
  // neighbours' CTAs often find it evicted (evict-first) before they read it
  const CUtensorMapL2promotion promo =
      box_bytes <= 64 ? CU_TENSOR_MAP_L2_PROMOTION_L2_64B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  CUresult r = fn(map, dt, 4, c->data, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, promo,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(FD_ERR_UNSUPPORTED, "cuTensorMapEncodeTiled rejected the cache layout (%d)", (int)r);
  return FD_OK;
}

// The descriptor of a cache depends only on its pointer, shape and strides,
// which a serving loop keeps fixed; re-encode only when they change.
fd_status cached_cache_map(CUtensorMap *map, const fd_tensor *c, fd_plan *pl, int which) {
  static_assert(sizeof(CUtensorMap) <= sizeof(pl->map_cache[0].map), "map cache slot");
  fd_plan::MapEntry &e = pl->map_cache[which];
  bool hit = e.valid && e.data == c->data;
  for (int i = 0; hit && i < 4; ++i) hit = e.shape[i] == c->shape[i] && e.stride[i] == c->stride[i];
  if (!hit) {
    FD_TRY(encode_cache_map(reinterpret_cast<CUtensorMap *>(e.map), c, pl));
    e.valid = true;
    e.data = c->data;
    for (int i = 0; i < 4; ++i) {
      e.shape[i] = c->shape[i];
      e.stride[i] = c->stride[i];
    }
  }
  std::memcpy(map, e.map, sizeof(CUtensorMap));
  return FD_OK;
}

}  // namespace

extern "C" fd_status fd_decode_paged(const fd_tensor *q, const fd_tensor *k_cache,
                                     const fd_tensor *v_cache, const fd_tensor *kv_scales,
                                     const fd_tensor *page_table, const fd_tensor *cache_seqlens,
                                     int q_per_req, int num_splits, fd_tensor *out, fd_tensor *lse,
                                     fd_stream_t stream) {
  fd_plan *pl = g_plan;
  if (!pl) return fail(FD_ERR_NO_PLAN, "no current plan on this thread (call fd_set_plan)");
  const int D = pl->d;
  // ---- q
  FD_TRY(check_tensor(q, "q", 4));
  if (q->dtype != FD_BF16) return fail(FD_ERR_INVALID_ARG, "q must be bf16");
  const int B = static_cast<int>(q->shape[0]);
  const int Tq = static_cast<int>(q->shape[1]);
  if (q->shape[2] != pl->hq || q->shape[3] != D)
    return fail(FD_ERR_INVALID_ARG, "q shape [%lld, %lld, %lld, %lld] does not match the plan (Hq=%d, D=%d)",
                (long long)q->shape[0], (long long)q->shape[1], (long long)q->shape[2], (long long)q->shape[3],
                pl->hq, D);
  if (B < 1 || B > pl->max_batch) return fail(FD_ERR_INVALID_ARG, "batch %d not in [1, %d]", B, pl->max_batch);
  if (q_per_req != Tq) return fail(FD_ERR_INVALID_ARG, "q_per_req %d != q.shape[1] %d", q_per_req, Tq);
  if (Tq < 1 || Tq > pl->max_q) return fail(FD_ERR_INVALID_ARG, "q_per_req %d not in [1, %d]", Tq, pl->max_q);
  if (!aligned(q->data, 16) || q->stride[0] % 8 || q->stride[1] % 8 || q->stride[2] % 8)
    return fail(FD_ERR_UNSUPPORTED, "q rows must be 16-byte aligned");
  // ---- caches
  const int want_dt = pl->kv_dtype;
  const int rowe = pl->kv_dtype == FD_INT4X2 ? D / 2 : D;
  for (int i = 0; i < 2; ++i) {
    const fd_tensor *c = i == 0 ? k_cache : v_cache;
    const char *nm = i == 0 ? "k_cache" : "v_cache";
    FD_TRY(check_tensor(c, nm, 4));
    if (c->dtype != want_dt) return fail(FD_ERR_INVALID_ARG, "%s dtype %d != plan kv dtype %d", nm, c->dtype, want_dt);
    if (c->shape[1] != pl->page || c->shape[2] != pl->hkv || c->shape[3] != rowe)
      return fail(FD_ERR_INVALID_ARG, "%s shape [N, %lld, %lld, %lld] != [N, P=%d, Hkv=%d, %d]", nm,
                  (long long)c->shape[1], (long long)c->shape[2], (long long)c->shape[3], pl->page, pl->hkv, rowe);
    if (c->shape[0] < 1 || c->shape[0] > 0x7fffffff)
      return fail(FD_ERR_INVALID_ARG, "%s must hold 1 .. 2^31-1 pages", nm);
    const int es = elem_bytes(c->dtype);
    if (!aligned(c->data, 16) || (c->stride[0] * es) % 16 || (c->stride[1] * es) % 16 || (c->stride[2] * es) % 16)
      return fail(FD_ERR_UNSUPPORTED, "%s base and strides must be multiples of 16 bytes", nm);
  }
  for (int i = 0; i < 4; ++i)
    if (k_cache->shape[i] != v_cache->shape[i]) return fail(FD_ERR_INVALID_ARG, "k_cache and v_cache shapes differ");
  const int num_pages = static_cast<int>(k_cache->shape[0]);
  // ---- scales
  const bool quant = pl->kv_dtype != FD_BF16;
  const int ng = pl->kv_dtype == FD_INT4X2 ? D / 32 : 1;
  if (quant) {
    FD_TRY(check_tensor(kv_scales, "kv_scales", 5));
    if (kv_scales->dtype != FD_FP32) return fail(FD_ERR_INVALID_ARG, "kv_scales must be fp32");
    if (kv_scales->shape[0] != 2 || kv_scales->shape[1] != num_pages || kv_scales->shape[2] != pl->page ||
        kv_scales->shape[3] != pl->hkv || kv_scales->shape[4] != ng)
      return fail(FD_ERR_INVALID_ARG, "kv_scales shape must be [2, %d, %d, %d, %d]", num_pages, pl->page, pl->hkv, ng);
    if (!aligned(kv_scales->data, 4 * ng))
      return fail(FD_ERR_UNSUPPORTED, "kv_scales base must be %d-byte aligned", 4 * ng);
    for (int i = 0; i < 4; ++i)
      if (kv_scales->stride[i] % ng)
        return fail(FD_ERR_UNSUPPORTED, "kv_scales strides must be multiples of %d", ng);
  } else if (kv_scales && kv_scales->data) {
    return fail(FD_ERR_INVALID_ARG, "kv_scales must be NULL for a bf16 cache");
  }
  // ---- metadata
  FD_TRY(check_tensor(page_table, "page_table", 2));
  if (page_table->dtype != FD_INT32 || page_table->shape[0] != B || page_table->shape[1] < 1)
    return fail(FD_ERR_INVALID_ARG, "page_table must be int32 [B=%d, W>=1]", B);
  if (page_table->shape[1] > 0x7fffffff / pl->page)
    return fail(FD_ERR_UNSUPPORTED, "page_table too wide");
  FD_TRY(check_tensor(cache_seqlens, "cache_seqlens", 1));
  if (cache_seqlens->dtype != FD_INT32 || cache_seqlens->shape[0] != B)
    return fail(FD_ERR_INVALID_ARG, "cache_seqlens must be int32 [B=%d]", B);
  // ---- outputs
  FD_TRY(check_tensor(out, "out", 4));
  if (out->dtype != FD_BF16 && out->dtype != FD_FP32) return fail(FD_ERR_INVALID_ARG, "out must be bf16 or fp32");
  if (out->shape[0] != B || out->shape[1] != Tq || out->shape[2] != pl->hq || out->shape[3] != D)
    return fail(FD_ERR_INVALID_ARG, "out shape must be [B, Tq, Hq, D]");
  {
    const int vec = out->dtype == FD_BF16 ? 8 : 4;
    if (!aligned(out->data, 16) || out->stride[0] % vec || out->stride[1] % vec || out->stride[2] % vec)
      return fail(FD_ERR_UNSUPPORTED, "out rows must be 16-byte aligned");
  }
  if (lse && lse->data) {
    FD_TRY(check_tensor(lse, "lse", 3, false));
    if (lse->dtype != FD_FP32 || lse->shape[0] != B || lse->shape[1] != Tq || lse->shape[2] != pl->hq)
      return fail(FD_ERR_INVALID_ARG, "lse must be fp32 [B, Tq, Hq]");
  }
  // ---- splits
  int S = num_splits;
  if (S < 0 || S > pl->max_splits) return fail(FD_ERR_INVALID_ARG, "num_splits %d not in [0, %d]", S, pl->max_splits);
  if (S == 0) {
    // inside the decode-attention warmup phase (outside capture) the call
    // first tunes its batch at the representative length if needed
    FD_TRY(fd::autotune_on_call(pl, B, reinterpret_cast<cudaStream_t>(stream)));
    S = fd::choose_splits(pl, B, pl->seqlen_hint);
  }
  if (pl->device < 0) return fail(FD_ERR_WORKSPACE, "host-only plan cannot decode");
  // Balanced splits (more than one request, a workspace with room for at
  // least two partials per output row): s_cap partial rows per output row.
  const size_t out_rows = static_cast<size_t>(B) * Tq * pl->hq;
  const int s_room = pl->o_part ? static_cast<int>(std::min<size_t>(64, pl->ws_rows / out_rows)) : 0;
  const bool balanced = pl->split_policy == FD_SPLIT_BALANCED && B > 1 && s_room >= 2;
  const int s_cap = balanced ? s_room : S;
  if (S > 1 && (!pl->o_part || out_rows * S > pl->ws_rows))
    return fail(FD_ERR_WORKSPACE, "plan workspace too small");
  // any request may be split: merge kernel (or fused merge) needed
  const bool merge = S > 1 || balanced;

  fd::DeviceGuard guard(pl->device);
  if (!guard.ok) return fail(FD_ERR_CUDA, "cannot make device %d current", pl->device);

  CUtensorMap tmk, tmv;
  FD_TRY(cached_cache_map(&tmk, k_cache, pl, 0));
  FD_TRY(cached_cache_map(&tmv, v_cache, pl, 1));

  fd::Stage1Params p;
  std::memset(&p, 0, sizeof(p));
  p.q = static_cast<const __nv_bfloat16 *>(q->data);
  p.q_sb = q->stride[0];
  p.q_st = q->stride[1];
  p.q_sh = q->stride[2];
  if (quant) {
    p.kv_scales = static_cast<const float *>(kv_scales->data);
    p.sc_sk = kv_scales->stride[0];
    p.sc_sp = kv_scales->stride[1];
    p.sc_ss = kv_scales->stride[2];
    p.sc_sh = kv_scales->stride[3];
  }
  p.page_table = static_cast<const int *>(page_table->data);
  p.pt_sb = page_table->stride[0];
  p.seqlens = static_cast<const int *>(cache_seqlens->data);
  p.sl_s = cache_seqlens->stride[0];
  p.num_pages = num_pages;
  p.page_size = pl->page;
  p.log2_page = pl->log2_page;
  p.max_pages = static_cast<int>(page_table->shape[1]);
  p.Tq = Tq;
  p.Hq = pl->hq;
  p.Hkv = pl->hkv;
  p.G = pl->hq / pl->hkv;
  p.R = p.G * Tq;
  p.row_tiles = (p.R + 15) / 16;
  p.num_splits = S;
  p.chunk_min = 0;
  p.balanced = balanced ? 1 : 0;
  p.batch = B;
  p.s_cap = s_cap;
  p.scale_log2 = pl->scale * 1.4426950408889634f;
  p.o_part = pl->o_part;
  p.lse_part = pl->lse_part;
  p.out = out->data;
  p.out_f32 = out->dtype == FD_FP32;
  p.o_sb = out->stride[0];
  p.o_st = out->stride[1];
  p.o_sh = out->stride[2];
  if (lse && lse->data) {
    p.lse = static_cast<float *>(lse->data);
    p.l_sb = lse->stride[0];
    p.l_st = lse->stride[1];
    p.l_sh = lse->stride[2];
  }
  p.status = pl->status;
  // The fused merge (FD_MERGE=fused) serves the equal policy only: under the
  // balanced one a request with no keys has no split CTA to write its rows.
  p.counters = (S > 1 && !balanced && !pl->merge_kernel) ? pl->counters : nullptr;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaEvent_t ev[3] = {nullptr, nullptr, nullptr};
  // Profiling events; under stream capture they become timed event nodes of
  // the graph (external records), so a replayed graph is profiled without
  // host launch gaps.
  unsigned rec_flags = cudaEventRecordDefault;
  if (pl->profiling) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    FD_CUDA_TRY(cudaStreamIsCapturing(st, &cs));
    if (cs == cudaStreamCaptureStatusActive) rec_flags = cudaEventRecordExternal;
    for (auto &x : ev) FD_CUDA_TRY(cudaEventCreate(&x));
    for (auto &x : ev) pl->prof_events.push_back(x);
    FD_CUDA_TRY(cudaEventRecordWithFlags(ev[0], st, rec_flags));
  }
  dim3 grid(p.row_tiles * S, pl->hkv, B);
  if (balanced) {
    // The batch has at most B * (S + 1) splits: sum_b ceil(n_b / cp) <=
    // n_total / cp + B, and n_total / cp <= B * S.
    const long long units = std::min<long long>(static_cast<long long>(B) * (S + 1), static_cast<long long>(B) * s_cap);
    const long long x = units * pl->hkv * p.row_tiles;
    if (x > 0x7fffffffLL) return fail(FD_ERR_UNSUPPORTED, "balanced split grid too large (%lld CTAs)", x);
    grid = dim3(static_cast<unsigned>(x), 1, 1);
  }
  // One wave of the expected CTAs (B * S splits; the balanced grid's extra
  // CTAs exit at once): one CTA per SM with a deeper ring.
  const long ctas = static_cast<long>(p.row_tiles) * S * pl->hkv * B;
  const bool deep = ctas <= pl->num_sms;
  // the tcgen05 kernel: quantised caches, head_dim 128, one row tile per CTA, merge by stage 2
  const bool tc = pl->quant_tc && pl->kind != fd::KV_BF16 && D == 128 && !p.counters;
  // NVTX ranges mark each stage's enqueue on the host timeline (nsys / ncu)
  nvtxRangePushA("fd_stage1");
  cudaError_t e = tc ? fd::launch_stage1_tc(pl->kind, !merge, tmk, tmv, p, grid, st)
                     : fd::launch_stage1(pl->kind, D, !merge, deep, tmk, tmv, p, grid, st);
  nvtxRangePop();
  if (pl->profiling) FD_CUDA_TRY(cudaEventRecordWithFlags(ev[1], st, rec_flags));
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "stage-1 launch failed: %s (%d)", cudaGetErrorString(e), (int)e);
  if (merge && !p.counters) {
    fd::Stage2Params p2;
    p2.o_part = pl->o_part;
    p2.lse_part = pl->lse_part;
    p2.B = B;
    p2.Tq = Tq;
    p2.Hq = pl->hq;
    p2.D = D;
    p2.num_splits = S;
    p2.balanced = p.balanced;
    p2.s_cap = s_cap;
    p2.seqlens = p.seqlens;
    p2.sl_s = p.sl_s;
    p2.log2_page = p.log2_page;
    p2.max_pages = p.max_pages;
    p2.chunk_min = p.chunk_min;
    p2.out = p.out;
    p2.out_f32 = p.out_f32;
    p2.o_sb = p.o_sb;
    p2.o_st = p.o_st;
    p2.o_sh = p.o_sh;
    p2.lse = p.lse;
    p2.l_sb = p.l_sb;
    p2.l_st = p.l_st;
    p2.l_sh = p.l_sh;
    nvtxRangePushA("fd_stage2");
    e = fd::launch_stage2(p2, st, !pl->profiling);
    nvtxRangePop();
    if (e != cudaSuccess) return fail(FD_ERR_CUDA, "stage-2 launch failed: %s (%d)", cudaGetErrorString(e), (int)e);
  }
  if (pl->profiling) FD_CUDA_TRY(cudaEventRecordWithFlags(ev[2], st, rec_flags));
  return FD_OK;
}

extern "C" fd_status fd_graph_metadata(const fd_tensor *req_to_token, const fd_tensor *req_pool_indices,
                                       const fd_tensor *seq_lens, int page_size, int q_mode, const fd_tensor *q_in,
                                       int q_stride, fd_tensor *page_table, fd_tensor *cache_seqlens,
                                       fd_tensor *cu_seqlens_k, fd_tensor *cu_seqlens_q, fd_tensor *status,
                                       fd_stream_t stream) {
  FD_TRY(check_tensor(req_to_token, "req_to_token", 2, false));
  if (req_to_token->dtype != FD_INT32) return fail(FD_ERR_INVALID_ARG, "req_to_token must be int32");
  FD_TRY(check_tensor(req_pool_indices, "req_pool_indices", 1, false));
  if (req_pool_indices->dtype != FD_INT32 && req_pool_indices->dtype != FD_INT64)
    return fail(FD_ERR_INVALID_ARG, "req_pool_indices must be int32 or int64");
  const int64_t B = req_pool_indices->shape[0];
  if (B > 65535) return fail(FD_ERR_UNSUPPORTED, "batch %lld > 65535", (long long)B);
  FD_TRY(check_tensor(seq_lens, "seq_lens", 1, false));
  if (seq_lens->dtype != FD_INT32 || seq_lens->shape[0] != B)
    return fail(FD_ERR_INVALID_ARG, "seq_lens must be int32 [B=%lld]", (long long)B);
  if (page_size < 1) return fail(FD_ERR_INVALID_ARG, "page_size %d < 1", page_size);
  if (q_mode != FD_QMODE_PRESET && q_mode != FD_QMODE_CUMSUM && q_mode != FD_QMODE_STRIDED)
    return fail(FD_ERR_INVALID_ARG, "q_mode %d unknown", q_mode);
  if (q_mode != FD_QMODE_STRIDED) {
    FD_TRY(check_tensor(q_in, "q_in", 1, false));
    const int64_t want = q_mode == FD_QMODE_PRESET ? B + 1 : B;
    if (q_in->dtype != FD_INT32 || q_in->shape[0] != want)
      return fail(FD_ERR_INVALID_ARG, "q_in must be int32 [%lld]", (long long)want);
  } else if (q_stride < 0) {
    return fail(FD_ERR_INVALID_ARG, "q_stride %d < 0", q_stride);
  }
  FD_TRY(check_tensor(page_table, "page_table", 2));
  if (page_table->dtype != FD_INT32 || page_table->shape[0] != B || page_table->shape[1] < 1)
    return fail(FD_ERR_INVALID_ARG, "page_table must be int32 [B=%lld, W>=1]", (long long)B);
  FD_TRY(check_tensor(cache_seqlens, "cache_seqlens", 1, false));
  if (cache_seqlens->dtype != FD_INT32 || cache_seqlens->shape[0] != B)
    return fail(FD_ERR_INVALID_ARG, "cache_seqlens must be int32 [B]");
  for (int i = 0; i < 2; ++i) {
    const fd_tensor *c = i ? cu_seqlens_q : cu_seqlens_k;
    const char *nm = i ? "cu_seqlens_q" : "cu_seqlens_k";
    FD_TRY(check_tensor(c, nm, 1));
    if (c->dtype != FD_INT32 || c->shape[0] != B + 1) return fail(FD_ERR_INVALID_ARG, "%s must be int32 [B + 1]", nm);
  }
  if (status && status->data) {
    FD_TRY(check_tensor(status, "status", 1));
    if (status->dtype != FD_INT32 || status->shape[0] < 1) return fail(FD_ERR_INVALID_ARG, "status must be int32 [1]");
  }
  fd::MetaParams p;
  std::memset(&p, 0, sizeof(p));
  p.req_to_token = static_cast<const int *>(req_to_token->data);
  p.rt_sr = req_to_token->stride[0];
  p.rt_sc = req_to_token->stride[1];
  p.pool_rows = req_to_token->shape[0];
  p.pool_cols = req_to_token->shape[1];
  p.pool_idx = req_pool_indices->data;
  p.idx64 = req_pool_indices->dtype == FD_INT64;
  p.idx_s = req_pool_indices->stride[0];
  p.seq_lens = static_cast<const int *>(seq_lens->data);
  p.sl_s = seq_lens->stride[0];
  p.B = static_cast<int>(B);
  p.P = page_size;
  p.W = static_cast<int>(std::min<int64_t>(page_table->shape[1], 0x7fffffff));
  p.q_mode = q_mode;
  p.q_in = q_mode != FD_QMODE_STRIDED ? static_cast<const int *>(q_in->data) : nullptr;
  p.q_s = q_mode != FD_QMODE_STRIDED ? q_in->stride[0] : 0;
  p.q_stride = q_stride;
  p.page_table = static_cast<int *>(page_table->data);
  p.pt_sb = page_table->stride[0];
  p.cache_seqlens = static_cast<int *>(cache_seqlens->data);
  if (cache_seqlens->stride[0] != 1 && B > 1) return fail(FD_ERR_UNSUPPORTED, "cache_seqlens must be contiguous");
  p.cu_k = static_cast<int *>(cu_seqlens_k->data);
  p.cu_q = static_cast<int *>(cu_seqlens_q->data);
  p.status = (status && status->data) ? static_cast<unsigned *>(status->data) : nullptr;
  cudaError_t e = fd::launch_graph_metadata(p, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(FD_ERR_CUDA, "graph-metadata launch failed: %s (%d)", cudaGetErrorString(e), (int)e);
  return FD_OK;
}

extern "C" fd_status fd_profile_begin(fd_plan *plan) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  if (plan->device < 0) return fail(FD_ERR_WORKSPACE, "host-only plan cannot profile");
  plan->profiling = true;
  return FD_OK;
}

extern "C" fd_status fd_profile_end(fd_plan *plan, int *calls, double *stage1_ms, double *stage2_ms) {
  if (!plan) return fail(FD_ERR_INVALID_ARG, "plan is NULL");
  fd::DeviceGuard guard(plan->device);
  plan->profiling = false;
  double t1 = 0.0, t2 = 0.0;
  fd_status st = FD_OK;
  const size_t n = plan->prof_events.size() / 3;
  for (size_t i = 0; i < n; ++i) {
    cudaEvent_t *e = &plan->prof_events[3 * i];
    float a = 0.f, b = 0.f;
    if (st == FD_OK && (cudaEventSynchronize(e[2]) != cudaSuccess || cudaEventElapsedTime(&a, e[0], e[1]) != cudaSuccess ||
                        cudaEventElapsedTime(&b, e[1], e[2]) != cudaSuccess))
      st = fail(FD_ERR_CUDA, "profiling events failed");
    t1 += a;
    t2 += b;
  }
  for (cudaEvent_t e : plan->prof_events) cudaEventDestroy(e);
  plan->prof_events.clear();
  if (calls) *calls = static_cast<int>(n);
  if (stage1_ms) *stage1_ms = t1;
  if (stage2_ms) *stage2_ms = t2;
  return st;
}
