// fd_static.cu - a decode entry point that allocates no device memory.
//
// Some callers cannot call cudaMalloc. A serving engine may have reserved all
// of the GPU's memory for its own pool before it loads this library. A plugin
// may live inside a host process that forbids foreign device allocations.
// For such callers, fd_decode_paged_static runs the same kernels as
// fd_decode_paged, but without a plan. The split workspace is a
// fixed array in this file (kStaticScratchBytes, 32 MiB). The library holds
// that array on every GPU that loads it, until the process exits.
//
// On the first call on a device, with that device current, the call does a
// one-time set-up:
//  * it looks up the array's device address with cudaGetSymbolAddress;
//  * it reads the device's SM count and compute capability (attribute
//    queries, which allocate nothing);
//  * it raises the kernels' shared-memory limit.
//
// This path always merges splits with the stage-2 kernel: the array holds
// only the fp32 split partials and their LSEs.
//
// The call never allocates. It rejects a workspace need larger than the array
// with FD_ERR_WORKSPACE. All calls share the array; calls that overlap on the
// GPU race on it, so serialise them on one stream. The kernels overwrite
// every workspace row they read, so nothing needs clearing between calls.
#include <cuda_runtime.h>

#include <cmath>
#include <cstring>
#include <mutex>

#include "fd.h"
#include "kernels.h"
#include "plan.h"

namespace {

constexpr size_t kStaticScratchBytes = 32ull << 20;
constexpr int kMaxDevices = 64;
constexpr int kMaxHeads = 4096;

// The scratch lives here, in device global memory, one copy per device.
static __device__ __align__(256) float g_static_scratch[kStaticScratchBytes / sizeof(float)];
// Kernels record bad metadata here; this entry point does not report it.
static __device__ __align__(256) unsigned g_static_status;

struct DeviceSetup {
  float *scratch = nullptr;
  unsigned *status = nullptr;
  int num_sms = 0;        // the stage-1 variant choice depends on it, as in a plan
  unsigned prepared = 0;  // bit (kind * 2 + (D == 128)) : shared-memory limit raised
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];

// One-time set-up on the current device. Takes the array addresses; never allocates.
fd_status setup_device(int dev, int kind, int head_dim, DeviceSetup *out) {
  if (dev < 0 || dev >= kMaxDevices) return fd::fail(FD_ERR_UNSUPPORTED, "device %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_setup_mu);
  DeviceSetup &s = g_setup[dev];
  if (!s.scratch) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess)
      return fd::fail(FD_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
    void *q = nullptr;
    e = cudaGetSymbolAddress(&q, g_static_status);
    if (e != cudaSuccess)
      return fd::fail(FD_ERR_CUDA, "cudaGetSymbolAddress(status) failed: %s", cudaGetErrorString(e));
    int sms = 0, major = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (e != cudaSuccess)
      return fd::fail(FD_ERR_CUDA, "device attribute query failed: %s", cudaGetErrorString(e));
    if (major < 10)
      return fd::fail(FD_ERR_UNSUPPORTED, "device %d has compute capability %d.x; the kernels need 10.x or later",
                      dev, major);
    s.scratch = static_cast<float *>(p);
    s.status = static_cast<unsigned *>(q);
    s.num_sms = sms;
  }
  const unsigned bit = 1u << (kind * 2 + (head_dim == 128 ? 1 : 0));
  if (!(s.prepared & bit)) {
    cudaError_t e = fd::stage1_prepare(kind, head_dim);
    if (e != cudaSuccess)
      return fd::fail(FD_ERR_CUDA, "kernel set-up failed: %s", cudaGetErrorString(e));
    s.prepared |= bit;
  }
  *out = s;
  return FD_OK;
}

}  // namespace

extern "C" fd_status fd_decode_paged_static(const fd_tensor *q, const fd_tensor *k_cache,
                                            const fd_tensor *v_cache, const fd_tensor *kv_scales,
                                            const fd_tensor *page_table, const fd_tensor *cache_seqlens,
                                            int q_per_req, int num_splits, float softmax_scale,
                                            fd_tensor *out, fd_tensor *lse, fd_stream_t stream) {
  // Geometry comes from the descriptors; fd_decode_paged re-checks all of them.
  if (!q || !k_cache || q->ndim != 4 || k_cache->ndim != 4)
    return fd::fail(FD_ERR_INVALID_ARG, "q and k_cache must be 4-D descriptors");
  if (num_splits < 1 || num_splits > 64)
    return fd::fail(FD_ERR_INVALID_ARG, "num_splits %d not in [1, 64] (no tuning table here)", num_splits);
  if (!(softmax_scale >= 0.f) || std::isinf(softmax_scale))
    return fd::fail(FD_ERR_INVALID_ARG, "softmax_scale must be finite and >= 0");
  const int B = static_cast<int>(q->shape[0]), Tq = static_cast<int>(q->shape[1]);
  const int Hq = static_cast<int>(q->shape[2]), D = static_cast<int>(q->shape[3]);
  const int P = static_cast<int>(k_cache->shape[1]), Hkv = static_cast<int>(k_cache->shape[2]);
  int kind;
  switch (k_cache->dtype) {
    case FD_BF16: kind = fd::KV_BF16; break;
    case FD_INT8: kind = fd::KV_I8; break;
    case FD_INT4X2: kind = fd::KV_I4; break;
    default: return fd::fail(FD_ERR_UNSUPPORTED, "k_cache dtype %d not supported", k_cache->dtype);
  }
  if (D != 64 && D != 128) return fd::fail(FD_ERR_UNSUPPORTED, "head_dim %d not supported (64 or 128)", D);
  if (P < 8 || P > 256 || (P & (P - 1)))
    return fd::fail(FD_ERR_UNSUPPORTED, "page_size %d must be a power of two in [8, 256]", P);
  // (the head bound keeps the size product below in range: < 2^51)
  if (B < 1 || B > 65535 || Tq < 1 || Tq > 64 || Hkv < 1 || Hq < 1 || Hq > kMaxHeads || Hq % Hkv)
    return fd::fail(FD_ERR_INVALID_ARG, "bad batch / query tokens / head counts (Hq at most %d)", kMaxHeads);
  const size_t rows = static_cast<size_t>(B) * Tq * Hq * num_splits;
  const size_t need = num_splits > 1 ? rows * (static_cast<size_t>(D) + 1) * sizeof(float) : 0;
  if (need > kStaticScratchBytes)
    return fd::fail(FD_ERR_WORKSPACE,
                    "this call needs %zu bytes of split workspace (batch x tokens x heads x splits = %zu rows "
                    "of %d floats + LSE); the static scratch holds %zu bytes: use fewer splits or "
                    "fd_decode_paged with a plan",
                    need, rows, D, kStaticScratchBytes);

  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "cudaGetDevice failed: %s", cudaGetErrorString(e));
  DeviceSetup s;
  fd_status st = setup_device(dev, kind, D, &s);
  if (st != FD_OK) return st;

  // A plan on the stack whose workspace is the static scratch (no allocation).
  fd_plan pl;
  pl.device = dev;
  pl.num_sms = s.num_sms;
  pl.max_batch = B;
  pl.max_q = Tq;
  pl.hq = Hq;
  pl.hkv = Hkv;
  pl.d = D;
  pl.page = P;
  int lp = 0;
  while ((1 << lp) < P) ++lp;
  pl.log2_page = lp;
  pl.kv_dtype = static_cast<fd_dtype>(k_cache->dtype);
  pl.kind = kind;
  pl.max_splits = num_splits;
  pl.split_policy = FD_SPLIT_EQUAL;  // the scratch is sized for num_splits rows per output row
  pl.scale = softmax_scale > 0.f ? softmax_scale : 1.0f / std::sqrt(static_cast<float>(D));
  pl.o_part = s.scratch;
  pl.lse_part = s.scratch + rows * D;
  pl.ws_rows = rows;
  pl.status = s.status;
  pl.merge_kernel = true;  // splits merge in the stage-2 kernel: no counters
  pl.counters = nullptr;
  pl.n_counters = 0;

  fd_plan *prev = fd_get_plan();
  fd_set_plan(&pl);
  st = fd_decode_paged(q, k_cache, v_cache, kv_scales, page_table, cache_seqlens, q_per_req, num_splits, out,
                       lse, stream);
  fd_set_plan(prev);
  return st;
}
