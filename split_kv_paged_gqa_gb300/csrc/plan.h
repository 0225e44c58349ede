// plan.h - the plan object behind the opaque fd_plan handle.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <map>
#include <string>
#include <utility>
#include <vector>

#include "fd.h"

struct fd_plan {
  // geometry
  int device = -1;
  int max_batch = 0, max_q = 0, hq = 0, hkv = 0, d = 0, page = 0, log2_page = 0;
  fd_dtype kv_dtype = FD_BF16;
  int kind = 0;  // fd::KvKind
  int max_splits = 1;
  float scale = 0.f;
  int num_sms = 152;
  std::string gpu_name = "host";

  // device memory owned by the plan
  float *o_part = nullptr;    // [max_batch * max_q * hq * max_splits, d]
  float *lse_part = nullptr;  // [max_batch * max_q * hq * max_splits]
  size_t ws_rows = 0;
  unsigned *status = nullptr;
  unsigned *counters = nullptr;  // [max_batch * hkv * max row tiles], fused split merge
  size_t n_counters = 0;
  bool merge_kernel = true;      // merge splits with the stage-2 kernel (FD_MERGE=fused: in stage 1)
  int split_policy = FD_SPLIT_BALANCED;  // an fd_split_policy
  bool quant_tc = false;  // INT8 / INT4 with head_dim 128 on the tcgen05 stage-1 kernel (FD_QUANT_KERNEL=tc)

  // num_splits selection
  int seqlen_hint = 0;  // host-known max of cache_seqlens (0: unknown)
  int mean_hint = 0;    // host-known mean of cache_seqlens (0: unknown)
  std::map<std::pair<int, int>, int> table;         // (batch, bucket) -> num_splits
  std::map<std::pair<int, int>, double> table_time;  // (batch, bucket) -> best time
  std::map<std::pair<int, int>, int> memo;          // nearest-key lookups, cleared on save
  std::string cache_dir;
  bool cache_loaded = false;
  fd_timer_fn timer = nullptr;
  void *timer_user = nullptr;
  fd_tune_inputs_fn input_hook = nullptr;  // representative tuning inputs (rebuild hook)
  void *input_user = nullptr;
  int searches = 0, cache_hits = 0;

  // last encoded TMA descriptors of the K and V caches (host-side cache:
  // encoding costs microseconds of CPU per call otherwise)
  struct MapEntry {
    bool valid = false;
    const void *data = nullptr;
    int64_t shape[4] = {0, 0, 0, 0};
    int64_t stride[4] = {0, 0, 0, 0};
    alignas(64) unsigned char map[128];
  };
  MapEntry map_cache[2];

  // per-stage timing events (fd_profile_begin / fd_profile_end)
  bool profiling = false;
  std::vector<cudaEvent_t> prof_events;  // 3 per call: start, after stage 1, after stage 2
};

namespace fd {

// Thread-local error text (defined in fd_api.cpp).
fd_status fail(fd_status s, const char *fmt, ...);

// num_splits for a call with batch B and host-known max length (0 = unknown).
int choose_splits(fd_plan *plan, int batch, int max_seqlen);

// Warmup-scope tuning of a decode call with num_splits = 0 (autotune.cu):
// inside the decode-attention warmup phase and outside capture, tunes the
// call's batch at the representative KV length if the table lacks it.
fd_status autotune_on_call(fd_plan *plan, int batch, cudaStream_t stream);

// Autotune cache helpers (autotune.cu).
std::string autotune_key(const fd_plan *plan);
fd_status autotune_load(fd_plan *plan);
fd_status autotune_save(fd_plan *plan);

// Scoped device switch: makes `dev` current, restores the previous device.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (dev < 0) return;
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
  }
};

}  // namespace fd
