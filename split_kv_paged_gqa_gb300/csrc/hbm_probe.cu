// hbm_probe.cu - HBM bandwidth probes: a read-only stream and a copy.
//
// They give the roofline of the decode kernels a denominator measured on the
// same GPU in the same process. The decode path is a read stream (KV pages
// in, a few KB of outputs out), so its natural ceiling is what a pure read
// stream reaches; a copy moves as many bytes out as in and pays the bus
// turnarounds between reads and writes, so it sits a little lower.
//
// The read probe reads the way the decode kernels do: bulk copies (the TMA
// engine) of 32 KiB chunks into a ring of shared-memory stages, issued by one
// thread and completed on mbarriers; the other warps fold every 16-byte word
// that lands into an XOR, combined into the caller's 16-byte sink with one
// atomic per warp, so the sink holds a checkable value: the XOR of all
// 16-byte words of the buffer. One CTA per SM, six stages (192 KiB in flight
// per SM); each CTA streams one run of consecutive chunks (dealing chunks
// round robin instead measured 3 % lower).
//
// The copy probe moves 16-byte vectors (non-coherent loads, plain stores;
// streaming stores measured 1.5 % lower in the median), eight loads in flight
// per thread, four 512-thread CTAs per SM; the buffer is
// cut into 64 KiB tiles dealt to the CTAs round robin, and load u of thread t
// takes word u * 512 + t of a tile, so each load instruction of a CTA covers
// 8 KiB of consecutive memory.
#include <cuda_runtime.h>

#include <stdint.h>

#include "fd.h"
#include "plan.h"
#include "ptx.cuh"

namespace {

using namespace fd;

// 1-D bulk copy (TMA engine) of `bytes` (a multiple of 16; both addresses
// 16-byte aligned) into shared memory, completing its bytes on bar.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, unsigned bytes, uint64_t *bar,
                                          uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// ---- read probe
constexpr int kRThreads = 256;  // warp 0 issues the copies; warps 1..7 fold
constexpr int kRStages = 6;
constexpr unsigned kRChunk = 32768;
constexpr int kRSmem = kRStages * static_cast<int>(kRChunk) + 2 * kRStages * 8;

// Waits give up after a second and set this word (the probe has no status
// output of its own; a read that gave up leaves a wrong XOR in the sink).
__device__ unsigned g_probe_status;
constexpr unsigned long long kProbeWaitNs = 1000000000ull;

__global__ void __launch_bounds__(kRThreads, 1) hbm_read_kernel(const uint8_t *__restrict__ src, size_t bytes,
                                                               uint32_t *sink) {
  extern __shared__ __align__(1024) uint8_t ring[];
  uint64_t *full = reinterpret_cast<uint64_t *>(ring + kRStages * kRChunk);
  uint64_t *empty = full + kRStages;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int i = 0; i < kRStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kRThreads / 32 - 1);
    }
    fence_mbar_init();
  }
  __syncthreads();
  // CTA b streams chunks [b * per, b * per + mine): one run of consecutive
  // memory per CTA
  const size_t n_chunks = (bytes + kRChunk - 1) / kRChunk;
  const size_t per = (n_chunks + gridDim.x - 1) / gridDim.x;
  const size_t first = static_cast<size_t>(blockIdx.x) * per;
  const size_t mine = first < n_chunks ? (n_chunks - first < per ? n_chunks - first : per) : 0;
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      size_t k = 0;
      for (; k < mine; ++k) {
        const int st = static_cast<int>(k % kRStages);
        const unsigned ph = static_cast<unsigned>((k / kRStages) & 1);
        if (!mbar_wait(&empty[st], ph ^ 1, &g_probe_status, kProbeWaitNs)) break;
        const size_t off = (first + k) * static_cast<size_t>(kRChunk);
        const unsigned sz = static_cast<unsigned>(bytes - off < kRChunk ? bytes - off : kRChunk);
        mbar_arrive_expect_tx(&full[st], sz);
        bulk_load(ring + st * kRChunk, src + off, sz, &full[st], pol);
      }
      // drain: the latest phase of every stage this thread filled has landed
      for (size_t j = k > kRStages ? k - kRStages : 0; j < k; ++j)
        mbar_wait(&full[j % kRStages], static_cast<unsigned>((j / kRStages) & 1), &g_probe_status, kProbeWaitNs);
    }
  } else {
    const int t = threadIdx.x - 32;
    for (size_t k = 0; k < mine; ++k) {
      const int st = static_cast<int>(k % kRStages);
      const unsigned ph = static_cast<unsigned>((k / kRStages) & 1);
      if (!mbar_wait_warp(&full[st], ph, &g_probe_status, kProbeWaitNs)) break;
      const size_t off = (first + k) * static_cast<size_t>(kRChunk);
      const int words = static_cast<int>((bytes - off < kRChunk ? bytes - off : kRChunk) / 16);
      const uint4 *buf = reinterpret_cast<const uint4 *>(ring + st * kRChunk);
      for (int i = t; i < words; i += kRThreads - 32) {
        const uint4 v = buf[i];
        acc.x ^= v.x;
        acc.y ^= v.y;
        acc.z ^= v.z;
        acc.w ^= v.w;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[st]);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc.x ^= __shfl_xor_sync(0xffffffffu, acc.x, o);
    acc.y ^= __shfl_xor_sync(0xffffffffu, acc.y, o);
    acc.z ^= __shfl_xor_sync(0xffffffffu, acc.z, o);
    acc.w ^= __shfl_xor_sync(0xffffffffu, acc.w, o);
  }
  if (lane == 0 && warp > 0) {
    atomicXor(sink + 0, acc.x);
    atomicXor(sink + 1, acc.y);
    atomicXor(sink + 2, acc.z);
    atomicXor(sink + 3, acc.w);
  }
}

// ---- copy probe
constexpr int kThreads = 512;
constexpr int kCtasPerSm = 4;
constexpr int kUnroll = 8;
constexpr size_t kTile = static_cast<size_t>(kThreads) * kUnroll;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__global__ void __launch_bounds__(kThreads) hbm_copy_kernel(const uint4 *__restrict__ src, uint4 *__restrict__ dst,
                                                          size_t n) {
  const size_t full_tiles = n / kTile;
  for (size_t t = blockIdx.x; t < full_tiles; t += gridDim.x) {
    const size_t base = t * kTile + threadIdx.x;
    uint4 v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) v[k] = ld_stream(src + base + k * kThreads);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) dst[base + k * kThreads] = v[k];
  }
  // the partial last tile, word by word
  if (blockIdx.x == full_tiles % gridDim.x) {
    for (size_t i = full_tiles * kTile + threadIdx.x; i < n; i += kThreads) dst[i] = ld_stream(src + i);
  }
}

fd_status num_sms(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  return FD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fd_status fd_probe_hbm_read(const void *src, size_t bytes, uint32_t *sink, fd_stream_t stream) {
  if (!src || !sink) return fd::fail(FD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(sink) || bytes % 16)
    return fd::fail(FD_ERR_UNSUPPORTED, "src and sink must be 16-byte aligned and bytes a multiple of 16");
  if (bytes == 0) return FD_OK;
  int sms = 0;
  const fd_status st = num_sms(&sms);
  if (st != FD_OK) return st;
  cudaError_t e = cudaFuncSetAttribute(hbm_read_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem);
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "read probe set-up failed: %s", cudaGetErrorString(e));
  const size_t n_chunks = (bytes + kRChunk - 1) / kRChunk;
  const unsigned grid = static_cast<unsigned>(n_chunks < static_cast<size_t>(sms) ? n_chunks : sms);
  hbm_read_kernel<<<grid, kRThreads, kRSmem, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint8_t *>(src), bytes, sink);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "read probe launch failed: %s", cudaGetErrorString(e));
  return FD_OK;
}

extern "C" fd_status fd_probe_hbm_copy(const void *src, void *dst, size_t bytes, fd_stream_t stream) {
  if (!src || !dst) return fd::fail(FD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(dst) || bytes % 16)
    return fd::fail(FD_ERR_UNSUPPORTED, "src and dst must be 16-byte aligned and bytes a multiple of 16");
  const char *a = static_cast<const char *>(src);
  const char *b = static_cast<const char *>(dst);
  if (a < b + bytes && b < a + bytes) return fd::fail(FD_ERR_INVALID_ARG, "src and dst overlap");
  if (bytes == 0) return FD_OK;
  int sms = 0;
  const fd_status st = num_sms(&sms);
  if (st != FD_OK) return st;
  // a whole number of CTAs per SM, fewer when the buffer is small
  const size_t n16 = bytes / 16;
  const size_t full = static_cast<size_t>(sms) * kCtasPerSm;
  const size_t need = (n16 + kTile - 1) / kTile;
  const unsigned grid = static_cast<unsigned>(need < full ? (need > 0 ? need : 1) : full);
  hbm_copy_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), n16);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "copy probe launch failed: %s", cudaGetErrorString(e));
  return FD_OK;
}
