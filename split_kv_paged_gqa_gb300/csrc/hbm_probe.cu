// hbm_probe.cu - HBM bandwidth probes: a read-only stream and a copy.
//
// They give the roofline of the decode kernels a denominator measured on the
// same GPU in the same process. The decode path is a read stream (KV pages
// in, a few KB of outputs out), so its natural ceiling is what a pure read
// stream reaches; a copy moves as many bytes out as in and pays the bus
// turnarounds between reads and writes, so it sits a little lower.
//
// Both kernels walk the buffer with 16-byte vector accesses, eight
// independent loads in flight per thread, on a grid of a whole number of CTAs
// per SM, each CTA streaming through 64 KiB tiles of consecutive memory. The read kernel folds every word it loads into an
// XOR per thread and combines those into the caller's 16-byte sink with one
// atomic per warp, so no load can be dropped by the compiler and the sink
// holds a checkable value: the XOR of all 16-byte words of the buffer.
#include <cuda_runtime.h>

#include <stdint.h>

#include "fd.h"
#include "plan.h"

namespace {

constexpr int kThreads = 512;
constexpr int kCtasPerSm = 4;
constexpr int kUnroll = 8;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// The buffer is cut into tiles of kThreads * kUnroll words (64 KiB), dealt to
// the CTAs round robin; within a tile, load u of thread t takes word
// u * kThreads + t, so each of a CTA's kUnroll loads in flight covers 8 KiB of
// consecutive memory (DRAM pages stay open, as with the decode kernels' TMA
// boxes of whole cache pages).
constexpr size_t kTile = static_cast<size_t>(kThreads) * kUnroll;

__global__ void __launch_bounds__(kThreads) hbm_read_kernel(const uint4 *__restrict__ src, size_t n, uint32_t *sink) {
  uint4 acc = make_uint4(0u, 0u, 0u, 0u);
  const size_t full_tiles = n / kTile;
  for (size_t t = blockIdx.x; t < full_tiles; t += gridDim.x) {
    const uint4 *p = src + t * kTile + threadIdx.x;
    uint4 v[kUnroll];
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) v[k] = ld_stream(p + k * kThreads);
#pragma unroll
    for (int k = 0; k < kUnroll; ++k) {
      acc.x ^= v[k].x;
      acc.y ^= v[k].y;
      acc.z ^= v[k].z;
      acc.w ^= v[k].w;
    }
  }
  // the partial last tile, word by word
  if (blockIdx.x == full_tiles % gridDim.x) {
    for (size_t i = full_tiles * kTile + threadIdx.x; i < n; i += kThreads) {
      const uint4 v = ld_stream(src + i);
      acc.x ^= v.x;
      acc.y ^= v.y;
      acc.z ^= v.z;
      acc.w ^= v.w;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    acc.x ^= __shfl_xor_sync(0xffffffffu, acc.x, o);
    acc.y ^= __shfl_xor_sync(0xffffffffu, acc.y, o);
    acc.z ^= __shfl_xor_sync(0xffffffffu, acc.z, o);
    acc.w ^= __shfl_xor_sync(0xffffffffu, acc.w, o);
  }
  if ((threadIdx.x & 31) == 0) {
    atomicXor(sink + 0, acc.x);
    atomicXor(sink + 1, acc.y);
    atomicXor(sink + 2, acc.z);
    atomicXor(sink + 3, acc.w);
  }
}

__device__ __forceinline__ void st_stream(uint4 *p, const uint4 &v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
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
    for (int k = 0; k < kUnroll; ++k) st_stream(dst + base + k * kThreads, v[k]);
  }
  if (blockIdx.x == full_tiles % gridDim.x) {
    for (size_t i = full_tiles * kTile + threadIdx.x; i < n; i += kThreads) st_stream(dst + i, ld_stream(src + i));
  }
}

fd_status probe_grid(size_t n16, unsigned *grid) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "device query failed: %s", cudaGetErrorString(e));
  // a whole number of CTAs per SM, fewer when the buffer is small
  const size_t full = static_cast<size_t>(sms) * kCtasPerSm;
  const size_t need = (n16 + kTile - 1) / kTile;
  *grid = static_cast<unsigned>(need < full ? (need > 0 ? need : 1) : full);
  return FD_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" fd_status fd_probe_hbm_read(const void *src, size_t bytes, uint32_t *sink, fd_stream_t stream) {
  if (!src || !sink) return fd::fail(FD_ERR_INVALID_ARG, "NULL pointer");
  if (!aligned16(src) || !aligned16(sink) || bytes % 16)
    return fd::fail(FD_ERR_UNSUPPORTED, "src and sink must be 16-byte aligned and bytes a multiple of 16");
  if (bytes == 0) return FD_OK;
  unsigned grid = 0;
  const fd_status st = probe_grid(bytes / 16, &grid);
  if (st != FD_OK) return st;
  hbm_read_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(static_cast<const uint4 *>(src),
                                                                                 bytes / 16, sink);
  const cudaError_t e = cudaGetLastError();
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
  unsigned grid = 0;
  const fd_status st = probe_grid(bytes / 16, &grid);
  if (st != FD_OK) return st;
  hbm_copy_kernel<<<grid, kThreads, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4 *>(src), static_cast<uint4 *>(dst), bytes / 16);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fd::fail(FD_ERR_CUDA, "copy probe launch failed: %s", cudaGetErrorString(e));
  return FD_OK;
}
