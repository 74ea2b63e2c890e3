// Host-to-device copy driven by the SMs (opt_copy_from_host).
//
// The gradients of a training step may arrive in page-locked host memory.
// On GB300 hosts the copy engines' host-to-device rate from such memory
// varies with the pages and over time (from 211 GB/s down to 13-40 GB/s on
// some buffers of some hosts), while SM loads of the same buffers over the
// coherent CPU-GPU link hold 211 GB/s.  This kernel reads the host buffer
// with plain loads and writes device memory: 32 CTAs of 256 threads, 128
// bytes per thread per iteration (eight 16-byte loads issued before their
// stores, about 1 MB in flight over the link), a grid-stride loop.  Its CTAs
// need no shared memory and few registers, so they fit on an SM beside a
// Newton-Schulz GEMM CTA, and the copy overlaps the optimizer's kernels on
// another stream while leaving most SMs untouched.

#include <cuda_runtime.h>

#include "internal.h"

namespace mpopt {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyCtas = 16;
constexpr int kCopyUnroll = 12;

__global__ void __launch_bounds__(kCopyThreads)
copy_from_host_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t n16,
                      const uint32_t* __restrict__ src4, uint32_t* __restrict__ dst4, size_t n4_tail_begin,
                      size_t n4) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  // kCopyUnroll 16-byte elements per thread and iteration, all loaded
  // before any is stored
  for (; i + (kCopyUnroll - 1) * stride < n16; i += kCopyUnroll * stride) {
    uint4 v[kCopyUnroll];
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) v[k] = __ldcs(src + i + k * stride);
#pragma unroll
    for (int k = 0; k < kCopyUnroll; ++k) __stcs(dst + i + k * stride, v[k]);
  }
  for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
  // 4-byte words after the last whole 16 bytes (or all of them when the
  // pointers do not allow 16-byte accesses)
  for (size_t j = n4_tail_begin + static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x; j < n4;
       j += stride)
    dst4[j] = src4[j];
}

}  // namespace

cudaError_t launch_copy_from_host(void* dst, const void* src, size_t bytes, cudaStream_t stream) {
  if (bytes == 0) return cudaSuccess;
  const bool vec = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15u) == 0;
  const size_t n4 = bytes / 4;
  const size_t n16 = vec ? bytes / 16 : 0;
  const size_t work = vec ? n16 : n4;
  const size_t per_cta = kCopyUnroll * static_cast<size_t>(kCopyThreads);
  size_t grid = (work + per_cta - 1) / per_cta;
  if (grid > static_cast<size_t>(kCopyCtas)) grid = kCopyCtas;
  if (grid == 0) grid = 1;
  copy_from_host_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, stream>>>(
      static_cast<const uint4*>(src), static_cast<uint4*>(dst), n16, static_cast<const uint32_t*>(src),
      static_cast<uint32_t*>(dst), n16 * 4, n4);
  return cudaGetLastError();
}

}  // namespace mpopt
