// Global gradient-norm clipping for sm_103a ("02 · Optimizer：算法与 infra"
// §11.1; §11.4: one norm over the gradients of both optimizer groups):
//
//   total_norm = sqrt(sum_p ||g_p||^2)
//   clip_coeff = max_norm / (total_norm + 1e-6);  scale = clip_coeff if < 1 else 1
//
// grad_sumsq_kernel walks every gradient in 16K-element chunks (the same
// chunking as the AdamW kernel, descriptors in kernel parameter space) and
// writes one fp32 sum of squares per chunk; clip_finalize_kernel adds the
// chunks in double in a fixed order, so the result does not depend on the
// launch shape.  The scale stays on the device: the AdamW and Muon kernels read
// it and multiply each gradient as they load it, so main_grad itself is never
// rewritten.

#include "internal.h"

namespace mpopt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int find_norm_tensor(const NormTensorDesc* t, int n, int64_t chunk) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t[mid].chunk_begin <= chunk) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads)
grad_sumsq_kernel(const __grid_constant__ NormBatch batch, float* partials) {
  __shared__ float warp_sums[kThreads / 32];
  for (int64_t chunk = blockIdx.x; chunk < batch.total_chunks; chunk += gridDim.x) {
    const NormTensorDesc d = batch.t[find_norm_tensor(batch.t, batch.n, chunk)];
    const int64_t begin = (chunk - d.chunk_begin) * kAdamwChunk;
    const int64_t n = min(kAdamwChunk, d.numel - begin);
    const float* g = d.g + begin;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    int64_t done = 0;
    if ((reinterpret_cast<uintptr_t>(g) & 15u) == 0) {
      const int64_t n4 = n / 4;
      for (int64_t j = threadIdx.x; j < n4; j += blockDim.x) {
        const float4 x = reinterpret_cast<const float4*>(g)[j];
        acc.x += x.x * x.x;
        acc.y += x.y * x.y;
        acc.z += x.z * x.z;
        acc.w += x.w * x.w;
      }
      done = 4 * n4;
    }
    for (int64_t j = done + threadIdx.x; j < n; j += blockDim.x) acc.x += g[j] * g[j];
    float ss = (acc.x + acc.y) + (acc.z + acc.w);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
      float t = 0.f;
      for (int w = 0; w < kThreads / 32; ++w) t += warp_sums[w];
      partials[batch.partial_offset + chunk] = t;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(1024)
clip_finalize_kernel(const float* partials, int64_t n, float max_norm, float* scale_out, float* norm_out,
                     float* user_scale, float* user_norm) {
  __shared__ double sh[1024];
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < n; i += blockDim.x) acc += static_cast<double>(partials[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double total = sqrt(sh[0]);
    double scale = 1.0;
    if (max_norm > 0.f) {
      const double coeff = static_cast<double>(max_norm) / (total + 1e-6);
      if (coeff < 1.0) scale = coeff;
    }
    *scale_out = static_cast<float>(scale);
    *norm_out = static_cast<float>(total);
    if (user_scale) *user_scale = static_cast<float>(scale);
    if (user_norm) *user_norm = static_cast<float>(total);
  }
}

}  // namespace

cudaError_t launch_grad_sumsq(const NormBatch& batch, float* partials, cudaStream_t stream) {
  if (batch.n <= 0 || batch.total_chunks <= 0) return cudaSuccess;
  // one CTA per chunk, in chunk order: a contiguous sweep of the tensors
  const int64_t grid = batch.total_chunks < 0x7fffffff ? batch.total_chunks : 0x7fffffff;
  grad_sumsq_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(batch, partials);
  return cudaGetLastError();
}

cudaError_t launch_clip_finalize(const float* partials, int64_t n_partials, float max_norm, float* scale_out,
                                 float* norm_out, float* user_scale, float* user_norm, cudaStream_t stream) {
  clip_finalize_kernel<<<1, 1024, 0, stream>>>(partials, n_partials, max_norm, scale_out, norm_out, user_scale,
                                               user_norm);
  return cudaGetLastError();
}

}  // namespace mpopt
