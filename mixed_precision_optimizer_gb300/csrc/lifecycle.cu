// Master-weight lifecycle: main_param <- fp32(model_param) for every
// low-precision parameter ("02 · Optimizer：算法与 infra" §9.2:
// reload_model_params refreshes the fp32 masters after the model copy was
// changed from outside; "支持FP32优化器" §9.3-§9.4: the plain-checkpoint and
// model-only restore branches rebuild main_param this way).  bf16 -> fp32 is
// exact (the bf16 pattern with 16 zero bits appended).  Multi-tensor, one
// launch per 900 tensors, descriptors in kernel parameter space.

#include "internal.h"

namespace mpopt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ int find_reload_tensor(const ReloadDesc* t, int n, int64_t chunk) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t[mid].chunk_begin <= chunk) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads) reload_kernel(const __grid_constant__ ReloadBatch batch) {
  for (int64_t chunk = blockIdx.x; chunk < batch.total_chunks; chunk += gridDim.x) {
    const ReloadDesc d = batch.t[find_reload_tensor(batch.t, batch.n, chunk)];
    const int64_t begin = (chunk - d.chunk_begin) * kAdamwChunk;
    const int64_t end = min(begin + kAdamwChunk, d.numel);
    for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x)
      d.dst[i] = __uint_as_float(static_cast<uint32_t>(d.src[i]) << 16);
  }
}

}  // namespace

cudaError_t launch_reload(const ReloadBatch& batch, cudaStream_t stream) {
  if (batch.n <= 0 || batch.total_chunks <= 0) return cudaSuccess;
  // one CTA per chunk, in chunk order: a contiguous sweep of the tensors
  const int64_t grid = batch.total_chunks < 0x7fffffff ? batch.total_chunks : 0x7fffffff;
  reload_kernel<<<static_cast<unsigned>(grid), kThreads, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace mpopt
