// Multi-tensor AdamW for sm_103a: one launch updates every tensor of the list
// in a single HBM pass (read p, g, m, v; write p, m, v and the bf16 copy).
//
// Definition: "02 · Optimizer：算法与 infra" §2 (Adam, bias correction, eps
// outside the square root) and §3 (AdamW, decoupled weight decay), with the
// bf16 writeback of §9.2.  Per element, in fp32, every operation rounded to
// nearest and no contraction into FMA (the __f*_rn intrinsics):
//
//   g = main_grad * clip_scale         (clip_scale = 1 without clipping)
//   m = beta1*m + (1-beta1)*g          v = beta2*v + (1-beta2)*(g*g)
//   mhat = m / (1-beta1^t)             vhat = v / (1-beta2^t)
//   p = p*(1 - lr*lambda) - lr * (mhat / (sqrt(vhat) + eps))
//   model = bf16_rne(p)
//
// Work decomposition: every tensor is cut into 16K-element chunks; the grid
// has one CTA per chunk of the launch, and each CTA finds its chunk's tensor
// by binary search in the descriptor table, which is passed in the kernel's
// parameter space (up to 400 tensors per launch; longer lists take several
// launches).  Inside
// a chunk each warp takes 256 consecutive elements at a time: lane l the
// float4s l and 32 + l of every array, so that each of the warp's loads of
// p, g, m, v and streaming stores of p, m, v covers 512 contiguous bytes (two
// adjacent float4s a lane left every 32-byte sector half used by each
// instruction), and each 8-byte store of the bf16 copy 256.  Groups of 8
// after the last whole warp block take 8 consecutive elements a thread;
// elements before the first 16-byte-aligned group (views with an offset) and
// after the last full group take the same arithmetic one at a time.

#include "internal.h"

namespace mpopt {
namespace {

__device__ __forceinline__ void adamw_elem(float& p, float g, float& m, float& v,
                                           const AdamwScalars& s) {
  m = __fadd_rn(__fmul_rn(s.beta1, m), __fmul_rn(s.one_minus_beta1, g));
  v = __fadd_rn(__fmul_rn(s.beta2, v), __fmul_rn(s.one_minus_beta2, __fmul_rn(g, g)));
  const float mhat = __fdiv_rn(m, s.bias_c1);
  const float vhat = __fdiv_rn(v, s.bias_c2);
  const float den = __fadd_rn(__fsqrt_rn(vhat), s.eps);
  const float upd = __fdiv_rn(mhat, den);
  p = __fsub_rn(__fmul_rn(p, s.decay), __fmul_rn(s.lr, upd));
}

// fp32 -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FC0.
// Adding 0x7FFF plus the lowest kept bit to the pattern carries into the kept
// half exactly when the dropped half is above one half, or exactly one half
// with an odd kept half.  A carry out of the mantissa bumps the exponent, so
// the largest finite values round to infinity.
__device__ __forceinline__ uint32_t bf16_bits_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
}

__device__ __forceinline__ float4 ld_stream(const float* ptr) {
  float4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w) : "l"(ptr));
  return r;
}

__device__ __forceinline__ float4 ld_v4(const float* ptr) {
  return *reinterpret_cast<const float4*>(ptr);
}

// Streaming (evict-first) stores: nothing written here is read again within
// the step.
__device__ __forceinline__ void st_v4(float* ptr, const float4& v) {
  asm volatile("st.global.cs.v4.f32 [%0], {%1,%2,%3,%4};" ::"l"(ptr), "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_u2(void* ptr, uint32_t x, uint32_t y) {
  asm volatile("st.global.cs.v2.u32 [%0], {%1,%2};" ::"l"(ptr), "r"(x), "r"(y) : "memory");
}

__device__ __forceinline__ int find_tensor(const AdamwTensorDesc* t, int n, int64_t chunk) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {            // last tensor whose chunk_begin <= chunk
    const int mid = (lo + hi + 1) >> 1;
    if (t[mid].chunk_begin <= chunk) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void scalar_range(const AdamwTensorDesc& d, int64_t begin, int64_t end,
                                             const AdamwScalars& s, float gs) {
  for (int64_t i = begin + threadIdx.x; i < end; i += blockDim.x) {
    float p = d.p[i], m = d.m[i], v = d.v[i];
    adamw_elem(p, __fmul_rn(d.g[i], gs), m, v, s);
    d.p[i] = p;
    d.m[i] = m;
    d.v[i] = v;
    if (d.model) d.model[i] = static_cast<uint16_t>(bf16_bits_rne(p));
  }
}

__global__ void __launch_bounds__(kAdamwThreads, 4)
adamw_mta_kernel(const __grid_constant__ AdamwBatch batch) {
  const AdamwScalars& s = batch.s;
  // clipping factor (exactly 1 without clipping, so g * gs == g)
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;
  for (int64_t chunk = blockIdx.x; chunk < batch.total_chunks; chunk += gridDim.x) {
    const int ti = find_tensor(batch.t, batch.n, chunk);
    const AdamwTensorDesc d = batch.t[ti];
    const int64_t c = chunk - d.chunk_begin;
    if (d.head < 0) {          // pointers cannot be co-aligned: element at a time
      const int64_t b = c * kAdamwChunk;
      scalar_range(d, b, min(b + kAdamwChunk, d.numel), s, gs);
      continue;
    }
    const int64_t head = d.head;
    const int64_t begin = head + c * kAdamwChunk;
    const int64_t end = min(begin + kAdamwChunk, d.numel);
    if (c == 0) scalar_range(d, 0, head, s, gs);
    const int64_t ngroups = (end > begin) ? (end - begin) / 8 : 0;
    // A warp takes 256 consecutive elements (32 groups of 8): lane l the
    // float4s l and 32 + l, so that every load and store instruction of the
    // warp covers 512 contiguous bytes (256 for the bf16 copy).
    const int lane = threadIdx.x & 31;
    const int64_t nwarp_blocks = ngroups / 32;
    for (int64_t wb = threadIdx.x >> 5; wb < nwarp_blocks; wb += blockDim.x >> 5) {
      const int64_t e = begin + 256 * wb + 4 * lane, e1 = e + 128;
      float4 p0 = ld_v4(d.p + e), p1 = ld_v4(d.p + e1);
      float4 g0 = ld_stream(d.g + e), g1 = ld_stream(d.g + e1);
      g0.x = __fmul_rn(g0.x, gs); g0.y = __fmul_rn(g0.y, gs); g0.z = __fmul_rn(g0.z, gs); g0.w = __fmul_rn(g0.w, gs);
      g1.x = __fmul_rn(g1.x, gs); g1.y = __fmul_rn(g1.y, gs); g1.z = __fmul_rn(g1.z, gs); g1.w = __fmul_rn(g1.w, gs);
      float4 m0 = ld_v4(d.m + e), m1 = ld_v4(d.m + e1);
      float4 v0 = ld_v4(d.v + e), v1 = ld_v4(d.v + e1);
      adamw_elem(p0.x, g0.x, m0.x, v0.x, s);
      adamw_elem(p0.y, g0.y, m0.y, v0.y, s);
      adamw_elem(p0.z, g0.z, m0.z, v0.z, s);
      adamw_elem(p0.w, g0.w, m0.w, v0.w, s);
      adamw_elem(p1.x, g1.x, m1.x, v1.x, s);
      adamw_elem(p1.y, g1.y, m1.y, v1.y, s);
      adamw_elem(p1.z, g1.z, m1.z, v1.z, s);
      adamw_elem(p1.w, g1.w, m1.w, v1.w, s);
      st_v4(d.p + e, p0);
      st_v4(d.p + e1, p1);
      st_v4(d.m + e, m0);
      st_v4(d.m + e1, m1);
      st_v4(d.v + e, v0);
      st_v4(d.v + e1, v1);
      if (d.model) {
        st_u2(d.model + e, bf16_bits_rne(p0.x) | (bf16_bits_rne(p0.y) << 16),
              bf16_bits_rne(p0.z) | (bf16_bits_rne(p0.w) << 16));
        st_u2(d.model + e1, bf16_bits_rne(p1.x) | (bf16_bits_rne(p1.y) << 16),
              bf16_bits_rne(p1.z) | (bf16_bits_rne(p1.w) << 16));
      }
    }
    // groups after the last whole warp block: 8 consecutive elements a thread
    for (int64_t j = 32 * nwarp_blocks + threadIdx.x; j < ngroups; j += blockDim.x) {
      const int64_t e = begin + 8 * j;
      float4 p0 = ld_v4(d.p + e), p1 = ld_v4(d.p + e + 4);
      float4 g0 = ld_stream(d.g + e), g1 = ld_stream(d.g + e + 4);
      g0.x = __fmul_rn(g0.x, gs); g0.y = __fmul_rn(g0.y, gs); g0.z = __fmul_rn(g0.z, gs); g0.w = __fmul_rn(g0.w, gs);
      g1.x = __fmul_rn(g1.x, gs); g1.y = __fmul_rn(g1.y, gs); g1.z = __fmul_rn(g1.z, gs); g1.w = __fmul_rn(g1.w, gs);
      float4 m0 = ld_v4(d.m + e), m1 = ld_v4(d.m + e + 4);
      float4 v0 = ld_v4(d.v + e), v1 = ld_v4(d.v + e + 4);
      adamw_elem(p0.x, g0.x, m0.x, v0.x, s);
      adamw_elem(p0.y, g0.y, m0.y, v0.y, s);
      adamw_elem(p0.z, g0.z, m0.z, v0.z, s);
      adamw_elem(p0.w, g0.w, m0.w, v0.w, s);
      adamw_elem(p1.x, g1.x, m1.x, v1.x, s);
      adamw_elem(p1.y, g1.y, m1.y, v1.y, s);
      adamw_elem(p1.z, g1.z, m1.z, v1.z, s);
      adamw_elem(p1.w, g1.w, m1.w, v1.w, s);
      st_v4(d.p + e, p0);
      st_v4(d.p + e + 4, p1);
      st_v4(d.m + e, m0);
      st_v4(d.m + e + 4, m1);
      st_v4(d.v + e, v0);
      st_v4(d.v + e + 4, v1);
      if (d.model) {
        st_u2(d.model + e, bf16_bits_rne(p0.x) | (bf16_bits_rne(p0.y) << 16),
              bf16_bits_rne(p0.z) | (bf16_bits_rne(p0.w) << 16));
        st_u2(d.model + e + 4, bf16_bits_rne(p1.x) | (bf16_bits_rne(p1.y) << 16),
              bf16_bits_rne(p1.z) | (bf16_bits_rne(p1.w) << 16));
      }
    }
    // ragged tail of the tensor (only the last chunk has one)
    if (end == d.numel) scalar_range(d, begin + 8 * ngroups, end, s, gs);
  }
}

}  // namespace

cudaError_t launch_adamw(const AdamwBatch& batch, cudaStream_t stream) {
  if (batch.n <= 0 || batch.total_chunks <= 0) return cudaSuccess;
  // one CTA per chunk, launched in chunk order: the chunks in flight at any
  // moment are one contiguous sweep of the tensors (measured on GB300 over
  // 1.05e9 parameters: 6.94 TB/s, against 6.37 TB/s for a persistent grid of
  // twice the resident CTAs striding over the chunks)
  const int64_t grid = batch.total_chunks < 0x7fffffff ? batch.total_chunks : 0x7fffffff;
  adamw_mta_kernel<<<static_cast<unsigned>(grid), kAdamwThreads, 0, stream>>>(batch);
  return cudaGetLastError();
}

}  // namespace mpopt
