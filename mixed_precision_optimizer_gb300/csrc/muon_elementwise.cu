// Muon elementwise stages for sm_103a: momentum and Nesterov lerps, the
// Frobenius norm, and the fp16 operand copies that feed the tensor-core
// Newton-Schulz GEMMs.
//
// Definitions ("02 · Optimizer：算法与 infra" §1, §5.2; "优化器：AdamW、Muon 与
// 分布式优化器", Muon section):
//   m      <- lerp(m, g, 1 - mu) = m + (1 - mu) (g - m)
//   gtilde  = lerp(g, m, mu)     = g + mu (m - g)           (Nesterov; else m)
//   X0      = gtilde / (||gtilde||_F + eps), transposed when rows > cols
//
// Pass 1 (muon_momentum_kernel) updates m in place and writes per-block sums
// of gtilde^2 in a fixed order; muon_norm_kernel reduces them in double to
// 1/(||gtilde||_F + eps).  Pass 2 (muon_operand_kernel) recomputes gtilde from
// g and the new m (the same arithmetic, so the same values), scales it, and
// writes the fp16 operand X0 in the wide orientation (rows = min side) into the
// zero-padded workspace; both X X^T and C X read that one copy.
// Normalising before the fp16 conversion keeps every operand in [-1.3, 1.3].

#include <cuda_fp16.h>

#include "internal.h"

namespace mpopt {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ uint16_t f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  return static_cast<uint16_t>((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

// gtilde from g and the already-updated momentum m (or G itself for ns_only).
__device__ __forceinline__ float gtilde(const MuonScalars& s, float g, float m_new) {
  if (s.ns_only) return g;
  return s.nesterov ? g + s.mu * (m_new - g) : m_new;
}

// grid: (norm blocks per matrix, matrices).  Each block owns elements
// [blk * 8192, blk * 8192 + 8192) of its matrix in W layout.
__global__ void __launch_bounds__(kThreads)
muon_momentum_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ float warp_sums[kThreads / 32];
  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t n = static_cast<int64_t>(M.R) * M.C;
  const int64_t base = static_cast<int64_t>(blockIdx.x) * kNormElemsPerBlock;
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;   // clipping factor (1: none)
  float ss = 0.f;
  if (M.vec4 && base + kNormElemsPerBlock <= n) {   // 16-byte aligned, full block: float4 path
    const float4* g4 = reinterpret_cast<const float4*>(M.g + base);
    float4* m4 = reinterpret_cast<float4*>(M.m + base);
#pragma unroll 4
    for (int k = 0; k < kNormElemsPerBlock / 4 / kThreads; ++k) {
      const int j = k * kThreads + threadIdx.x;
      float4 g = g4[j];
      g.x *= gs;
      g.y *= gs;
      g.z *= gs;
      g.w *= gs;
      float4 v;
      if (s.ns_only) {
        v = g;
      } else {
        float4 m = m4[j];
        m.x = m.x + s.one_minus_mu * (g.x - m.x);
        m.y = m.y + s.one_minus_mu * (g.y - m.y);
        m.z = m.z + s.one_minus_mu * (g.z - m.z);
        m.w = m.w + s.one_minus_mu * (g.w - m.w);
        m4[j] = m;
        v = make_float4(gtilde(s, g.x, m.x), gtilde(s, g.y, m.y), gtilde(s, g.z, m.z), gtilde(s, g.w, m.w));
      }
      ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
    }
  } else {
    for (int k = 0; k < kNormElemsPerBlock / kThreads; ++k) {
      const int64_t i = base + k * kThreads + threadIdx.x;
      if (i >= n) break;
      const float g = M.g[i] * gs;
      float v;
      if (s.ns_only) {
        v = g;
      } else {
        const float m_old = M.m[i];
        const float m = m_old + s.one_minus_mu * (g - m_old);
        M.m[i] = m;
        v = gtilde(s, g, m);
      }
      ss += v * v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) t += warp_sums[w];
    buf.partial[static_cast<int64_t>(mat) * gridDim.x + blockIdx.x] = t;
  }
}

// grid: matrices; inv_norm[mat] = 1 / (sqrt(sum of partials) + eps), in double.
__global__ void muon_norm_kernel(NsBuffers buf, int64_t blocks_per_mat, float eps) {
  __shared__ double sh[256];
  const int mat = blockIdx.x;
  const float* p = buf.partial + mat * blocks_per_mat;
  double acc = 0.0;
  for (int64_t i = threadIdx.x; i < blocks_per_mat; i += blockDim.x) acc += static_cast<double>(p[i]);
  sh[threadIdx.x] = acc;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) sh[threadIdx.x] += sh[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) buf.inv_norm[mat] = static_cast<float>(1.0 / (sqrt(sh[0]) + static_cast<double>(eps)));
}

// grid: (operand tiles per matrix, matrices); one 64 x 64 tile of the padded
// W-layout space per block.  Writes the fp16 operand X0 in the wide layout
// [Ap][Bp]: directly when W is wide, through a shared-memory transpose when W
// is tall (stored as the transpose of the wide layout).  Each thread moves 4
// consecutive elements per step: a 16-byte load of g and of m (when the rows
// are 16-byte aligned, else four scalar loads) and an 8-byte store of 4 fp16.
__global__ void __launch_bounds__(kThreads)
muon_operand_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ uint16_t tile[kPrepTile][kPrepTile + 2];   // odd word stride: few bank conflicts
  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t Ap = grp.Ap, Bp = grp.Bp;
  const bool tr = M.transposed != 0;
  const int64_t wcols_p = tr ? Ap : Bp;                 // padded W-layout width
  const int64_t tiles_x = wcols_p / kPrepTile;
  const int64_t ty = blockIdx.x / tiles_x, tx = blockIdx.x % tiles_x;
  const int64_t r0 = ty * kPrepTile, c0 = tx * kPrepTile;
  const int R = M.R, C = M.C;
  const float inv = buf.inv_norm[mat];
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;   // clipping factor (1: none)
  const int lc = (threadIdx.x % 16) * 4;       // first of 4 columns
  const int lr0 = threadIdx.x / 16;            // 0..15
  const bool vec = M.vec4 && (C % 4 == 0);     // every row start 16-byte aligned
  uint16_t* Xh = buf.Xh[0] + static_cast<int64_t>(mat) * Ap * Bp;   // [Ap][Bp]
#pragma unroll
  for (int k = 0; k < kPrepTile / 16; ++k) {
    const int lr = lr0 + 16 * k;
    const int64_t r = r0 + lr, c = c0 + lc;
    float val[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < R) {
      const int64_t i = r * C + c;
      if (vec && c + 3 < C) {
        const float4 g = *reinterpret_cast<const float4*>(M.g + i);
        float4 m = make_float4(0.f, 0.f, 0.f, 0.f);
        if (!s.ns_only) m = *reinterpret_cast<const float4*>(M.m + i);
        val[0] = gtilde(s, g.x * gs, m.x) * inv;
        val[1] = gtilde(s, g.y * gs, m.y) * inv;
        val[2] = gtilde(s, g.z * gs, m.z) * inv;
        val[3] = gtilde(s, g.w * gs, m.w) * inv;
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q)
          if (c + q < C) val[q] = gtilde(s, M.g[i + q] * gs, s.ns_only ? 0.f : M.m[i + q]) * inv;
      }
    }
    const uint16_t h0 = f16_bits(val[0]), h1 = f16_bits(val[1]), h2 = f16_bits(val[2]), h3 = f16_bits(val[3]);
    if (tr) {
      tile[lr][lc + 0] = h0;
      tile[lr][lc + 1] = h1;
      tile[lr][lc + 2] = h2;
      tile[lr][lc + 3] = h3;
    } else {
      *reinterpret_cast<uint2*>(Xh + r * Bp + c) =
          make_uint2(static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16),
                     static_cast<uint32_t>(h2) | (static_cast<uint32_t>(h3) << 16));
    }
  }
  if (!tr) return;   // uniform per block
  __syncthreads();
  // tall W: wide row i (= W column c0 + i) gets W rows r0 .. r0 + 63
#pragma unroll
  for (int k = 0; k < kPrepTile / 16; ++k) {
    const int i = lr0 + 16 * k;
    const int j = lc;
    const uint2 packed = make_uint2(static_cast<uint32_t>(tile[j][i]) | (static_cast<uint32_t>(tile[j + 1][i]) << 16),
                                    static_cast<uint32_t>(tile[j + 2][i]) | (static_cast<uint32_t>(tile[j + 3][i]) << 16));
    *reinterpret_cast<uint2*>(Xh + (c0 + i) * Bp + r0 + j) = packed;
  }
}

// ns_steps == 0: O = X0 = gtilde * inv_norm (plain momentum SGD: O = gtilde);
// apply the update (or write O).
__global__ void muon_apply_direct_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t n = static_cast<int64_t>(M.R) * M.C;
  const float inv = buf.inv_norm[mat];
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float o = gtilde(s, M.g[i] * gs, s.ns_only ? 0.f : M.m[i]) * (s.no_normalize ? 1.f : inv);
    if (s.ns_only) {
      M.O[i] = o;
    } else {
      const float w = M.W[i] * s.decay - M.step_scale * o;
      M.W[i] = w;
      if (M.Wb) M.Wb[i] = bf16_rne(w);
    }
  }
}

}  // namespace

cudaError_t launch_muon_momentum(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                                 cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(norm_blocks_per_matrix(grp)), static_cast<unsigned>(grp.count));
  muon_momentum_kernel<<<grid, kThreads, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

cudaError_t launch_muon_norm(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                             cudaStream_t stream) {
  muon_norm_kernel<<<grp.count, 256, 0, stream>>>(buf, norm_blocks_per_matrix(grp), s.eps);
  return cudaGetLastError();
}

cudaError_t launch_muon_operands(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                                 cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(operand_blocks_per_matrix(grp)), static_cast<unsigned>(grp.count));
  muon_operand_kernel<<<grid, kThreads, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

cudaError_t launch_muon_apply_direct(const MuonGroup& grp, const NsBuffers& buf,
                                     const MuonScalars& s, cudaStream_t stream) {
  const int64_t n = grp.A * grp.B;
  int64_t blocks = (n + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(grp.count));
  muon_apply_direct_kernel<<<grid, 256, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

}  // namespace mpopt
