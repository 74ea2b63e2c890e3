// Muon elementwise stages for sm_103a: momentum and Nesterov lerps, the
// Frobenius norm, and the fp16 iterate that feeds the tensor-core
// Newton-Schulz GEMMs.
//
// Definitions ("02 · Optimizer：算法与 infra" §1, §5.2; "优化器：AdamW、Muon 与
// 分布式优化器", Muon section):
//   m      <- lerp(m, g, 1 - mu) = m + (1 - mu) (g - m)
//   gtilde  = lerp(g, m, mu)     = g + mu (m - g)           (Nesterov; else m)
//   X0      = gtilde / (||gtilde||_F + eps), transposed when rows > cols
//
// Newton-Schulz path, one pass over g and m:
//   muon_sample_kernel    a power of two x_scale per matrix from a strided
//                         sample of |gtilde|, mapping the sampled maximum just
//                         below 2^kXScaleExp;
//   muon_prologue_kernel  updates m in place and writes fp16(gtilde * x_scale)
//                         in the wide orientation (rows = min side) into the
//                         zero-padded workspace, with one sum of squares per
//                         64 x 64 tile and the matrix's max |gtilde * x_scale|;
//   muon_norm_kernel      1/(||gtilde||_F + eps) in double and
//                         x0_scale = 1/(x_scale (||gtilde||_F + eps)); the first
//                         X X^T and C X epilogues multiply by it (squared for
//                         X X^T), so X0 is never written normalised;
//   muon_fixup_kernel     for a matrix whose iterate left fp16's normal range
//                         (the sample missed an element more than 2^(16 -
//                         kXScaleExp) times its maximum, or every element is
//                         so small that fp16 would lose precision) rewrites X0
//                         normalised from g and the new m, and its x0_scale is
//                         1; for every other matrix it returns at once.
// Scaling by a power of two is exact, so fp16(gtilde * x_scale) carries
// gtilde to fp16's 11-bit precision, like the normalised value it stands for.
//
// Path without Newton-Schulz (ns_steps = 0, momentum SGD): muon_momentum_kernel
// (m and per-8192-element partial sums), muon_norm_kernel, then
// muon_apply_direct_kernel.

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

// grid: matrices; inv_norm[mat] = 1 / (sqrt(sum of partials) + eps), in
// double.  Newton-Schulz path: also x0_scale and the fix-up flag.  The
// iterate fp16(gtilde * x_scale) is fit for use when its max lies in
// [2^(kXScaleExp - 4), 65504]: then no element overflowed, and elements down to
// 2^-24 of the max stay normal numbers; a zero matrix needs nothing either.
__global__ void muon_norm_kernel(NsBuffers buf, int64_t blocks_per_mat, float eps, int ns_path) {
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
  if (threadIdx.x == 0) {
    const double inv = 1.0 / (sqrt(sh[0]) + static_cast<double>(eps));
    buf.inv_norm[mat] = static_cast<float>(inv);
    if (ns_path) {
      const float amax = __uint_as_float(buf.amax[mat]);   // NaN compares false: fix
      const bool fit = amax == 0.f || (amax >= static_cast<float>(1 << (kXScaleExp - 4)) && amax <= 65504.f);
      buf.fix[mat] = fit ? 0u : 1u;
      buf.x0_scale[mat] = fit ? static_cast<float>(inv / static_cast<double>(buf.x_scale[mat])) : 1.f;
    }
  }
}

// grid: matrices.  x_scale[mat] = 2^(kXScaleExp - e) where the largest sampled
// |gtilde| lies in [2^(e-1), 2^e); 1 when the sample is all zero or not
// finite.  Also clears the matrix's max for the prologue.
__global__ void __launch_bounds__(kThreads)
muon_sample_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ uint32_t warp_max[kThreads / 32];
  const int mat = blockIdx.x;
  const MuonMat& M = grp.mats[mat];
  const int64_t n = static_cast<int64_t>(M.R) * M.C;
  const int64_t ns = n < kScaleSamples ? n : kScaleSamples;
  const int64_t stride = n / ns;
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;
  uint32_t mx = 0;
  for (int64_t k = threadIdx.x; k < ns; k += kThreads) {
    const int64_t i = k * stride;
    const float g = M.g[i] * gs;
    float v = g;
    if (!s.ns_only) {
      const float m_old = M.m[i];
      v = gtilde(s, g, m_old + s.one_minus_mu * (g - m_old));
    }
    mx = max(mx, __float_as_uint(fabsf(v)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t t = 0;
    for (int w = 0; w < kThreads / 32; ++w) t = max(t, warp_max[w]);
    const float amax = __uint_as_float(t);
    float scale = 1.f;
    if (amax > 0.f && amax <= 3.0e38f) {
      int e = 0;
      frexpf(amax, &e);                      // amax in [2^(e-1), 2^e)
      int k = kXScaleExp - e;
      k = k < -120 ? -120 : (k > 120 ? 120 : k);
      scale = ldexpf(1.f, k);
    }
    buf.x_scale[mat] = scale;
    buf.amax[mat] = 0u;
  }
}

// grid: (tiles per matrix, matrices); one 64 x 64 tile of the padded W-layout
// space per block.  Each thread takes 4 consecutive elements of 4 rows: the
// momentum update in place (16-byte loads and stores of g and m when the rows
// are 16-byte aligned), gtilde, and the fp16 iterate fp16(gtilde * x_scale) in
// the wide layout [Ap][Bp] (through a shared-memory transpose when W is
// tall); elements outside R x C are written as zeros.  One sum of squares of
// gtilde per tile, in a fixed order; the matrix's max |gtilde * x_scale| by an
// atomic max on its bits.
__global__ void __launch_bounds__(kThreads)
muon_prologue_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ uint16_t tile[kPrepTile][kPrepTile + 2];   // odd word stride: few bank conflicts
  __shared__ float warp_sums[kThreads / 32];
  __shared__ uint32_t warp_max[kThreads / 32];
  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t Ap = grp.Ap, Bp = grp.Bp;
  const bool tr = M.transposed != 0;
  const int64_t wcols_p = tr ? Ap : Bp;                 // padded W-layout width
  const int64_t tiles_x = wcols_p / kPrepTile;
  const int64_t ty = blockIdx.x / tiles_x, tx = blockIdx.x % tiles_x;
  const int64_t r0 = ty * kPrepTile, c0 = tx * kPrepTile;
  const int R = M.R, C = M.C;
  const float xs = buf.x_scale[mat];
  const float gs = s.grad_scale ? *s.grad_scale : 1.f;   // clipping factor (1: none)
  const int lc = (threadIdx.x % 16) * 4;       // first of 4 columns
  const int lr0 = threadIdx.x / 16;            // 0..15
  const bool vec = M.vec4 && (C % 4 == 0);     // every row start 16-byte aligned
  uint16_t* Xh = buf.Xh[0] + static_cast<int64_t>(mat) * Ap * Bp;   // [Ap][Bp]
  float ss = 0.f;
  uint32_t mx = 0;
  // every 16-byte load of the tile first: a load of g or m cannot be moved
  // above a store to m, which the compiler must assume may alias it, so
  // loads interleaved with the stores would wait for each other
  float4 gq[kPrepTile / 16], mq[kPrepTile / 16];
#pragma unroll
  for (int k = 0; k < kPrepTile / 16; ++k) {
    const int64_t r = r0 + lr0 + 16 * k, c = c0 + lc;
    gq[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    mq[k] = gq[k];
    if (r < R && vec && c + 3 < C) {
      const int64_t i = r * C + c;
      gq[k] = *reinterpret_cast<const float4*>(M.g + i);
      if (!s.ns_only) mq[k] = *reinterpret_cast<const float4*>(M.m + i);
    }
  }
#pragma unroll
  for (int k = 0; k < kPrepTile / 16; ++k) {
    const int lr = lr0 + 16 * k;
    const int64_t r = r0 + lr, c = c0 + lc;
    float val[4] = {0.f, 0.f, 0.f, 0.f};
    if (r < R) {
      const int64_t i = r * C + c;
      if (vec && c + 3 < C) {
        float4 g = gq[k];
        g.x *= gs;
        g.y *= gs;
        g.z *= gs;
        g.w *= gs;
        if (s.ns_only) {
          val[0] = g.x;
          val[1] = g.y;
          val[2] = g.z;
          val[3] = g.w;
        } else {
          float4 m = mq[k];
          m.x = m.x + s.one_minus_mu * (g.x - m.x);
          m.y = m.y + s.one_minus_mu * (g.y - m.y);
          m.z = m.z + s.one_minus_mu * (g.z - m.z);
          m.w = m.w + s.one_minus_mu * (g.w - m.w);
          *reinterpret_cast<float4*>(M.m + i) = m;
          val[0] = gtilde(s, g.x, m.x);
          val[1] = gtilde(s, g.y, m.y);
          val[2] = gtilde(s, g.z, m.z);
          val[3] = gtilde(s, g.w, m.w);
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (c + q < C) {
            const float g = M.g[i + q] * gs;
            if (s.ns_only) {
              val[q] = g;
            } else {
              const float m_old = M.m[i + q];
              const float m = m_old + s.one_minus_mu * (g - m_old);
              M.m[i + q] = m;
              val[q] = gtilde(s, g, m);
            }
          }
        }
      }
    }
    uint16_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      ss += val[q] * val[q];
      const float x = val[q] * xs;
      mx = max(mx, __float_as_uint(fabsf(x)));
      h[q] = f16_bits(x);
    }
    if (tr) {
      tile[lr][lc + 0] = h[0];
      tile[lr][lc + 1] = h[1];
      tile[lr][lc + 2] = h[2];
      tile[lr][lc + 3] = h[3];
    } else {
      *reinterpret_cast<uint2*>(Xh + r * Bp + c) =
          make_uint2(static_cast<uint32_t>(h[0]) | (static_cast<uint32_t>(h[1]) << 16),
                     static_cast<uint32_t>(h[2]) | (static_cast<uint32_t>(h[3]) << 16));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    ss += __shfl_xor_sync(0xffffffffu, ss, off);
    mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if ((threadIdx.x & 31) == 0) {
    warp_sums[threadIdx.x >> 5] = ss;
    warp_max[threadIdx.x >> 5] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    uint32_t tm = 0;
    for (int w = 0; w < kThreads / 32; ++w) {
      t += warp_sums[w];
      tm = max(tm, warp_max[w]);
    }
    buf.partial[static_cast<int64_t>(mat) * gridDim.x + blockIdx.x] = t;
    if (tm) atomicMax(buf.amax + mat, tm);
  }
  if (!tr) return;   // uniform per block
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

// Fix-up.  grid: (up to kFixupBlocks, matrices); a block returns at once
// unless its matrix's iterate left fp16's normal range, and otherwise walks
// that matrix's 64 x 64 tiles of the padded W-layout space, rewriting X0 =
// fp16(gtilde / (||gtilde||_F + eps)) in the wide layout [Ap][Bp] from g and
// the updated m (the same arithmetic as the prologue, so the same gtilde):
// directly when W is wide, through a shared-memory transpose when W is tall.
// Each thread moves 4 consecutive elements per step: a 16-byte load of g and
// of m (when the rows are 16-byte aligned, else four scalar loads) and an
// 8-byte store of 4 fp16.
constexpr int kFixupBlocks = 64;

__global__ void __launch_bounds__(kThreads)
muon_fixup_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ uint16_t tile[kPrepTile][kPrepTile + 2];   // odd word stride: few bank conflicts
  const int mat = blockIdx.y;
  if (buf.fix[mat] == 0u) return;   // uniform per block
  const MuonMat& M = grp.mats[mat];
  const int64_t Ap = grp.Ap, Bp = grp.Bp;
  const bool tr = M.transposed != 0;
  const int64_t wcols_p = tr ? Ap : Bp;                 // padded W-layout width
  const int64_t tiles_x = wcols_p / kPrepTile;
  const int64_t n_tiles = (Ap / kPrepTile) * (Bp / kPrepTile);
  for (int64_t tile_id = blockIdx.x; tile_id < n_tiles; tile_id += gridDim.x) {
    __syncthreads();   // the previous tile's transpose has been read
    const int64_t ty = tile_id / tiles_x, tx = tile_id % tiles_x;
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
    if (!tr) continue;   // uniform per block
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

cudaError_t launch_muon_norm(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, bool ns_path,
                             cudaStream_t stream) {
  const int64_t blocks = ns_path ? operand_blocks_per_matrix(grp) : norm_blocks_per_matrix(grp);
  muon_norm_kernel<<<grp.count, 256, 0, stream>>>(buf, blocks, s.eps, ns_path ? 1 : 0);
  return cudaGetLastError();
}

cudaError_t launch_muon_sample(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                               cudaStream_t stream) {
  muon_sample_kernel<<<grp.count, kThreads, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

cudaError_t launch_muon_prologue(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                                 cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(operand_blocks_per_matrix(grp)), static_cast<unsigned>(grp.count));
  muon_prologue_kernel<<<grid, kThreads, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

cudaError_t launch_muon_fixup(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                              cudaStream_t stream) {
  const int64_t tiles = operand_blocks_per_matrix(grp);
  dim3 grid(static_cast<unsigned>(tiles < kFixupBlocks ? tiles : kFixupBlocks), static_cast<unsigned>(grp.count));
  muon_fixup_kernel<<<grid, kThreads, 0, stream>>>(grp, buf, s);
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
