// Muon elementwise stages for sm_103a: momentum and Nesterov lerps, the sum of
// squares for the Frobenius norm, and the bf16 operand copies that feed the
// tensor-core Newton-Schulz GEMMs.
//
// Definitions ("02 · Optimizer：算法与 infra" §1, §5.2; "优化器：AdamW、Muon 与
// 分布式优化器", Muon section):
//   m      <- lerp(m, g, 1 - mu) = m + (1 - mu) (g - m)
//   gtilde  = lerp(g, m, mu)     = g + mu (m - g)           (Nesterov; else m)
//   X0      = gtilde / (||gtilde||_F + eps), transposed when rows > cols
//
// The normalisation is not applied here: the prep pass writes gtilde itself
// (fp32 master copy, bf16 copy, bf16 transposed copy) into the padded,
// wide-oriented workspace buffers together with per-block sums of squares; a
// second tiny kernel turns those into 1/(||gtilde||_F + eps), which the first
// Newton-Schulz GEMMs fold into their epilogues.  One pass over g and m
// therefore does the whole elementwise part.

#include "internal.h"

namespace mpopt {
namespace {

constexpr int kPrepThreads = 256;

__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  return static_cast<uint16_t>((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

// grid: (prep tiles per matrix, matrices); block: 256 threads; one 64 x 64 tile
// of the padded W-layout space per block.
__global__ void __launch_bounds__(kPrepThreads)
muon_prep_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  __shared__ float tile[kPrepTile][kPrepTile + 1];
  __shared__ float warp_sums[kPrepThreads / 32];

  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t Ap = grp.Ap, Bp = grp.Bp;
  const bool tr = M.transposed != 0;
  // padded W-layout extents
  const int64_t wcols_p = tr ? Ap : Bp;
  const int64_t tiles_x = wcols_p / kPrepTile;
  const int64_t ty = blockIdx.x / tiles_x, tx = blockIdx.x % tiles_x;
  const int64_t r0 = ty * kPrepTile, c0 = tx * kPrepTile;
  const int R = M.R, C = M.C;

  const int lc = threadIdx.x % kPrepTile;       // column within the tile
  const int lr0 = threadIdx.x / kPrepTile;      // first row (0..3)
  float* X = buf.X + static_cast<int64_t>(mat) * Ap * Bp;
  uint16_t* Xb = buf.Xb + static_cast<int64_t>(mat) * Ap * Bp;
  uint16_t* Xt = buf.Xt[0] + static_cast<int64_t>(mat) * Ap * Bp;

  float ss = 0.f;
  #pragma unroll 4
  for (int k = 0; k < kPrepTile / 4; ++k) {
    const int lr = lr0 + 4 * k;
    const int64_t r = r0 + lr, c = c0 + lc;
    float val = 0.f;
    if (r < R && c < C) {
      const int64_t i = r * C + c;
      const float g = M.g[i];
      if (s.ns_only) {
        val = g;
      } else {
        const float m = M.m[i];
        const float mn = m + s.one_minus_mu * (g - m);
        M.m[i] = mn;
        val = s.nesterov ? g + s.mu * (mn - g) : mn;
      }
    }
    ss += val * val;
    tile[lr][lc] = val;
    // W-layout outputs: X (not transposed) or Xt (transposed)
    if (!tr) {
      X[r * Bp + c] = val;
      Xb[r * Bp + c] = bf16_rne(val);
    } else {
      Xt[r * Ap + c] = bf16_rne(val);
    }
  }
  __syncthreads();
  // transposed outputs: element (W row r, W col c) goes to row c, column r
  #pragma unroll 4
  for (int k = 0; k < kPrepTile / 4; ++k) {
    const int i = lr0 + 4 * k;                   // output row within tile (= W col)
    const int j = lc;                            // output col within tile (= W row)
    const float val = tile[j][i];
    const int64_t orow = c0 + i, ocol = r0 + j;
    if (!tr) {
      Xt[orow * Ap + ocol] = bf16_rne(val);
    } else {
      X[orow * Bp + ocol] = val;
      Xb[orow * Bp + ocol] = bf16_rne(val);
    }
  }
  // block sum of squares, fixed order (deterministic)
  #pragma unroll
  for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
  if ((threadIdx.x & 31) == 0) warp_sums[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.f;
    for (int w = 0; w < kPrepThreads / 32; ++w) t += warp_sums[w];
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

// ns_steps == 0: O = X0 = gtilde * inv_norm; apply the update (or write O).
__global__ void muon_apply_direct_kernel(const MuonGroup grp, NsBuffers buf, MuonScalars s) {
  const int mat = blockIdx.y;
  const MuonMat& M = grp.mats[mat];
  const int64_t n = static_cast<int64_t>(M.R) * M.C;
  const float inv = buf.inv_norm[mat];
  const float* X = buf.X + static_cast<int64_t>(mat) * grp.Ap * grp.Bp;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = i / M.C, c = i % M.C;
    const float x = M.transposed ? X[c * grp.Bp + r] : X[r * grp.Bp + c];
    const float o = x * inv;
    if (s.ns_only) {
      M.O[i] = o;
    } else {
      const float w = M.W[i] * s.decay - s.step_scale * o;
      M.W[i] = w;
      if (M.Wb) M.Wb[i] = bf16_rne(w);
    }
  }
}

}  // namespace

cudaError_t launch_muon_prep(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                             cudaStream_t stream) {
  const int64_t blocks = prep_blocks_per_matrix(grp);
  dim3 grid(static_cast<unsigned>(blocks), static_cast<unsigned>(grp.count));
  muon_prep_kernel<<<grid, kPrepThreads, 0, stream>>>(grp, buf, s);
  return cudaGetLastError();
}

cudaError_t launch_muon_norm(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                             cudaStream_t stream) {
  muon_norm_kernel<<<grp.count, 256, 0, stream>>>(buf, prep_blocks_per_matrix(grp), s.eps);
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
