// Internal declarations shared by the host side of the C ABI (api.cu) and the
// kernels.  Not part of the public interface.
#pragma once

#include <cstddef>
#include <cstdint>
#include <vector>
#include <cuda_runtime.h>

namespace mpopt {

// ---------------------------------------------------------------- AdamW ----

// Elements per multi-tensor chunk.  A chunk is the unit of work a CTA takes.
constexpr int64_t kAdamwChunk = 16384;
constexpr int kAdamwThreads = 256;

// One tensor of the AdamW list, as the kernel sees it (device-resident table).
struct AdamwTensorDesc {
  float* p;
  const float* g;
  float* m;
  float* v;
  uint16_t* model;       // bf16 bits, or nullptr (fp32-native parameter)
  int64_t numel;
  int64_t chunk_begin;   // index of this tensor's first chunk in the launch
  int32_t head;          // scalar elements before the first 8-aligned group; -1: scalar only
  int32_t pad_;
};
static_assert(sizeof(AdamwTensorDesc) == 64, "descriptor layout");

// Per-step fp32 scalars, formed on the host in double and rounded once.
struct AdamwScalars {
  float lr, beta1, beta2, eps;
  float one_minus_beta1, one_minus_beta2;
  float bias_c1, bias_c2;   // 1 - beta^t
  float decay;              // 1 - lr * weight_decay
  int32_t pad_;
  const float* grad_scale;  // device scalar multiplying every gradient (clipping), or nullptr
};

// Descriptors travel in the kernel's parameter space (no upload, no workspace):
// up to kAdamwBatch tensors per launch.
constexpr int kAdamwBatch = 400;
struct AdamwBatch {
  AdamwScalars s;
  int32_t n;
  int32_t pad_;
  int64_t total_chunks;
  AdamwTensorDesc t[kAdamwBatch];
};
static_assert(sizeof(AdamwBatch) <= 32000, "kernel parameter space");

cudaError_t launch_adamw(const AdamwBatch& batch, cudaStream_t stream);

// ----------------------------------------------------------------- Muon ----

// Newton-Schulz works on padded, wide-oriented buffers: A = min(R, C) rows
// padded to Ap, B = max(R, C) columns padded to Bp, both multiples of kNsPad.
constexpr int64_t kNsPad = 256;
constexpr int kMaxGroup = 64;         // matrices per batched launch

// One Muon matrix of a batched group (kernel-parameter table).
// Matrices of one group share (A, B) = (min, max) of their shape but not
// necessarily the orientation: an R x C matrix with R > C is transposed into
// the wide orientation.
struct MuonMat {
  float* W;               // fp32 master [R x C]
  const float* g;         // fp32 gradient [R x C]
  float* m;               // fp32 momentum [R x C]
  uint16_t* Wb;           // bf16 model copy or nullptr
  float* O;               // opt_newton_schulz only: fp32 output [R x C], else nullptr
  int32_t R, C;           // this matrix's shape (W layout)
  int32_t transposed;     // R > C: the wide orientation is W^T
  int32_t vec4;           // g and m 16-byte aligned: vector path in the momentum pass
  float step_scale;       // lr * update scale of this matrix (scale mode, shape)
  int32_t pad_;
};

struct MuonGroup {
  int32_t count;          // matrices in this group
  int32_t pad_;
  int64_t A, B, Ap, Bp;   // A = min(R, C), B = max(R, C), padded
  MuonMat mats[kMaxGroup];
};

// Workspace buffers of one group (all device pointers into the workspace).
// Newton-Schulz operands are fp16 (kind::f16 tensor cores); accumulation fp32.
struct NsBuffers {
  uint16_t* Xh[2];   // fp16 iterate            [count][Ap][Bp], ping-pong
  uint16_t* Ah;      // fp16 Gram matrix        [count][Ap][Ap] (operand of A A and the b A term)
  uint16_t* Ch;      // fp16 a I + b A + c A A  [count][Ap][Ap]
  uint16_t* Th[2];   // two more fp16 [count][Ap][Ap] for grouped iterations, or nullptr
  float* partial;    // per-block sums of squares [count][max(norm blocks, prologue tiles)]
  // per matrix, [count] each:
  float* inv_norm;   // 1 / (||G||_F + eps)
  float* x_scale;    // power of two: the prologue writes fp16(gtilde * x_scale) as the iterate
  uint32_t* amax;    // bits of max |gtilde * x_scale| (non-negative floats order as integers)
  float* x0_scale;   // 1 / (x_scale (||G||_F + eps)), or 1 after a fix-up: X0 = x0_scale * iterate
  uint32_t* fix;     // 1: the iterate left fp16's normal range, the fix-up rewrites X0 normalised
  uint32_t* status;  // workspace header word
};
constexpr int kMatStats = 5;   // per-matrix words above, after the partial sums

struct MuonScalars {
  float mu, one_minus_mu;
  int nesterov;
  float eps;
  float a, b, c;
  float decay;        // 1 - lr * weight_decay
  int ns_steps;
  int ns_only;        // opt_newton_schulz: G is read from g, O written, no momentum/update
  int no_normalize;   // plain momentum SGD: the direction is gtilde itself
  const float* grad_scale;  // device scalar multiplying every gradient (clipping), or nullptr
  float sched[16][3]; // (a, b, c) of each iteration
  int stall_first_stage;    // self-test: withhold one TMA stage of the first X X^T launch
};

// Elementwise pass 1 (momentum, norm partials): fixed elements per block so the
// reduction order, and hence the result, does not depend on the launch.
constexpr int64_t kNormElemsPerBlock = 8192;
inline int64_t norm_blocks_per_matrix(const MuonGroup& g) {
  return (g.A * g.B + kNormElemsPerBlock - 1) / kNormElemsPerBlock;
}
// Prologue of the Newton-Schulz path: 64 x 64 tiles of the padded W-layout
// space, one partial sum of squares per tile.
constexpr int kPrepTile = 64;
inline int64_t operand_blocks_per_matrix(const MuonGroup& g) {
  return (g.Ap / kPrepTile) * (g.Bp / kPrepTile);
}
constexpr int64_t partials_per_matrix(int64_t A, int64_t B, int64_t Ap, int64_t Bp) {
  const int64_t blocks = (A * B + kNormElemsPerBlock - 1) / kNormElemsPerBlock;
  const int64_t tiles = (Ap / kPrepTile) * (Bp / kPrepTile);
  return blocks > tiles ? blocks : tiles;
}
// Samples per matrix that set x_scale: the largest sampled |gtilde| is mapped
// just below 2^kXScaleExp, leaving 2^(16 - kXScaleExp) of headroom below
// fp16's largest finite value for the elements the sample missed.
constexpr int kScaleSamples = 4096;
constexpr int kXScaleExp = 10;

// Path without Newton-Schulz (ns_steps = 0, momentum SGD): momentum pass with
// norm partials per 8192 elements, the norm, then the update.
cudaError_t launch_muon_momentum(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                                 cudaStream_t stream);
// Newton-Schulz path: the sample that sets x_scale, then the prologue (momentum,
// Nesterov, the fp16 iterate in the wide orientation, tile partial sums and
// the max), the norm (and x0_scale / fix), and the fix-up, which rewrites X0
// only for matrices whose iterate left fp16's normal range.
cudaError_t launch_muon_sample(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                               cudaStream_t stream);
cudaError_t launch_muon_prologue(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                                 cudaStream_t stream);
// ns_path: partials are the prologue's tiles, and x0_scale / fix are set too
cudaError_t launch_muon_norm(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, bool ns_path,
                             cudaStream_t stream);
cudaError_t launch_muon_fixup(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s,
                              cudaStream_t stream);
// ns_steps == 0: O = X0 (no tensor-core work); writes the update / output.
cudaError_t launch_muon_apply_direct(const MuonGroup& grp, const NsBuffers& buf,
                                     const MuonScalars& s, cudaStream_t stream);

// Tensor-core GEMM stages of one Newton-Schulz iteration.
enum NsGemmMode : int { kGram = 0, kPoly = 1, kBx = 2, kBxFinal = 3 };

// Grouped iterations.  Every C_k is a polynomial in the first Gram matrix of
// its group, so g consecutive iterations k0 .. k0+g-1 need only one X X^T and
// one C X: A_{k+1} = C_k (A_k C_k) and M = C_{k0+g-1} ... C_k0 are products of
// [Ap][Ap] symmetric matrices, and X_{k0+g} = M X_k0.  Each extra iteration
// trades one X X^T (A^2 B) and one C X (2 A^2 B) for four A^3 products, which
// pays when B is well above A.  Groups hold at most kNsMaxGroupIters
// iterations: the product M spans eigenvalues up to a^g, and its fp16
// rounding grows with that range.
constexpr int kNsMaxGroupIters = 3;
// Sizes of the groups of ns_steps iterations, in order: all 1 when not
// grouped, else ceil(ns_steps / 3) groups as equal as possible, the larger
// first (5 -> 3, 2).
std::vector<int> ns_group_sizes(int ns_steps, bool grouped);
// By default a shape class is grouped when padded B >= 2 padded A (a merged
// iteration then does at least a fifth less tensor-core work; 60 % less for
// 4096 x 14336) and A >= 1024 (smaller launches are bound by latency, and a
// group launches more of them).
inline bool ns_grouping_pays(int64_t Ap, int64_t Bp) { return Bp >= 2 * Ap && Ap >= 1024; }

// The GEMMs of iterations it0 .. it0+g-1 (g = 1: X X^T, the polynomial, C X);
// group_index selects the iterate buffer (the groups alternate between the two).
cudaError_t launch_ns_group(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, int it0, int g,
                            int group_index, cudaStream_t stream);

// Device-status codes written to the workspace header.
enum : uint32_t {
  kStatusOk = 0,
  kStatusTimeoutFull = 1,     // MMA waited too long for a TMA stage
  kStatusTimeoutEmpty = 2,    // producer waited too long for a free stage
  kStatusTimeoutAcc = 3,      // epilogue waited too long for an accumulator
  kStatusTimeoutAccFree = 4,  // MMA waited too long for a free accumulator
  kStatusTimeoutDrain = 5,
  kStatusTimeoutTile = 6,     // a role waited too long for the next tile index
  kStatusTimeoutWload = 7     // an epilogue warp waited too long for its block of W
};

// Workspace-header words (uint32 index) of the GEMM tile scheduler: the count
// of tiles claimed after each pair's first, and the count of CTAs that have
// finished.  The last CTA of a launch resets both, and each step clears the
// header before its first launch.
constexpr int kSchedWord = 32;

// ------------------------------------------------------------- clipping ----

// Global gradient norm: one fp32 partial sum of squares per 16K-element chunk
// of every gradient (Muon and AdamW alike), then one fp64 reduction.
constexpr int kNormBatch = 1200;
struct NormTensorDesc {
  const float* g;
  int64_t numel;
  int64_t chunk_begin;   // first chunk of this tensor within the launch
};
struct NormBatch {
  int32_t n;
  int32_t pad_;
  int64_t total_chunks;
  int64_t partial_offset;   // where this launch's chunks start in the partial buffer
  NormTensorDesc t[kNormBatch];
};
static_assert(sizeof(NormBatch) <= 32000, "kernel parameter space");

cudaError_t launch_grad_sumsq(const NormBatch& batch, float* partials, cudaStream_t stream);
// scale_out = max_norm / (sqrt(sum) + 1e-6) when that is below 1, else 1
// (1 as well when max_norm <= 0); norm_out = sqrt(sum); user_scale and
// user_norm (optional) receive copies.
cudaError_t launch_clip_finalize(const float* partials, int64_t n_partials, float max_norm, float* scale_out,
                                 float* norm_out, float* user_scale, float* user_norm, cudaStream_t stream);

// ------------------------------------------------------------ lifecycle ----

constexpr int kReloadBatch = 900;
struct ReloadDesc {
  const uint16_t* src;   // bf16 model parameter
  float* dst;            // fp32 main_param
  int64_t numel;
  int64_t chunk_begin;
};
struct ReloadBatch {
  int32_t n;
  int32_t pad_;
  int64_t total_chunks;
  ReloadDesc t[kReloadBatch];
};
static_assert(sizeof(ReloadBatch) <= 32000, "kernel parameter space");

cudaError_t launch_reload(const ReloadBatch& batch, cudaStream_t stream);

// Host-to-device copy of page-locked host memory by SM loads
// (opt_copy_from_host); src is the device-visible address of the host buffer.
cudaError_t launch_copy_from_host(void* dst, const void* src, size_t bytes, cudaStream_t stream);

int num_sms();   // SM count of the current device (cached per device)

// Launch instrumentation (opt_profile_launches).  A launch site calls
// prof_begin(kernel, count, a, b, stream) before and prof_end(stream) after
// its launch; both are no-ops while instrumentation is off.
void prof_begin(int kernel, int count, int64_t a, int64_t b, cudaStream_t stream);
void prof_end(cudaStream_t stream);

}  // namespace mpopt
