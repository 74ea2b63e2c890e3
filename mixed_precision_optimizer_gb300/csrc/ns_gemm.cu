// Newton-Schulz GEMMs on the 5th-generation tensor cores (sm_103a).
//
// One quintic iteration ("02 · Optimizer：算法与 infra" §5.2; "优化器：AdamW、
// Muon 与分布式优化器", newton_schulz in the Muon section) on the wide iterate
// X (A x B, A <= B), X' = a X + (b A + c A A) X with A = X X^T, is computed as
// three GEMMs with fused epilogues, all fp16 x fp16 -> fp32 (TMEM):
//
//   gram : A = X X^T                        -> A fp16 in full (each block below the
//                                              diagonal also stored as its mirror)
//   poly : C = a I + b A + c (A A)          -> C fp16 (b A from the same fp16 A that
//                                              feeds A A, so the polynomial is
//                                              evaluated at one rounded matrix)
//   bx   : X' = C X                         -> X' fp16 (next iterate; C X reads X
//                                              itself as an MN-major B operand)
//          (last iteration: W <- W (1 - lr*lambda) - lr*0.2*sqrt(max(A,B)) * X',
//           from the fp32 accumulator, in W's own orientation, with its bf16 copy)
//
// Number formats: folding a I into C keeps the large cancelling terms a X and
// B X (|a| = 3.44, B ~ -2.74 near unit singular values) inside one rounded
// operand, and fp16 operands (11-bit significands, values normalised into
// [-1.3, 1.3] before the first conversion) keep the rounding of C and X well
// below the tolerance; both run at the same tensor-core rate as bf16.
//
// Kernel structure: CTA pairs (clusters of 2, one CTA per SM), persistent over
// 256 x 256 output tiles, each pair computing a tile with cta_group::2 MMAs:
//   warp 0    TMA producer in both CTAs: this CTA's 128 rows of A and 128 rows
//             of B per k-block, 128-byte swizzled, into a 5-stage ring; both
//             CTAs' copies complete on the even CTA's barrier
//   warp 1    TMEM allocator (both CTAs) and, in the even CTA, the MMA issuer:
//             tcgen05.mma.cta_group::2 M=256 N=256, 4 MMAs per 128-byte
//             k-block, commits multicast to both CTAs to free the stage; a
//             2 x 256-column accumulator per CTA lets the epilogue of one tile
//             overlap the main loop of the next
//   warps 2-9 epilogue in both CTAs: two warps per TMEM lane quarter, each
//             taking 128 of the 256 columns of this CTA's 128 rows, 32 at a
//             time (tcgen05.ld), fused math; each warp stages its 32 x 32
//             output blocks (and, for the symmetric products, their mirror
//             blocks, written column-wise) in its own 8 KB of shared memory
//             and writes them with TMA stores; the last C X, a read-modify-
//             write of W in W's own orientation, loads each 32 x 32 block of
//             W there by TMA, updates it in place and stores it and its bf16
//             copy by TMA (plain loads and stores through a transpose slab
//             when a matrix does not meet TMA's alignment rules)
//   warp 10   tile scheduler in the even CTA: claims tiles from a launch-wide
//             counter and publishes them to both CTAs through a ring of
//             tile indices, ahead of the roles that read it
// Per MMA each SM stages 8 KB of operands (A and B halves) instead of the
// 12 KB a single-CTA 128 x 256 tile needs.
//
// The Gram matrix and the polynomial are symmetric: only the 256x256 blocks
// on or below the diagonal are computed, and off-diagonal blocks are also
// stored transposed.
//
// Every wait on an mbarrier is bounded (about 2 s of %globaltimer).  A wait
// that runs out records a status code in the workspace header, raises a CTA
// abort flag, and every role leaves its loop; the MMA issuer drains its
// outstanding MMAs and the producer its outstanding copies (again with bounded
// waits) before TMEM is released.

#include <cuda.h>
#include <cuda_fp16.h>

#include "../../include/mpopt.h"
#include "internal.h"

namespace mpopt {
namespace {

constexpr int BM = 128;                       // rows of the tile held by one CTA
constexpr int BM_PAIR = 256;                  // rows of the tile of a CTA pair (MMA M)
constexpr int BN = 256;                       // columns of the tile (MMA N)
constexpr int BN_HALF = 128;                  // B rows staged by one CTA
constexpr int kStages = 5;
constexpr int kRowBytes = 128;                 // one swizzle row per k-block
constexpr int kStageA = BM * kRowBytes;        // 16 KB: this CTA's 128 rows of A
constexpr int kStageB = BN_HALF * kRowBytes;   // 16 KB: this CTA's 128 rows of B
constexpr int kStageBytes = kStageA + kStageB; // per CTA; the pair's stage is twice this
constexpr int kMnBlockBytes = 64 * kRowBytes;   // MN-major B: one 64-column block of 64 K rows
constexpr int kEpiWarps = 8;                   // two warps per TMEM lane quarter
constexpr int kThreads = 96 + 32 * kEpiWarps;  // TMA warp, MMA warp, epilogue warps, scheduler warp
constexpr int kTmemCols = 512;                 // 2 accumulators x 256 fp32 columns
constexpr int kSlabWords = 32 * 33;            // 32 x 32 fp32 transpose slab, padded rows
constexpr int kWarpScratch = 8192;             // per epilogue warp: transpose slab or TMA-store staging
constexpr int kSlabBytes = kEpiWarps * kWarpScratch;
constexpr int kOutBlockBytes = 32 * 32 * 2;    // one 32 x 32 fp16 block staged for a TMA store
constexpr int kOutBlockBytes32 = 32 * 32 * 4;  // one 32 x 32 fp32 block
static_assert(kSlabWords * 4 <= kWarpScratch, "transpose slab larger than a warp's scratch");
static_assert(kOutBlockBytes32 + 2 * kOutBlockBytes <= kWarpScratch, "W staging larger than a warp's scratch");
static_assert(4 * kOutBlockBytes <= kWarpScratch, "two staging buffers of a block and its mirror");
constexpr uint32_t kSmemBytes = kStages * kStageBytes + kSlabBytes + 1024 /*align*/ + 256 /*barriers*/;
static_assert(kSmemBytes <= 232448, "dynamic shared memory above the 227 KB a CTA may use");
constexpr unsigned long long kWaitLimitNs = 2000000000ull;
constexpr int kTileSlots = 3;                  // tile-index ring between the scheduler and the other roles
// consumers of one ring slot, all arriving on the even CTA's barrier: both
// CTAs' producers, the MMA warp, and every epilogue warp of both CTAs
constexpr uint32_t kTileConsumers = 2 + 1 + 2 * kEpiWarps;
constexpr int kBarrierBytes = (2 * kStages + 5 + 2 * kTileSlots + kEpiWarps) * 8 + 8 + 4 * kTileSlots;
static_assert(kBarrierBytes <= 256, "barrier block larger than its 256-byte reservation");

struct GemmParams {
  int mode;             // NsGemmMode
  int k_blocks;
  int tiles_per_mat;
  int total_tiles;
  int tiles_m;          // bx: Ap / BM_PAIR
  int count;
  int64_t Ap, Bp;
  const uint16_t* Ah;   // poly: fp16 A, for the b A term (the gram writes it through map_out)
  uint16_t* Ch;         // poly: out
  uint16_t* Xh;         // bx: fp16 iterate out (the other buffer of the pair)
  float a, b, c;
  float decay;
  int ns_only;
  uint32_t* status;
  uint32_t* sched;      // [0]: tiles claimed after the first, [1]: CTAs finished
  int stall;            // self-test: the even CTA of pair 0 never signals its first stage
  int w_tma;            // last C X: W and its bf16 copy move through TMA, with the maps in WMaps
  const float* in_scale;  // first iteration: per-matrix x0_scale (X0 = x0_scale * iterate); X X^T's
                          // output is multiplied by its square and C X's by it; nullptr later
};

// Tensor maps of the last C X's update, one pair per matrix of the group
// (a kernel parameter: 16 KB).  Both have a 32 x 32 box in W's own layout.
struct WMaps {
  CUtensorMap w[kMaxGroup];    // fp32 master W [R][C], 128-byte swizzle
  CUtensorMap wb[kMaxGroup];   // bf16 model copy [R][C], 64-byte swizzle
};

// Arguments only the last C X reads: the group's matrices (W, its bf16 copy,
// the update scale) and their tensor maps.  The other launches take the empty
// form, so that their parameter blocks stay under 1 KB: launches whose
// parameters are tens of KB fill the driver's launch queue after about 180
// pending launches and then block the host thread until earlier ones finish.
template <bool kFinal>
struct FinalArgs {
  int32_t unused;
};
template <>
struct FinalArgs<true> {
  MuonGroup grp;
  WMaps wm;
};
static_assert(3 * sizeof(CUtensorMap) + sizeof(GemmParams) + sizeof(FinalArgs<true>) + 256 <= 32764,
              "kernel parameters above the 32 KB parameter space");
static_assert(3 * sizeof(CUtensorMap) + sizeof(GemmParams) + sizeof(FinalArgs<false>) <= 1024,
              "parameters of the non-final GEMM launches above 1 KB");

// ------------------------------------------------------------ PTX helpers --

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Bounded wait: true when the phase completed; false when the CTA is aborting
// (another role timed out) or this wait ran out of time (then it raises the
// abort flag and records `code` in the workspace header).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                          uint32_t* status, uint32_t code) {
  if (mbar_try(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1u;
        atomicCAS(status, 0u, code);
        return false;
      }
    }
  }
}

// Tile load into this CTA's shared memory; completion is signalled on `bar`,
// a shared::cluster address that may be the even CTA's barrier.
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y, int z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// The same for a 4-D tensor map (the MN-major operand: column blocks as a dimension).
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x,
                                            int y, int z, int w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

// L2 policy for data touched once (W of the last C X): evicted first, so
// that it does not push the GEMM operands out of L2.
__device__ __forceinline__ uint64_t l2_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// A 2-D box into this CTA's own shared memory, completing on this CTA's
// barrier, with an L2 policy.
__device__ __forceinline__ void tma_load_2d_local(uint32_t dst, const CUtensorMap* map, uint32_t bar, int x, int y,
                                                  uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, uint32_t src, int x, int y, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(src), "l"(pol)
               : "memory");
}

// Tile store from this CTA's shared memory to global memory (bulk async-group
// of the issuing thread).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap* map, uint32_t src, int x, int y, int z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%1, %2, %3}], [%4];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(src)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until at most one of this thread's bulk groups still reads shared memory.
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Wait until all of this thread's bulk groups have completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Make this thread's generic-proxy shared-memory writes visible to the TMA.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Shared-memory matrix descriptor: K-major operand, 128-byte swizzle, rows of
// 128 bytes, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// Shared-memory matrix descriptor: MN-major operand, 128-byte swizzle.  The
// tile is stored as 64-element (128-byte) wide column blocks, each 64 K rows
// of 128 bytes: 8-row groups 1024 bytes apart (stride byte offset) and column
// blocks 8192 bytes apart (leading byte offset).
__device__ __forceinline__ uint64_t smem_desc_mn(uint32_t addr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr & 0x3FFFFu) >> 4);   // start address
  d |= static_cast<uint64_t>(kMnBlockBytes >> 4) << 16;  // leading byte offset: next 64 columns
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset: next 8 K rows
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version
  d |= static_cast<uint64_t>(2) << 61;                   // 128-byte swizzle
  return d;
}

// Instruction descriptor for kind::f16: fp32 accumulator (bits 4-5 = 1), A and
// B fp16 (format 0 in bits 7-9 and 10-12), A K-major, B K-major or MN-major
// (bit 16), N = 256 (bits 17-22, N >> 3), M = 256 across the CTA pair
// (bits 24-28, M >> 4).
__host__ __device__ constexpr uint32_t instr_desc(bool b_mn_major) {
  return (1u << 4) | (0u << 7) | (0u << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(BN >> 3) << 17) | (static_cast<uint32_t>(BM_PAIR >> 4) << 24);
}

// Pair MMA, issued by the even CTA: D[256 x 256] (+)= A[256 x 16] B[16 x 256]
// with A's rows 0-127 / 128-255 and B's columns 0-127 / 128-255 in the shared
// memory of the even / odd CTA at the descriptors' offsets; each CTA's TMEM
// receives its own 128 rows of D.
__device__ __forceinline__ void mma(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` (same shared-memory offset) in both CTAs of the pair once all
// previously issued MMAs of this thread have completed.
__device__ __forceinline__ void mma_commit_pair(uint32_t bar) {
  const uint16_t both = 3;
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(bar),
      "h"(both)
      : "memory");
}

// Arrive on `bar` in this CTA only once all previously issued MMAs completed.
__device__ __forceinline__ void mma_commit_local(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}

// The shared::cluster address of the variable at `addr` in CTA `rank` of the pair.
__device__ __forceinline__ uint32_t peer_addr(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ void mbar_arrive_local(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Store to the shared memory of a CTA of this cluster (address from mapa).
__device__ __forceinline__ void st_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// Wait for a phase completed by an arrive.release.cluster from the other CTA,
// so that the data it published before arriving is visible here.
__device__ __forceinline__ bool mbar_try_acq_cluster(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_acq_cluster(uint32_t bar, uint32_t parity, volatile uint32_t* abort_flag,
                                                      uint32_t* status, uint32_t code) {
  if (mbar_try_acq_cluster(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_acq_cluster(bar, parity)) return true;
    if ((i & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_ns() - t0 > kWaitLimitNs) {
        *abort_flag = 1u;
        atomicCAS(status, 0u, code);
        return false;
      }
    }
  }
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// ------------------------------------------------------- tile scheduling --

struct Tile {
  int mat, tm, tn;
  bool mirror;   // symmetric modes: also store the transposed tile
};

// A tile is a 256 x 256 block (tm, tn) of the output, computed by one CTA pair.
__device__ __forceinline__ Tile decode_tile(const GemmParams& P, int tile) {
  Tile t;
  t.mat = tile / P.tiles_per_mat;
  const int r = tile - t.mat * P.tiles_per_mat;
  if (P.mode == kGram || P.mode == kPoly) {
    // r enumerates the blocks (I, J) with J <= I of the symmetric output
    int I = static_cast<int>((sqrtf(8.f * static_cast<float>(r) + 1.f) - 1.f) * 0.5f);
    while ((I + 1) * (I + 2) / 2 <= r) ++I;
    while (I * (I + 1) / 2 > r) --I;
    const int J = r - I * (I + 1) / 2;
    t.tm = I;
    t.tn = J;
    t.mirror = (I != J);
  } else {
    t.tn = r / P.tiles_m;
    t.tm = r - t.tn * P.tiles_m;
    t.mirror = false;
  }
  return t;
}

// --------------------------------------------------------------- epilogue --

__device__ __forceinline__ uint16_t f16_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  return static_cast<uint32_t>(f16_bits(lo)) | (static_cast<uint32_t>(f16_bits(hi)) << 16);
}

// Staging of 32 x 32 fp16 blocks for TMA stores.  Lane t holds row t of the
// block (columns 0..31) in v.  The blocks use the 64-byte swizzle (16-byte
// chunk q of row r at chunk q ^ ((r >> 1) & 3)); the buffers are 1024-byte
// aligned.
__device__ __forceinline__ void stage_f16_rows(uint8_t* buf, int lane, const float (&v)[32]) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint32_t phys = static_cast<uint32_t>(q) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u);
    *reinterpret_cast<uint4*>(buf + lane * 64 + phys * 16) =
        make_uint4(pack_f16(v[8 * q], v[8 * q + 1]), pack_f16(v[8 * q + 2], v[8 * q + 3]),
                   pack_f16(v[8 * q + 4], v[8 * q + 5]), pack_f16(v[8 * q + 6], v[8 * q + 7]));
  }
}

// The transposed block: lane t writes column t (element (j, t) = v[j]).
__device__ __forceinline__ void stage_f16_cols(uint8_t* buf, int lane, const float (&v)[32]) {
  const uint32_t chunk = static_cast<uint32_t>(lane) >> 3, within = (static_cast<uint32_t>(lane) & 7u) * 2u;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const uint32_t phys = chunk ^ ((static_cast<uint32_t>(j) >> 1) & 3u);
    *reinterpret_cast<uint16_t*>(buf + j * 64 + phys * 16 + within) = f16_bits(v[j]);
  }
}

__device__ __forceinline__ void bulk_wait_read_0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }

// Warp-level 32 x 32 transpose through the warp's shared-memory slab: on
// entry lane t holds row t (columns 0..31) in v; on exit lane t holds column t
// (rows 0..31) in w.
__device__ __forceinline__ void warp_transpose(float* slab, int lane, const float (&v)[32], float (&w)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) slab[lane * 33 + j] = v[j];
  __syncwarp();
#pragma unroll
  for (int r = 0; r < 32; ++r) w[r] = slab[r * 33 + lane];
  __syncwarp();
}

// fp32 -> bf16 bits, round to nearest, ties to even; NaN -> 0x7FC0 (adding
// 0x7FFF plus the lowest kept bit carries into the kept half exactly when the
// dropped half is above one half, or one half with an odd kept half).
__device__ __forceinline__ uint16_t bf16_rne(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7fffffffu) > 0x7f800000u) return 0x7fc0u;
  return static_cast<uint16_t>((u + 0x7fffu + ((u >> 16) & 1u)) >> 16);
}

// One 32-row x 32-column block of the tile held by one epilogue warp: lane
// `lane` holds row row0 + lane, columns col0 .. col0 + 31, in v.
__device__ __forceinline__ void epilogue_block(const GemmParams& P, const MuonGroup& grp, const Tile& t,
                                               float* slab, int lane, int row0, int col0, float (&v)[32]) {
  const int row = row0 + lane;
  float w[32];
  {
    // last iteration: O = X' in the wide orientation (rows: A index, columns: B index).
    // The warp updates 32 runs of 32 consecutive W elements: for a tall W
    // (stored as the transpose of the wide layout) run j is W[col0 + j][row0 ..
    // row0 + 31] and lanes already hold rows; for a wide W run k is
    // W[row0 + k][col0 .. col0 + 31] and lanes need columns (transpose first).
    // All loads of W are issued before any store so their latencies overlap.
    const MuonMat& M = grp.mats[t.mat];
    const int64_t A = grp.A, B = grp.B, C = M.C;
    int64_t first, n_runs;
    bool lane_ok;
    if (M.transposed) {
#pragma unroll
      for (int j = 0; j < 32; ++j) w[j] = v[j];
      first = static_cast<int64_t>(col0) * C + row;
      n_runs = B - col0 < 32 ? B - col0 : 32;
      lane_ok = row < A;
    } else {
      warp_transpose(slab, lane, v, w);
      first = static_cast<int64_t>(row0) * C + col0 + lane;
      n_runs = A - row0 < 32 ? A - row0 : 32;
      lane_ok = col0 + lane < B;
    }
    if (lane_ok && n_runs > 0) {
      if (P.ns_only) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          if (j < n_runs) __stcs(M.O + first + j * C, w[j]);
      } else {
        float old[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) old[j] = (j < n_runs) ? __ldcs(M.W + first + j * C) : 0.f;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (j < n_runs) {
            const float wv = old[j] * P.decay - M.step_scale * w[j];
            __stcs(M.W + first + j * C, wv);
            if (M.Wb) __stcs(M.Wb + first + j * C, bf16_rne(wv));
          }
        }
      }
    }
  }
}

// ------------------------------------------------------------------ kernel --

// Kernel variants: kNonFinal for X X^T, A A and every C X but the last;
// kFinalTma for the last C X (mode kBxFinal) when W and its bf16 copy move
// through TMA; kFinalPlain for the last C X otherwise (plain loads and stores
// through a transpose slab; also the output of opt_newton_schulz).  Each
// variant compiles only its own epilogue.  The last C X reads the group's
// matrices and W maps from `fa`.
enum : int { kNonFinal = 0, kFinalTma = 1, kFinalPlain = 2 };

template <int kVariant>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
ns_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
               const __grid_constant__ CUtensorMap map_out, const __grid_constant__ GemmParams P,
               const __grid_constant__ FinalArgs<kVariant != kNonFinal> fa) {
  constexpr bool kFinal = kVariant != kNonFinal;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_a = smem;                                  // kStages x 16 KB
  uint8_t* stage_b = smem + kStages * kStageA;              // kStages x 16 KB
  uint8_t* scratch = smem + kStages * kStageBytes;         // kEpiWarps x 8 KB
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes + kSlabBytes);
  uint64_t* full = bars;                     // [kStages]  even CTA: both CTAs' copies landed
  uint64_t* empty = bars + kStages;          // [kStages]  both CTAs: stage free again
  uint64_t* acc_full = bars + 2 * kStages;   // [2]        both CTAs: accumulator ready
  uint64_t* acc_empty = acc_full + 2;        // [2]        even CTA: both epilogues drained it
  uint64_t* drain = acc_empty + 2;           // [1]        even CTA: all MMAs complete
  uint64_t* tile_full = drain + 1;           // [kTileSlots] both CTAs: next tile index published
  uint64_t* tile_empty = tile_full + kTileSlots;   // [kTileSlots] even CTA: every role has read it
  uint64_t* wload = tile_empty + kTileSlots; // [kEpiWarps] each epilogue warp: its block of W landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(wload + kEpiWarps);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile int* tile_ring = reinterpret_cast<volatile int*>(tmem_slot + 2);   // [kTileSlots]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();      // 0: even CTA (issues the MMAs), 1: odd CTA
  const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  // C X takes X [K = Ap][N = Bp] as an MN-major B operand; the symmetric
  // products take K-major rows for both operands
  const bool b_mn = P.mode == kBx || P.mode == kBxFinal;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(smem_u32(&acc_full[a]), 1);
      mbar_init(smem_u32(&acc_empty[a]), 2 * 32 * kEpiWarps);
    }
    mbar_init(smem_u32(drain), 1);
    for (int k = 0; k < kTileSlots; ++k) {
      mbar_init(smem_u32(&tile_full[k]), 1);
      mbar_init(smem_u32(&tile_empty[k]), kTileConsumers);
    }
    for (int w = 0; w < kEpiWarps; ++w) mbar_init(smem_u32(&wload[w]), 1);
    *abort_flag = 0u;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 0 && lane == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_a)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&map_b)) : "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();            // barriers of both CTAs initialised, TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  constexpr int kElemsPerKBlock = 64;          // 128 bytes of fp16 per row

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ TMA producer --
      // Tiles come from the scheduler warp through the tile ring.  Both CTAs
      // load their own halves; completion is counted on the even CTA's full
      // barrier, which expects both halves' bytes.
      bool ok = true;
      bool issued = false;
      // stage s of the ring, phase parity ph; addresses of stage 0 (a stage is a fixed offset)
      const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
      const uint32_t full0_even = peer_addr(full0, 0);   // both CTAs' loads complete on the even CTA's barrier
      const uint32_t sa0 = smem_u32(stage_a), sb0 = smem_u32(stage_b);
      uint32_t s = 0, ph = 0;
      // self-test of the bounded waits: the even CTA of pair 0 withholds its
      // first stage, so the MMA issuer's wait for it runs out
      const bool withhold = P.stall != 0 && rank == 0 && pair == 0;
      const uint32_t tempty_even = peer_addr(smem_u32(&tile_empty[0]), 0);
      for (uint32_t seq = 0; ok; ++seq) {
        const uint32_t slot = seq % kTileSlots, sph = (seq / kTileSlots) & 1u;
        int tile;
        if (rank == 0) {
          if (!mbar_wait(smem_u32(&tile_full[slot]), sph, abort_flag, P.status, kStatusTimeoutTile)) {
            ok = false;
            break;
          }
          tile = tile_ring[slot];
          mbar_arrive_local(smem_u32(&tile_empty[slot]));
        } else {
          if (!mbar_wait_acq_cluster(smem_u32(&tile_full[slot]), sph, abort_flag, P.status, kStatusTimeoutTile)) {
            ok = false;
            break;
          }
          tile = tile_ring[slot];
          mbar_arrive_remote(tempty_even + 8 * slot);
        }
        if (tile >= P.total_tiles) break;
        const Tile t = decode_tile(P, tile);
        const int arow = t.tm * BM_PAIR + static_cast<int>(rank) * BM;
        const int brow = t.tn * BN + static_cast<int>(rank) * BN_HALF;   // B rows (K-major) or columns (MN-major)
        for (int kb = 0; kb < P.k_blocks; ++kb) {
          if (!mbar_wait(empty0 + 8 * s, ph ^ 1u, abort_flag, P.status, kStatusTimeoutEmpty)) {
            ok = false;
            break;
          }
          if (!(withhold && seq == 0 && kb == 0)) {
            const uint32_t fb = full0_even + 8 * s;
            if (rank == 0) mbar_expect_tx(full0 + 8 * s, 2 * kStageBytes);
            const int kx = kb * kElemsPerKBlock;
            const uint32_t sa = sa0 + s * kStageA, sb = sb0 + s * kStageB;
            tma_load_3d(sa, &map_a, fb, kx, arow, t.mat);
            if (b_mn) {
              // MN-major B: this CTA's 128 columns as two 64-column blocks of 64 K
              // rows, one box of the 4-D map (blocks land kMnBlockBytes apart)
              tma_load_4d(sb, &map_b, fb, 0, kx, brow / 64, t.mat);
            } else {
              tma_load_3d(sb, &map_b, fb, kx, brow, t.mat);
            }
            issued = true;
          }
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      if (!ok && issued) {
        // abort: give copies already issued time to land before the CTA exits
        const unsigned long long t0 = global_ns();
        while (global_ns() - t0 < 10000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // ------------------------------------- MMA issuer (even CTA only) --
      const uint32_t idesc = b_mn ? instr_desc(true) : instr_desc(false);
      // operand descriptors of stage 0: a stage and a K step are offsets of the
      // start-address field (bits 0-13, address >> 4; shared memory stays below 256 KB)
      const uint64_t adesc0 = smem_desc(smem_u32(stage_a));
      const uint64_t bdesc0 = b_mn ? smem_desc_mn(smem_u32(stage_b)) : smem_desc(smem_u32(stage_b));
      const uint32_t b_kstep = b_mn ? (16 * kRowBytes) >> 4 : 32 >> 4;   // 16 MN-major rows or 32 bytes of a K-major row
      const uint32_t full0 = smem_u32(&full[0]), empty0 = smem_u32(&empty[0]);
      uint32_t s = 0, ph = 0;
      bool ok = true;
      for (uint32_t lt = 0; ok; ++lt) {   // lt: this pair's tile sequence number
        const uint32_t slot = lt % kTileSlots, sph = (lt / kTileSlots) & 1u;
        if (!mbar_wait(smem_u32(&tile_full[slot]), sph, abort_flag, P.status, kStatusTimeoutTile)) break;
        const int tile = tile_ring[slot];
        mbar_arrive_local(smem_u32(&tile_empty[slot]));
        if (tile >= P.total_tiles) break;
        const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1u;
        if (!mbar_wait(smem_u32(&acc_empty[acc]), acc_ph ^ 1u, abort_flag, P.status, kStatusTimeoutAccFree)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < P.k_blocks; ++kb) {
          // the operands were written by TMA and completed on this barrier:
          // its wait orders them before the MMAs, no tcgen05 fence needed
          if (!mbar_wait(full0 + 8 * s, ph, abort_flag, P.status, kStatusTimeoutFull)) {
            ok = false;
            break;
          }
          const uint64_t ad = adesc0 + s * (kStageA >> 4);
          const uint64_t bd = bdesc0 + s * (kStageB >> 4);
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)   // 4 MMAs of 16 K each
            mma(d_tmem, ad + 2 * kk, bd + b_kstep * kk, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
          mma_commit_pair(empty0 + 8 * s);
          if (++s == kStages) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(smem_u32(&acc_full[acc]));
      }
      // drain: every MMA issued by this thread has completed before TMEM goes;
      // a drain that runs out is recorded like any other timed-out wait
      mma_commit_local(smem_u32(drain));
      const unsigned long long t0 = global_ns();
      while (!mbar_try(smem_u32(drain), 0)) {
        if (global_ns() - t0 > kWaitLimitNs) {
          *abort_flag = 1u;
          atomicCAS(P.status, 0u, static_cast<uint32_t>(kStatusTimeoutDrain));
          break;
        }
      }
    }
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------ epilogue --
    const int quarter = warp & 3;             // TMEM lanes this warp may access
    const int half = (warp - 2) >> 2;         // which 128 of the 256 columns
    // this warp's 8 KB of scratch (1024-byte aligned): staging for the TMA
    // loads and stores of its blocks, or the transpose slab of the last C X
    // when W cannot move through TMA
    uint8_t* out_stage = scratch + (warp - 2) * kWarpScratch;
    float* slab = reinterpret_cast<float*>(out_stage);
    uint32_t out_blocks = 0;
    constexpr bool w_tma = kVariant == kFinalTma;
    const uint32_t wbar = smem_u32(&wload[warp - 2]);
    uint32_t wphase = 0;
    bool wait_failed = false;
    const uint32_t empty_even = peer_addr(smem_u32(&acc_empty[0]), 0);
    const uint32_t tempty_even = peer_addr(smem_u32(&tile_empty[0]), 0);
    for (uint32_t lt = 0;; ++lt) {   // lt: this pair's tile sequence number
      const uint32_t slot = lt % kTileSlots, sph = (lt / kTileSlots) & 1u;
      int tile = 0, got = 1;
      if (lane == 0) {
        got = (rank == 0 ? mbar_wait(smem_u32(&tile_full[slot]), sph, abort_flag, P.status, kStatusTimeoutTile)
                         : mbar_wait_acq_cluster(smem_u32(&tile_full[slot]), sph, abort_flag, P.status,
                                                 kStatusTimeoutTile))
                  ? 1
                  : 0;
        if (got) {
          tile = tile_ring[slot];
          if (rank == 0) mbar_arrive_local(smem_u32(&tile_empty[slot]));
          else mbar_arrive_remote(tempty_even + 8 * slot);
        }
      }
      got = __shfl_sync(0xffffffffu, got, 0);
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (!got || tile >= P.total_tiles) break;
      const uint32_t acc = lt & 1, acc_ph = (lt >> 1) & 1u;
      if (!mbar_wait(smem_u32(&acc_full[acc]), acc_ph, abort_flag, P.status, kStatusTimeoutAcc)) break;
      tc_fence_after();
      const Tile t = decode_tile(P, tile);
      const int row0 = t.tm * BM_PAIR + static_cast<int>(rank) * BM + quarter * 32;
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      // first iteration: the iterate is x_scale * gtilde; normalise here
      float in_f = 1.f;
      if (P.in_scale != nullptr) {
        in_f = P.in_scale[t.mat];
        if (!kFinal && P.mode == kGram) in_f *= in_f;
      }
      for (int c0 = half * (BN / 2); c0 < (half + 1) * (BN / 2); c0 += 32) {
        float v[32];
        // last C X through TMA: this block of W, in W's own layout (W rows are
        // the iterate's rows, or its columns for a tall W)
        bool tall = false;
        int wx = 0, wy = 0;
        if constexpr (kFinal) {
          tall = w_tma && fa.grp.mats[t.mat].transposed != 0;
          wx = tall ? row0 : t.tn * BN + c0;
          wy = tall ? t.tn * BN + c0 : row0;
          if (w_tma && lane == 0) {
            if (out_blocks > 0) bulk_wait_read_0();   // the previous block's stores have read the staging area
            mbar_expect_tx(wbar, kOutBlockBytes32);
            tma_load_2d_local(smem_u32(out_stage), &fa.wm.w[t.mat], wbar, wx, wy, l2_evict_first());
          }
        }
        __syncwarp();
        tmem_ld32(taddr + c0, v);
        if (P.in_scale != nullptr) {
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= in_f;
        }
        if constexpr (!kFinal) {
          if (P.mode == kBx) {
            // X' block: staged in shared memory, stored by one TMA store; two
            // staging buffers alternate
            uint8_t* buf = out_stage + (out_blocks & 1) * kOutBlockBytes;
            if (out_blocks >= 2 && lane == 0) bulk_wait_read_1();   // this buffer's previous store has read it
            __syncwarp();
            stage_f16_rows(buf, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&map_out, smem_u32(buf), t.tn * BN + c0, row0, t.mat);
              bulk_commit();
            }
            ++out_blocks;
          } else if (P.mode == kGram) {
            // A in fp16 (and the mirror block of an off-diagonal tile); two
            // staging buffers alternate
            const int col0 = t.tn * BN + c0;
            uint8_t* buf = out_stage + (out_blocks & 1) * (2 * kOutBlockBytes);
            if (out_blocks >= 2 && lane == 0) bulk_wait_read_1();   // this buffer's previous stores have read it
            __syncwarp();
            stage_f16_rows(buf, lane, v);
            if (t.tm != t.tn) stage_f16_cols(buf + kOutBlockBytes, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&map_out, smem_u32(buf), col0, row0, t.mat);
              if (t.tm != t.tn) tma_store_3d(&map_out, smem_u32(buf + kOutBlockBytes), row0, col0, t.mat);
              bulk_commit();
            }
            ++out_blocks;
          } else if (P.mode == kPoly) {
            // C = a I + b A + c (A A) in fp16 (and its mirror block); two
            // staging buffers alternate
            const int col0 = t.tn * BN + c0;
            const int row = row0 + lane;
            const uint16_t* Arow = P.Ah + static_cast<int64_t>(t.mat) * P.Ap * P.Ap + static_cast<int64_t>(row) * P.Ap + col0;
  #pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 a8 = __ldcs(reinterpret_cast<const uint4*>(Arow) + q);   // 8 fp16 values
              const uint32_t w[4] = {a8.x, a8.y, a8.z, a8.w};
  #pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&w[k]));
                v[8 * q + 2 * k + 0] = P.b * f.x + P.c * v[8 * q + 2 * k + 0];
                v[8 * q + 2 * k + 1] = P.b * f.y + P.c * v[8 * q + 2 * k + 1];
              }
            }
  #pragma unroll
            for (int j = 0; j < 32; ++j) v[j] += (row == col0 + j) ? P.a : 0.f;   // + a I
            uint8_t* buf = out_stage + (out_blocks & 1) * (2 * kOutBlockBytes);
            if (out_blocks >= 2 && lane == 0) bulk_wait_read_1();
            __syncwarp();
            stage_f16_rows(buf, lane, v);
            if (t.tm != t.tn) stage_f16_cols(buf + kOutBlockBytes, lane, v);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_3d(&map_out, smem_u32(buf), col0, row0, t.mat);
              if (t.tm != t.tn) tma_store_3d(&map_out, smem_u32(buf + kOutBlockBytes), row0, col0, t.mat);
              bulk_commit();
            }
            ++out_blocks;
          }
        } else {
          if constexpr (w_tma) {
            // W <- W (1 - lr wd) - lr scale X', updated in place in the staging
            // area (128-byte swizzle: 16-byte chunk q of row r at q ^ (r & 7)),
            // its bf16 copy staged 4 KB further (64-byte swizzle); both leave by
            // TMA stores, which clip at the matrix edge
            if (!mbar_wait(wbar, wphase, abort_flag, P.status, kStatusTimeoutWload)) {
              wait_failed = true;
              break;
            }
            wphase ^= 1u;
            const MuonMat& M = fa.grp.mats[t.mat];
            const float decay = P.decay, scale = M.step_scale;
            uint8_t* wbf = out_stage + kOutBlockBytes32;
            if (tall) {
              // lane t holds W column t of the block: element (j, t) for row j
              const uint32_t q32 = static_cast<uint32_t>(lane) >> 2, w32 = (static_cast<uint32_t>(lane) & 3u) * 4u;
              const uint32_t q16 = static_cast<uint32_t>(lane) >> 3, w16 = (static_cast<uint32_t>(lane) & 7u) * 2u;
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                float* e = reinterpret_cast<float*>(out_stage + j * 128 + ((q32 ^ (static_cast<uint32_t>(j) & 7u)) * 16) + w32);
                const float wv = *e * decay - scale * v[j];
                *e = wv;
                *reinterpret_cast<uint16_t*>(wbf + j * 64 + ((q16 ^ ((static_cast<uint32_t>(j) >> 1) & 3u)) * 16) + w16) =
                    bf16_rne(wv);
              }
            } else {
              // lane t holds W row t of the block
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                float4* e = reinterpret_cast<float4*>(out_stage + lane * 128 + ((static_cast<uint32_t>(q) ^ (static_cast<uint32_t>(lane) & 7u)) * 16));
                float4 o = *e;
                o.x = o.x * decay - scale * v[4 * q + 0];
                o.y = o.y * decay - scale * v[4 * q + 1];
                o.z = o.z * decay - scale * v[4 * q + 2];
                o.w = o.w * decay - scale * v[4 * q + 3];
                *e = o;
                v[4 * q + 0] = o.x;
                v[4 * q + 1] = o.y;
                v[4 * q + 2] = o.z;
                v[4 * q + 3] = o.w;
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const uint32_t phys = static_cast<uint32_t>(q) ^ ((static_cast<uint32_t>(lane) >> 1) & 3u);
                *reinterpret_cast<uint4*>(wbf + lane * 64 + phys * 16) = make_uint4(
                    static_cast<uint32_t>(bf16_rne(v[8 * q + 0])) | (static_cast<uint32_t>(bf16_rne(v[8 * q + 1])) << 16),
                    static_cast<uint32_t>(bf16_rne(v[8 * q + 2])) | (static_cast<uint32_t>(bf16_rne(v[8 * q + 3])) << 16),
                    static_cast<uint32_t>(bf16_rne(v[8 * q + 4])) | (static_cast<uint32_t>(bf16_rne(v[8 * q + 5])) << 16),
                    static_cast<uint32_t>(bf16_rne(v[8 * q + 6])) | (static_cast<uint32_t>(bf16_rne(v[8 * q + 7])) << 16));
              }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              const uint64_t pol = l2_evict_first();
              tma_store_2d(&fa.wm.w[t.mat], smem_u32(out_stage), wx, wy, pol);
              if (M.Wb) tma_store_2d(&fa.wm.wb[t.mat], smem_u32(wbf), wx, wy, pol);
              bulk_commit();
            }
            ++out_blocks;
          } else {
            epilogue_block(P, fa.grp, t, slab, lane, row0, t.tn * BN + c0, v);
          }
        }
      }
      if (wait_failed) break;
      tc_fence_before();
      mbar_arrive_remote(empty_even + acc * static_cast<uint32_t>(sizeof(uint64_t)));
    }
    if (wait_failed) {
      // a W block may still be on its way into the staging area: give it time to land
      const unsigned long long t0 = global_ns();
      while (global_ns() - t0 < 10000000ull) {
      }
    }
    if (lane == 0 && out_blocks > 0) bulk_wait_all();   // stores complete before the CTA exits
  } else if (lane == 0 && rank == 0) {
    // ----------------------------------------- tile scheduler (even CTA) --
    // Each pair starts with tile `pair` and then claims tiles from a
    // launch-wide counter, so the tiles in flight are always the most
    // recently claimed ones -- neighbours in the tile order, which share
    // operand panels in L2 -- however unevenly the pairs progress (with a
    // fixed stride they drift apart over a long launch and re-read their
    // panels from DRAM).  Every index, and finally one past the end, goes to
    // both CTAs through the tile ring.  Running in its own warp, the scheduler
    // fills the ring ahead of the roles that read it, so neither the
    // counter's round trip nor the publication to the odd CTA falls between
    // two tiles of the producers.
    const uint32_t ring_odd = peer_addr(smem_u32(const_cast<int*>(tile_ring)), 1);
    const uint32_t tfull_odd = peer_addr(smem_u32(&tile_full[0]), 1);
    for (uint32_t seq = 0;; ++seq) {
      const uint32_t slot = seq % kTileSlots, sph = (seq / kTileSlots) & 1u;
      if (!mbar_wait(smem_u32(&tile_empty[slot]), sph ^ 1u, abort_flag, P.status, kStatusTimeoutTile)) break;
      const int tile = seq == 0 ? pair : npairs + static_cast<int>(atomicAdd(P.sched, 1u));
      tile_ring[slot] = tile;
      st_cluster_u32(ring_odd + 4 * slot, static_cast<uint32_t>(tile));
      mbar_arrive_local(smem_u32(&tile_full[slot]));
      mbar_arrive_remote(tfull_odd + 8 * slot);
      if (tile >= P.total_tiles) break;
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();            // no CTA leaves while its partner may still signal it
  if (threadIdx.x == 0) {
    // the last CTA to finish (every claim of the launch is made by then)
    // resets the scheduler for the next launch on this workspace
    __threadfence();
    if (atomicAdd(P.sched + 1, 1u) == gridDim.x - 1) {
      atomicExch(P.sched, 0u);
      atomicExch(P.sched + 1, 0u);
    }
  }
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem_base), "r"(kTmemCols)
                 : "memory");
  }
}

// -------------------------------------------------------------- host side --

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 3-D map over `count` row-major fp16 matrices [rows][inner]; box = (64
// elements = 128 bytes of inner, box_rows, 1), 128-byte swizzle.
cudaError_t make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t count, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * 2), static_cast<cuuint64_t>(inner * rows * 2)};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(kRowBytes / 2), static_cast<cuuint32_t>(box_rows), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 4-D map over `count` row-major fp16 matrices [rows][inner] read as an MN-major
// operand: (64 columns, rows, inner / 64 column blocks, count), box (64, 64, 2,
// 1), 128-byte swizzle.  One box is 64 rows of two 64-column blocks, each block
// 64 x 128 bytes and stored 8 KB apart in shared memory.
cudaError_t make_map_mn(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t count) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(inner / 64),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(inner * 2), 128,
                                 static_cast<cuuint64_t>(inner * rows * 2)};
  const cuuint32_t box[4] = {64, 64, 2, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 3-D map over `count` row-major fp16 matrices [rows][inner] for the C X output:
// box 32 x 32 elements (64-byte rows), 64-byte swizzle.
cudaError_t make_out_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t count) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(count)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner * 2), static_cast<cuuint64_t>(inner * rows * 2)};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// 2-D map over one row-major matrix [rows][cols] of W (fp32, 128-byte swizzle)
// or of its bf16 copy (64-byte swizzle), box 32 x 32.
cudaError_t make_w_map(CUtensorMap* map, const void* base, int64_t cols, int64_t rows, bool bf16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols * (bf16 ? 2 : 4))};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        bf16 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Maps of every matrix of the group for the last C X; false when a matrix
// does not meet TMA's rules (16-byte aligned bases, row pitches a multiple of
// 16 bytes), and the update then takes plain loads and stores.
bool make_w_maps(const MuonGroup& grp, WMaps* wm) {
  for (int m = 0; m < grp.count; ++m) {
    const MuonMat& M = grp.mats[m];
    if ((reinterpret_cast<uintptr_t>(M.W) & 15u) != 0 || M.C % 4 != 0) return false;
    if (M.Wb && ((reinterpret_cast<uintptr_t>(M.Wb) & 15u) != 0 || M.C % 8 != 0)) return false;
    if (make_w_map(&wm->w[m], M.W, M.C, M.R, false) != cudaSuccess) return false;
    if (M.Wb && make_w_map(&wm->wb[m], M.Wb, M.C, M.R, true) != cudaSuccess) return false;
  }
  return true;
}

cudaError_t configure_gemm() {
  static thread_local int configured_dev = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_dev != dev) {
    e = cudaFuncSetAttribute(ns_gemm_kernel<kNonFinal>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ns_gemm_kernel<kFinalTma>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ns_gemm_kernel<kFinalPlain>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured_dev = dev;
  }
  return cudaSuccess;
}

int gemm_grid(const GemmParams& P) {
  const int max_pairs = num_sms() / 2;
  return 2 * (P.total_tiles < max_pairs ? P.total_tiles : max_pairs);
}

// X X^T, A A and every C X but the last
cudaError_t launch_gemm(const CUtensorMap& ma, const CUtensorMap& mb, const CUtensorMap& mo, const GemmParams& P,
                        cudaStream_t stream) {
  cudaError_t e = configure_gemm();
  if (e != cudaSuccess) return e;
  const FinalArgs<false> none{};
  ns_gemm_kernel<kNonFinal><<<gemm_grid(P), kThreads, kSmemBytes, stream>>>(ma, mb, mo, P, none);
  return cudaGetLastError();
}

// the last C X, which updates W (or writes the Newton-Schulz output)
cudaError_t launch_gemm_final(const CUtensorMap& ma, const CUtensorMap& mb, const GemmParams& P,
                              const FinalArgs<true>& fa, cudaStream_t stream) {
  cudaError_t e = configure_gemm();
  if (e != cudaSuccess) return e;
  if (P.w_tma)
    ns_gemm_kernel<kFinalTma><<<gemm_grid(P), kThreads, kSmemBytes, stream>>>(ma, mb, mb, P, fa);
  else
    ns_gemm_kernel<kFinalPlain><<<gemm_grid(P), kThreads, kSmemBytes, stream>>>(ma, mb, mb, P, fa);
  return cudaGetLastError();
}

}  // namespace

namespace {

// Launch parameters shared by every GEMM of a group of iterations.
GemmParams base_params(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s) {
  GemmParams P{};
  P.count = grp.count;
  P.Ap = grp.Ap;
  P.Bp = grp.Bp;
  P.decay = s.decay;
  P.ns_only = s.ns_only;
  P.status = buf.status;
  P.sched = buf.status + kSchedWord;
  P.in_scale = nullptr;
  return P;
}

// Symmetric product out = L R^T over the blocks on or below the diagonal,
// each off-diagonal block also stored as its mirror: the Gram matrix X X^T
// (L = R = X, K = Bp), or the product of two symmetric matrices that commute
// (K = Ap; R^T = R, and L R is symmetric), as in the grouped iterations.
cudaError_t launch_sym(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, const uint16_t* L,
                       const uint16_t* R, int64_t K, uint16_t* out, const float* in_scale, int stall, int kernel_id,
                       cudaStream_t stream) {
  const int64_t Ap = grp.Ap, cnt = grp.count;
  const int T = static_cast<int>(Ap / 256);
  cudaError_t e;
  CUtensorMap ma, mb, mo;
  if ((e = make_map(&ma, L, K, Ap, cnt, BM)) != cudaSuccess) return e;
  if ((e = make_map(&mb, R, K, Ap, cnt, BN_HALF)) != cudaSuccess) return e;
  if ((e = make_out_map(&mo, out, Ap, Ap, cnt)) != cudaSuccess) return e;
  GemmParams P = base_params(grp, buf, s);
  P.mode = kGram;
  P.k_blocks = static_cast<int>(K / 64);
  P.tiles_per_mat = T * (T + 1) / 2;
  P.total_tiles = P.tiles_per_mat * grp.count;
  P.stall = stall;
  P.in_scale = in_scale;
  prof_begin(kernel_id, grp.count, grp.A, grp.B, stream);
  e = launch_gemm(ma, mb, mo, P, stream);
  prof_end(stream);
  return e;
}

// The quintic's polynomial C = a I + b A + c (A A), fp16 in full.
cudaError_t launch_poly(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, const uint16_t* A,
                        uint16_t* out, int it, cudaStream_t stream) {
  const int64_t Ap = grp.Ap, cnt = grp.count;
  const int T = static_cast<int>(Ap / 256);
  cudaError_t e;
  CUtensorMap ma, mb, mo;
  if ((e = make_map(&ma, A, Ap, Ap, cnt, BM)) != cudaSuccess) return e;
  if ((e = make_map(&mb, A, Ap, Ap, cnt, BN_HALF)) != cudaSuccess) return e;
  if ((e = make_out_map(&mo, out, Ap, Ap, cnt)) != cudaSuccess) return e;
  GemmParams P = base_params(grp, buf, s);
  P.mode = kPoly;
  P.a = s.sched[it][0];
  P.b = s.sched[it][1];
  P.c = s.sched[it][2];
  P.k_blocks = static_cast<int>(Ap / 64);
  P.tiles_per_mat = T * (T + 1) / 2;
  P.total_tiles = P.tiles_per_mat * grp.count;
  P.Ah = A;
  P.Ch = out;
  prof_begin(OPT_KERNEL_NS_POLY, grp.count, grp.A, grp.B, stream);
  e = launch_gemm(ma, mb, mo, P, stream);
  prof_end(stream);
  return e;
}

// X' = M X (M K-major [Ap][Ap]; X [Ap][Bp] read as an MN-major B operand, one
// box of 64 K rows x two 64-column blocks per stage).  The last one updates W
// (or writes the Newton-Schulz output) instead of storing X'.
cudaError_t launch_bx(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, const uint16_t* M,
                      const uint16_t* X, uint16_t* X_next, bool last, const float* in_scale, cudaStream_t stream) {
  const int64_t Ap = grp.Ap, Bp = grp.Bp, cnt = grp.count;
  cudaError_t e;
  CUtensorMap ma, mb;
  if ((e = make_map(&ma, M, Ap, Ap, cnt, BM)) != cudaSuccess) return e;
  if ((e = make_map_mn(&mb, X, Bp, Ap, cnt)) != cudaSuccess) return e;
  GemmParams P = base_params(grp, buf, s);
  P.mode = last ? kBxFinal : kBx;
  P.k_blocks = static_cast<int>(Ap / 64);
  P.tiles_m = static_cast<int>(Ap / BM_PAIR);
  P.tiles_per_mat = static_cast<int>((Ap / BM_PAIR) * (Bp / BN));
  P.total_tiles = P.tiles_per_mat * grp.count;
  P.Xh = X_next;
  P.in_scale = in_scale;
  prof_begin(OPT_KERNEL_NS_BX, grp.count, grp.A, grp.B, stream);
  if (last) {
    // the last iteration's update of W moves through TMA when every matrix allows it
    static thread_local FinalArgs<true> fa;
    fa.grp = grp;
    P.w_tma = (!s.ns_only && make_w_maps(grp, &fa.wm)) ? 1 : 0;
    if (!P.w_tma) fa.wm = WMaps{};
    e = launch_gemm_final(ma, mb, P, fa, stream);
  } else {
    CUtensorMap mo;
    if ((e = make_out_map(&mo, X_next, Bp, Ap, cnt)) == cudaSuccess) e = launch_gemm(ma, mb, mo, P, stream);
  }
  prof_end(stream);
  return e;
}

}  // namespace

std::vector<int> ns_group_sizes(int ns_steps, bool grouped) {
  std::vector<int> sizes;
  if (!grouped) {
    sizes.assign(static_cast<size_t>(ns_steps), 1);
    return sizes;
  }
  const int groups = (ns_steps + kNsMaxGroupIters - 1) / kNsMaxGroupIters;
  for (int k = 0; k < groups; ++k) sizes.push_back(ns_steps / groups + (k < ns_steps % groups ? 1 : 0));
  return sizes;
}

cudaError_t launch_ns_group(const MuonGroup& grp, const NsBuffers& buf, const MuonScalars& s, int it0, int g,
                            int group_index, cudaStream_t stream) {
  const int64_t Ap = grp.Ap, Bp = grp.Bp;
  const bool first = it0 == 0;
  const float* in_scale = first ? buf.x0_scale : nullptr;   // X0 = x0_scale * iterate (first group only)
  const uint16_t* X = buf.Xh[group_index & 1];
  uint16_t* X_next = buf.Xh[(group_index + 1) & 1];
  // [Ap][Ap] fp16 buffers: the Gram matrix, the polynomial, and (grouped
  // iterations) two more; roles rotate so that no launch writes a buffer it reads
  uint16_t* sq[4] = {buf.Ah, buf.Ch, buf.Th[0], buf.Th[1]};
  auto free_slot = [](int x, int y, int z) {
    for (int k = 0; k < 4; ++k)
      if (k != x && k != y && k != z) return k;
    return -1;
  };
  cudaError_t e;
  int iA = 0, iC = 1, iM = 1;   // A_k, C_k and the running product M = C_k ... C_it0 (M = C_it0 at first)
  // A_it0 = X X^T; C_it0 = a I + b A + c A A
  if ((e = launch_sym(grp, buf, s, X, X, Bp, sq[iA], in_scale, first ? s.stall_first_stage : 0, OPT_KERNEL_NS_GRAM,
                      stream)) != cudaSuccess)
    return e;
  if ((e = launch_poly(grp, buf, s, sq[iA], sq[iC], it0, stream)) != cudaSuccess) return e;
  for (int j = 1; j < g; ++j) {
    if (!buf.Th[0] || !buf.Th[1]) return cudaErrorInvalidValue;
    // the next Gram matrix without the next iterate: X_{k+1} = C_k X_k, and
    // C_k commutes with A_k, so A_{k+1} = C_k A_k C_k = C_k (A_k C_k)
    const int iP = free_slot(iA, iC, iM);
    if ((e = launch_sym(grp, buf, s, sq[iA], sq[iC], Ap, sq[iP], nullptr, 0, OPT_KERNEL_NS_SYM, stream)) !=
        cudaSuccess)
      return e;
    if ((e = launch_sym(grp, buf, s, sq[iC], sq[iP], Ap, sq[iA], nullptr, 0, OPT_KERNEL_NS_SYM, stream)) !=
        cudaSuccess)
      return e;
    // C_{k+1} from A_{k+1}, into the product's buffer (no longer read)
    if ((e = launch_poly(grp, buf, s, sq[iA], sq[iP], it0 + j, stream)) != cudaSuccess) return e;
    const int iC_next = iP;
    const int iM_next = free_slot(iA, iC_next, iM);
    // M <- C_{k+1} M (every factor a polynomial in A_it0: they commute)
    if ((e = launch_sym(grp, buf, s, sq[iC_next], sq[iM], Ap, sq[iM_next], nullptr, 0, OPT_KERNEL_NS_SYM,
                        stream)) != cudaSuccess)
      return e;
    iC = iC_next;
    iM = iM_next;
  }
  // X_{it0+g} = M X_it0
  const bool last = it0 + g == s.ns_steps;
  return launch_bx(grp, buf, s, sq[iM], X, X_next, last, in_scale, stream);
}

}  // namespace mpopt
