// C ABI of libmpopt.so: argument validation, routing, workspace layout and
// the launch sequence of one optimizer step.  See include/mpopt.h for the
// contract of every entry point.

#include <cuda.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/mpopt.h"
#include "internal.h"

namespace mpopt {

int num_sms() {
  static thread_local int cached_dev = -1, cached = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (dev != cached_dev) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    cached = n;
    cached_dev = dev;
  }
  return cached;
}

namespace {
struct ProfState {
  cudaEvent_t const* events = nullptr;
  opt_launch_info* info = nullptr;
  int32_t capacity = 0;
  int32_t* count = nullptr;
  int32_t open = -1;
};
thread_local ProfState g_prof;
}  // namespace

void prof_begin(int kernel, int count, int64_t a, int64_t b, cudaStream_t stream) {
  if (!g_prof.count) return;
  const int32_t i = *g_prof.count;
  g_prof.open = -1;
  if (i < g_prof.capacity) {
    g_prof.info[i] = opt_launch_info{kernel, count, a, b};
    cudaEventRecord(g_prof.events[2 * i], stream);
    g_prof.open = i;
  }
}

void prof_end(cudaStream_t stream) {
  if (!g_prof.count) return;
  if (g_prof.open >= 0) cudaEventRecord(g_prof.events[2 * g_prof.open + 1], stream);
  g_prof.open = -1;
  ++*g_prof.count;
}

namespace {

constexpr size_t kHeaderBytes = 256;
constexpr size_t kAlign = 1024;

thread_local char g_last_cuda_error[256] = "";

opt_status cuda_fail(cudaError_t e, const char* where) {
  std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s (%s)", where, cudaGetErrorName(e),
                cudaGetErrorString(e));
  return OPT_ERR_CUDA;
}

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
int64_t pad_to(int64_t x, int64_t a) { return (x + a - 1) / a * a; }

bool finite(float x) { return std::isfinite(x); }

opt_status check_fp32_ptr(const void* p) {
  return (reinterpret_cast<uintptr_t>(p) & 3u) ? OPT_ERR_MISALIGNED : OPT_OK;
}

// Shape checks shared by both kinds (no pointer is read).
opt_status check_shape(const opt_tensor& t, bool muon) {
  if (t.rows < 0 || t.cols < 0) return OPT_ERR_INVALID_ARG;
  if (t.ndim < 0) return OPT_ERR_INVALID_ARG;
  if (t.rows > 0 && t.cols > (INT64_MAX / t.rows)) return OPT_ERR_INVALID_ARG;
  if (muon) {
    if (t.ndim != 2) return OPT_ERR_INVALID_ARG;
    if (t.rows > (int64_t(1) << 30) || t.cols > (int64_t(1) << 30)) return OPT_ERR_UNSUPPORTED;
    if (t.scale_rows < 0 || t.scale_cols < 0 || ((t.scale_rows == 0) != (t.scale_cols == 0)))
      return OPT_ERR_INVALID_ARG;
  }
  return OPT_OK;
}

// Per-tensor checks shared by both kinds.
opt_status check_tensor(const opt_tensor& t, bool muon) {
  const opt_status sh = check_shape(t, muon);
  if (sh != OPT_OK) return sh;
  const int64_t n = t.rows * t.cols;
  if (n == 0) return OPT_OK;
  if (!t.main_param || !t.main_grad || !t.exp_avg) return OPT_ERR_INVALID_ARG;
  if (!muon && !t.exp_avg_sq) return OPT_ERR_INVALID_ARG;
  opt_status s;
  if ((s = check_fp32_ptr(t.main_param)) != OPT_OK) return s;
  if ((s = check_fp32_ptr(t.main_grad)) != OPT_OK) return s;
  if ((s = check_fp32_ptr(t.exp_avg)) != OPT_OK) return s;
  if (!muon && (s = check_fp32_ptr(t.exp_avg_sq)) != OPT_OK) return s;
  if (t.model_param && (reinterpret_cast<uintptr_t>(t.model_param) & 1u)) return OPT_ERR_MISALIGNED;
  return OPT_OK;
}

opt_status check_adamw_hp(const opt_adamw_hp* hp) {
  if (!hp) return OPT_ERR_INVALID_ARG;
  if (!finite(hp->lr) || !finite(hp->eps) || !finite(hp->weight_decay)) return OPT_ERR_INVALID_ARG;
  if (!(hp->beta1 >= 0.f && hp->beta1 < 1.f) || !(hp->beta2 >= 0.f && hp->beta2 < 1.f)) return OPT_ERR_INVALID_ARG;
  if (hp->step < 1) return OPT_ERR_INVALID_ARG;
  return OPT_OK;
}

opt_status check_muon_hp(const opt_muon_hp* hp) {
  if (!hp) return OPT_ERR_INVALID_ARG;
  if (!finite(hp->lr) || !finite(hp->weight_decay) || !finite(hp->eps) || !finite(hp->ns_a) ||
      !finite(hp->ns_b) || !finite(hp->ns_c) || !finite(hp->scale_coeff))
    return OPT_ERR_INVALID_ARG;
  if (!(hp->momentum >= 0.f && hp->momentum < 1.f)) return OPT_ERR_INVALID_ARG;
  if (hp->eps < 0.f) return OPT_ERR_INVALID_ARG;
  if (hp->ns_steps < 0 || hp->ns_steps > 16) return OPT_ERR_INVALID_ARG;
  if (hp->scale_mode < OPT_SCALE_SPECTRAL || hp->scale_mode > OPT_SCALE_UNIT_RMS) return OPT_ERR_INVALID_ARG;
  if (hp->flags & ~(OPT_MUON_NO_ORTHOGONALIZE | OPT_MUON_NS_PER_ITERATION | OPT_MUON_NS_GROUPED))
    return OPT_ERR_INVALID_ARG;
  if ((hp->flags & OPT_MUON_NS_PER_ITERATION) && (hp->flags & OPT_MUON_NS_GROUPED)) return OPT_ERR_INVALID_ARG;
  if (hp->ns_schedule)
    for (int i = 0; i < 3 * hp->ns_steps; ++i)
      if (!finite(hp->ns_schedule[i])) return OPT_ERR_INVALID_ARG;
  return OPT_OK;
}

// Routing rule: "02 · Optimizer：算法与 infra" §5.5 / §14.2 -- Muon for 2-D
// parameters that are not embeddings or output heads, AdamW for the rest.
bool routes_to_muon(const opt_tensor& t, int32_t routing) {
  if (routing == OPT_KIND_ADAMW) return false;
  if (routing == OPT_KIND_MUON) return true;
  if (t.kind == OPT_KIND_MUON) return true;
  if (t.kind == OPT_KIND_ADAMW) return false;
  return t.ndim == 2 && !(t.flags & OPT_FLAG_EMBEDDING_OR_OUTPUT);
}

// ------------------------------------------------------------ AdamW plan --

// Elements to peel so that p, g, m, v (fp32) and model (bf16) are all 16-byte
// aligned at the same element index; -1 if no such index exists.
int32_t vector_head(const opt_tensor& t) {
  for (int h = 0; h < 8; ++h) {
    auto al = [h](const void* p, int esz) { return ((reinterpret_cast<uintptr_t>(p) + h * esz) & 15u) == 0; };
    if (al(t.main_param, 4) && al(t.main_grad, 4) && al(t.exp_avg, 4) && al(t.exp_avg_sq, 4) &&
        (!t.model_param || al(t.model_param, 2)))
      return h;
  }
  return -1;
}

AdamwTensorDesc describe(const opt_tensor& t, int64_t chunk_begin, int64_t& chunks) {
  const int64_t n = t.rows * t.cols;
  AdamwTensorDesc d{};
  d.p = t.main_param;
  d.g = t.main_grad;
  d.m = t.exp_avg;
  d.v = t.exp_avg_sq;
  d.model = t.model_param;
  d.numel = n;
  d.chunk_begin = chunk_begin;
  int32_t head = vector_head(t);
  if (head < 0) {
    chunks = (n + kAdamwChunk - 1) / kAdamwChunk;
  } else {
    if (head > n) head = static_cast<int32_t>(n);
    const int64_t body = n - head;
    chunks = body > 0 ? (body + kAdamwChunk - 1) / kAdamwChunk : 1;
  }
  d.head = head;
  return d;
}

AdamwScalars adamw_scalars(const opt_adamw_hp* hp) {
  // per-step scalars: double from the float hyper-parameters, rounded once
  const double lr = hp->lr, b1 = hp->beta1, b2 = hp->beta2, wd = hp->weight_decay;
  AdamwScalars s{};
  s.lr = hp->lr;
  s.beta1 = hp->beta1;
  s.beta2 = hp->beta2;
  s.eps = hp->eps;
  s.one_minus_beta1 = static_cast<float>(1.0 - b1);
  s.one_minus_beta2 = static_cast<float>(1.0 - b2);
  s.bias_c1 = static_cast<float>(1.0 - std::pow(b1, static_cast<double>(hp->step)));
  s.bias_c2 = static_cast<float>(1.0 - std::pow(b2, static_cast<double>(hp->step)));
  s.decay = static_cast<float>(1.0 - lr * wd);
  return s;
}

opt_status run_adamw(const opt_adamw_hp* hp, const std::vector<const opt_tensor*>& ts, cudaStream_t stream,
                     const float* grad_scale = nullptr) {
  static thread_local AdamwBatch batch;   // ~26 KB: kept off the stack
  batch.s = adamw_scalars(hp);
  batch.s.grad_scale = grad_scale;
  batch.n = 0;
  batch.total_chunks = 0;
  for (size_t i = 0; i <= ts.size(); ++i) {
    const bool flush = (i == ts.size()) || batch.n == kAdamwBatch;
    if (flush && batch.n > 0) {
      int64_t elems = 0;
      for (int32_t k = 0; k < batch.n; ++k) elems += batch.t[k].numel;
      prof_begin(OPT_KERNEL_ADAMW, batch.n, elems, 0, stream);
      const cudaError_t e = launch_adamw(batch, stream);
      prof_end(stream);
      if (e != cudaSuccess) return cuda_fail(e, "adamw launch");
      batch.n = 0;
      batch.total_chunks = 0;
    }
    if (i == ts.size()) break;
    if (ts[i]->rows * ts[i]->cols == 0) continue;
    int64_t chunks = 0;
    batch.t[batch.n] = describe(*ts[i], batch.total_chunks, chunks);
    batch.total_chunks += chunks;
    ++batch.n;
  }
  return OPT_OK;
}

// ------------------------------------------------------------- Muon plan --

struct ShapeClass {
  int64_t A, B;
  std::vector<const opt_tensor*> mats;
};

void shape_of(int64_t R, int64_t C, int64_t& A, int64_t& B, int64_t& Ap, int64_t& Bp) {
  A = R < C ? R : C;
  B = R < C ? C : R;
  Ap = pad_to(A, kNsPad);
  Bp = pad_to(B, kNsPad);
}

// Workspace of one group of `count` matrices with (min, max) = (A, B):
//   X x2 [Ap][Bp] fp16 (ping-pong), A [Ap][Ap] fp16, C [Ap][Ap] fp16,
//   (grouped iterations) two more [Ap][Ap] fp16, norm partials, inverse norms.
struct GroupLayout {
  size_t xh0, xh1, ah, ch, th0, th1, partial, inv, total;
};

GroupLayout group_layout(int64_t count, int64_t R, int64_t C, bool grouped) {
  int64_t A, B, Ap, Bp;
  shape_of(R, C, A, B, Ap, Bp);
  const size_t ab = static_cast<size_t>(Ap) * static_cast<size_t>(Bp);
  const size_t aa = static_cast<size_t>(Ap) * static_cast<size_t>(Ap);
  const size_t blocks = static_cast<size_t>(partials_per_matrix(A, B, Ap, Bp));
  GroupLayout L{};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off += align_up(bytes, kAlign);
    return o;
  };
  L.xh0 = take(count * ab * 2);
  L.xh1 = take(count * ab * 2);
  L.ah = take(count * aa * 2);
  L.ch = take(count * aa * 2);
  L.th0 = grouped ? take(count * aa * 2) : 0;
  L.th1 = grouped ? take(count * aa * 2) : 0;
  L.partial = take(count * blocks * 4);
  L.inv = take(count * kMatStats * 4);
  L.total = off;
  return L;
}

size_t group_bytes(int64_t count, int64_t R, int64_t C, bool grouped) {
  return group_layout(count, R, C, grouped).total;
}

// Whether a shape class takes grouped iterations by default (ns_grouping_pays).
bool class_grouped_by_default(int64_t A, int64_t B) {
  int64_t a, b, Ap, Bp;
  shape_of(A, B, a, b, Ap, Bp);
  return ns_grouping_pays(Ap, Bp);
}

NsBuffers carve(uint8_t* base, int64_t count, int64_t R, int64_t C, bool grouped, uint32_t* status) {
  const GroupLayout L = group_layout(count, R, C, grouped);
  NsBuffers b{};
  b.Xh[0] = reinterpret_cast<uint16_t*>(base + L.xh0);
  b.Xh[1] = reinterpret_cast<uint16_t*>(base + L.xh1);
  b.Ah = reinterpret_cast<uint16_t*>(base + L.ah);
  b.Ch = reinterpret_cast<uint16_t*>(base + L.ch);
  b.Th[0] = grouped ? reinterpret_cast<uint16_t*>(base + L.th0) : nullptr;
  b.Th[1] = grouped ? reinterpret_cast<uint16_t*>(base + L.th1) : nullptr;
  b.partial = reinterpret_cast<float*>(base + L.partial);
  b.inv_norm = reinterpret_cast<float*>(base + L.inv);
  b.x_scale = b.inv_norm + count;
  b.amax = reinterpret_cast<uint32_t*>(b.inv_norm + 2 * count);
  b.x0_scale = b.inv_norm + 3 * count;
  b.fix = reinterpret_cast<uint32_t*>(b.inv_norm + 4 * count);
  b.status = status;
  return b;
}

std::vector<ShapeClass> shape_classes(const std::vector<const opt_tensor*>& mats) {
  std::map<std::pair<int64_t, int64_t>, size_t> index;
  std::vector<ShapeClass> out;
  for (const opt_tensor* t : mats) {
    if (t->rows * t->cols == 0) continue;
    int64_t A, B, Ap, Bp;
    shape_of(t->rows, t->cols, A, B, Ap, Bp);
    auto key = std::make_pair(A, B);
    auto it = index.find(key);
    if (it == index.end()) {
      index[key] = out.size();
      out.push_back(ShapeClass{A, B, {}});
      out.back().mats.push_back(t);
    } else {
      out[it->second].mats.push_back(t);
    }
  }
  return out;
}

// Workspace for the Muon part with full groups (up to kMaxGroup matrices),
// with the buffers of grouped iterations for the classes that take them by
// default (for every class with `all_grouped`).
size_t muon_bytes(const std::vector<ShapeClass>& classes, bool all_grouped) {
  size_t need = 0;
  for (const ShapeClass& c : classes) {
    const int64_t cnt = static_cast<int64_t>(c.mats.size()) < kMaxGroup ? c.mats.size() : kMaxGroup;
    const size_t b = group_bytes(cnt, c.A, c.B, all_grouped || class_grouped_by_default(c.A, c.B));
    if (b > need) need = b;
  }
  return need;
}

struct MuonPlanHp {
  float lr, mu, wd, eps, a, b, c, scale_coeff;
  int nesterov, ns_steps, ns_only;
  const float* grad_scale;   // clipping factor on the device, or nullptr
  int scale_mode;            // OPT_SCALE_*
  int no_ortho;              // plain momentum SGD
  const float* schedule;     // host (a, b, c) per iteration, or nullptr: (a, b, c) every time
  int stall;                 // self-test of the bounded waits (opt_selftest_wait_timeout)
  int ns_order;              // 0: grouped iterations where they pay; OPT_MUON_NS_PER_ITERATION or
                             // OPT_MUON_NS_GROUPED (every shape, when the workspace has room)
};

// lr * update scale for a parameter of shape R x C ("02 · Optimizer：算法与
// infra" §5.4 Eq. 4 and §14.6): k sqrt(max(m, n)), k sqrt(max(1, m/n)) or
// k sqrt(m/n) with m = fan_out = R, n = fan_in = C; plain momentum SGD: k.
float step_scale_of(const MuonPlanHp& hp, int64_t R, int64_t C) {
  const double m = static_cast<double>(R), n = static_cast<double>(C);
  double f = 1.0;
  if (!hp.no_ortho) {
    if (hp.scale_mode == OPT_SCALE_SHAPE) f = std::sqrt(m / n > 1.0 ? m / n : 1.0);
    else if (hp.scale_mode == OPT_SCALE_UNIT_RMS) f = std::sqrt(m / n);
    else f = std::sqrt(m > n ? m : n);
  }
  return static_cast<float>(static_cast<double>(hp.lr) * static_cast<double>(hp.scale_coeff) * f);
}

// (a, b, c) of every iteration: the schedule when given, else the one triple.
void fill_schedule(const MuonPlanHp& hp, MuonScalars& s) {
  for (int it = 0; it < hp.ns_steps && it < 16; ++it) {
    s.sched[it][0] = hp.schedule ? hp.schedule[3 * it + 0] : hp.a;
    s.sched[it][1] = hp.schedule ? hp.schedule[3 * it + 1] : hp.b;
    s.sched[it][2] = hp.schedule ? hp.schedule[3 * it + 2] : hp.c;
  }
}

// Whether a class of (min, max) = (A, B) takes grouped iterations under hp
// (before the check that the workspace has room for their buffers).
bool wants_grouped(const MuonPlanHp& hp, int64_t A, int64_t B) {
  const int ns_steps = hp.no_ortho ? 0 : hp.ns_steps;
  return ns_steps >= 2 && hp.ns_order != OPT_MUON_NS_PER_ITERATION &&
         (hp.ns_order == OPT_MUON_NS_GROUPED || class_grouped_by_default(A, B));
}

// Grouped iterations multiply the group's first iterate once by the product
// M = C_{k0+g-1} ... C_k0, held in fp16.  C_k acts on each singular value s
// of its input as p_k(s^2), p_k(l) = a_k + b_k l + c_k l^2, and iteration k
// maps s to s |p_k(s^2)|.  The normalised input has every singular value in
// [0, 1], so the values iteration k can see lie in [0, S_k] with S_0 = 1 and
// S_{k+1} = max over [0, S_k] of s |p_k(s^2)|; the largest eigenvalue of M is
// at most the product of max |p_k| over [0, S_k] (3.44^3 = 41 for three
// iterations of the printed coefficients, about 42 with the grid's 1 %
// margin).  A group whose bound exceeds kNsGroupBound (16x below fp16's
// 65504) is split into single iterations.
constexpr double kNsGroupBound = 4096.0;

std::vector<int> fp16_safe_groups(const std::vector<int>& sizes, const MuonScalars& s, int ns_steps) {
  constexpr int kGrid = 4096;
  std::vector<double> bound(static_cast<size_t>(ns_steps));
  double smax = 1.0;
  for (int k = 0; k < ns_steps; ++k) {
    const double a = s.sched[k][0], b = s.sched[k][1], c = s.sched[k][2];
    double pmax = 0.0, next = 0.0;
    for (int i = 0; i <= kGrid; ++i) {
      const double x = smax * i / kGrid, l = x * x;
      const double p = std::fabs(a + b * l + c * l * l);
      pmax = std::max(pmax, p);
      next = std::max(next, x * p);
    }
    bound[static_cast<size_t>(k)] = pmax * 1.01;   // margin for the grid
    smax = std::min(next * 1.01, 1e30);
  }
  std::vector<int> out;
  int it = 0;
  for (const int g : sizes) {
    double prod = 1.0;
    for (int j = 0; j < g; ++j) prod *= bound[static_cast<size_t>(it + j)];
    if (g > 1 && !(prod <= kNsGroupBound)) out.insert(out.end(), static_cast<size_t>(g), 1);
    else out.push_back(g);
    it += g;
  }
  return out;
}

// Runs Muon on the matrices of one shape class; all of them must have rows x
// cols equal to (R, C) or (C, R) -- both orientations share a class.
opt_status run_muon_class(const MuonPlanHp& hp, const ShapeClass& cls, uint8_t* region, size_t region_bytes,
                          uint32_t* status, cudaStream_t stream, float* const* outputs /*ns_only*/) {
  // grouped iterations (launch_ns_group) when asked for or when they pay and
  // the region holds their two extra buffers for at least one matrix; then
  // the largest group of matrices that fits the region
  const int ns_steps = hp.no_ortho ? 0 : hp.ns_steps;
  const int64_t want = static_cast<int64_t>(cls.mats.size()) < kMaxGroup ? cls.mats.size() : kMaxGroup;
  const bool grouped = wants_grouped(hp, cls.A, cls.B) && group_bytes(1, cls.A, cls.B, true) <= region_bytes;
  int64_t cap = want;
  while (cap > 0 && group_bytes(cap, cls.A, cls.B, grouped) > region_bytes) --cap;
  if (cap == 0) return OPT_ERR_WORKSPACE;
  // matrices of both orientations share a group (the orientation is per matrix)
  for (size_t g0 = 0; g0 < cls.mats.size(); g0 += static_cast<size_t>(cap)) {
    {
      const size_t gn = std::min(cls.mats.size() - g0, static_cast<size_t>(cap));
      MuonGroup grp{};
      grp.count = static_cast<int32_t>(gn);
      grp.A = cls.A;
      grp.B = cls.B;
      grp.Ap = pad_to(cls.A, kNsPad);
      grp.Bp = pad_to(cls.B, kNsPad);
      for (size_t k = 0; k < gn; ++k) {
        const opt_tensor* t = cls.mats[g0 + k];
        MuonMat& M = grp.mats[k];
        M.W = t->main_param;
        M.g = t->main_grad;
        M.m = t->exp_avg;
        M.Wb = t->model_param;
        M.O = outputs ? outputs[g0 + k] : nullptr;
        M.R = static_cast<int32_t>(t->rows);
        M.C = static_cast<int32_t>(t->cols);
        M.transposed = t->rows > t->cols ? 1 : 0;
        M.vec4 = ((reinterpret_cast<uintptr_t>(M.g) | reinterpret_cast<uintptr_t>(M.m)) & 15u) == 0 ? 1 : 0;
        const int64_t sr = t->scale_rows > 0 ? t->scale_rows : t->rows;
        const int64_t sc = t->scale_cols > 0 ? t->scale_cols : t->cols;
        M.step_scale = step_scale_of(hp, sr, sc);
      }
      const NsBuffers buf = carve(region, static_cast<int64_t>(gn), cls.A, cls.B, grouped, status);
      MuonScalars s{};
      s.mu = hp.mu;
      s.one_minus_mu = static_cast<float>(1.0 - static_cast<double>(hp.mu));
      s.nesterov = hp.nesterov;
      s.eps = hp.eps;
      fill_schedule(hp, s);
      s.decay = static_cast<float>(1.0 - static_cast<double>(hp.lr) * static_cast<double>(hp.wd));
      s.no_normalize = hp.no_ortho;
      s.ns_steps = hp.ns_steps;
      s.ns_only = hp.ns_only;
      s.grad_scale = hp.grad_scale;
      s.stall_first_stage = (hp.stall && g0 == 0) ? 1 : 0;
      cudaError_t e = cudaSuccess;
      if (ns_steps > 0) {
        // one pass over g and m: momentum, Nesterov and the fp16 iterate,
        // scaled by a power of two from a sample; the normalisation is applied
        // by the first X X^T and C X epilogues (x0_scale)
        prof_begin(OPT_KERNEL_MUON_SAMPLE, grp.count, grp.A, grp.B, stream);
        e = launch_muon_sample(grp, buf, s, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon sample");
        prof_begin(OPT_KERNEL_MUON_PREP, grp.count, grp.A, grp.B, stream);
        e = launch_muon_prologue(grp, buf, s, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon prologue");
        prof_begin(OPT_KERNEL_MUON_NORM, grp.count, grp.A, grp.B, stream);
        e = launch_muon_norm(grp, buf, s, true, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon norm");
        prof_begin(OPT_KERNEL_MUON_OPERANDS, grp.count, grp.A, grp.B, stream);
        e = launch_muon_fixup(grp, buf, s, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon fix-up");
      } else {
        prof_begin(OPT_KERNEL_MUON_PREP, grp.count, grp.A, grp.B, stream);
        e = launch_muon_momentum(grp, buf, s, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon momentum");
        prof_begin(OPT_KERNEL_MUON_NORM, grp.count, grp.A, grp.B, stream);
        e = launch_muon_norm(grp, buf, s, false, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon norm");
      }
      if (ns_steps == 0) {
        prof_begin(OPT_KERNEL_MUON_APPLY, grp.count, grp.A, grp.B, stream);
        e = launch_muon_apply_direct(grp, buf, s, stream);
        prof_end(stream);
        if (e != cudaSuccess) return cuda_fail(e, "muon apply");
      }
      int it = 0, gi = 0;
      for (const int g : fp16_safe_groups(ns_group_sizes(ns_steps, grouped), s, ns_steps)) {
        e = launch_ns_group(grp, buf, s, it, g, gi++, stream);
        if (e != cudaSuccess) return cuda_fail(e, "newton-schulz gemm");
        it += g;
      }
    }
  }
  return OPT_OK;
}

opt_status check_workspace(const void* ws, size_t bytes, size_t need) {
  if (need == 0) return OPT_OK;
  if (!ws) return OPT_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(ws) & 255u) return OPT_ERR_WORKSPACE;
  if (bytes < need) return OPT_ERR_WORKSPACE;
  return OPT_OK;
}

struct Split {
  std::vector<const opt_tensor*> adamw, muon;
};

opt_status split_tensors(const opt_tensor* tensors, int32_t n, int32_t routing, Split& sp) {
  if (n < 0) return OPT_ERR_INVALID_ARG;
  if (n > 0 && !tensors) return OPT_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const opt_tensor& t = tensors[i];
    if (t.kind != OPT_KIND_AUTO && t.kind != OPT_KIND_ADAMW && t.kind != OPT_KIND_MUON) return OPT_ERR_INVALID_ARG;
    const bool muon = routes_to_muon(t, routing);
    const opt_status s = check_tensor(t, muon);
    if (s != OPT_OK) return s;
    (muon ? sp.muon : sp.adamw).push_back(&t);
  }
  return OPT_OK;
}

// The Muon plan's view of the caller's hyper-parameters.
MuonPlanHp plan_hp(const opt_muon_hp& h, const float* grad_scale) {
  MuonPlanHp hp{h.lr,          h.momentum,  h.weight_decay, h.eps,       h.ns_a,
                h.ns_b,        h.ns_c,      h.scale_coeff,  h.nesterov ? 1 : 0,
                h.ns_steps,    0,           grad_scale,     h.scale_mode,
                (h.flags & OPT_MUON_NO_ORTHOGONALIZE) ? 1 : 0, h.ns_schedule};
  hp.ns_order = h.flags & (OPT_MUON_NS_PER_ITERATION | OPT_MUON_NS_GROUPED);
  return hp;
}

// AdamW needs no workspace; Muon needs the status header and the group buffers.
size_t total_bytes(const std::vector<ShapeClass>& classes, bool all_grouped) {
  return classes.empty() ? 0 : kHeaderBytes + muon_bytes(classes, all_grouped);
}

// Minimum workspace: one matrix per Muon group.
size_t min_bytes(const std::vector<ShapeClass>& classes) {
  size_t m = 0;
  for (const ShapeClass& c : classes) m = std::max(m, group_bytes(1, c.A, c.B, false));
  return classes.empty() ? 0 : kHeaderBytes + m;
}

// Global-norm clipping of one step (opt_mixed_step_clipped).
struct ClipPlan {
  float max_norm;
  float* user_norm;
  float* user_scale;
};

// Header slots for the clipping factor and norm of the current step.
constexpr size_t kScaleSlot = 64, kNormSlot = 68;

int64_t clip_chunks(const Split& sp) {
  int64_t chunks = 0;
  for (const auto* list : {&sp.adamw, &sp.muon})
    for (const opt_tensor* t : *list) chunks += (t->rows * t->cols + kAdamwChunk - 1) / kAdamwChunk;
  return chunks;
}

size_t clip_bytes(const Split& sp) { return align_up(static_cast<size_t>(clip_chunks(sp)) * 4, kAlign); }

// Sum of squares of every gradient, then the clipping factor (device scalar).
opt_status run_clip(const Split& sp, const ClipPlan& clip, uint8_t* ws, cudaStream_t stream) {
  static thread_local NormBatch batch;
  float* partials = reinterpret_cast<float*>(ws + kHeaderBytes);
  int64_t offset = 0;
  batch.n = 0;
  batch.total_chunks = 0;
  batch.partial_offset = 0;
  std::vector<const opt_tensor*> all(sp.adamw);
  all.insert(all.end(), sp.muon.begin(), sp.muon.end());
  for (size_t i = 0; i <= all.size(); ++i) {
    const bool flush = (i == all.size()) || batch.n == kNormBatch;
    if (flush && batch.n > 0) {
      prof_begin(OPT_KERNEL_GRAD_NORM, batch.n, batch.total_chunks, 0, stream);
      const cudaError_t e = launch_grad_sumsq(batch, partials, stream);
      prof_end(stream);
      if (e != cudaSuccess) return cuda_fail(e, "gradient norm");
      offset += batch.total_chunks;
      batch.n = 0;
      batch.total_chunks = 0;
      batch.partial_offset = offset;
    }
    if (i == all.size()) break;
    const int64_t n = all[i]->rows * all[i]->cols;
    if (n == 0) continue;
    batch.t[batch.n] = NormTensorDesc{all[i]->main_grad, n, batch.total_chunks};
    batch.total_chunks += (n + kAdamwChunk - 1) / kAdamwChunk;
    ++batch.n;
  }
  prof_begin(OPT_KERNEL_CLIP_FINALIZE, 1, offset, 0, stream);
  const cudaError_t e = launch_clip_finalize(partials, offset, clip.max_norm, reinterpret_cast<float*>(ws + kScaleSlot),
                                             reinterpret_cast<float*>(ws + kNormSlot), clip.user_scale,
                                             clip.user_norm, stream);
  prof_end(stream);
  if (e != cudaSuccess) return cuda_fail(e, "clip factor");
  return OPT_OK;
}

opt_status mixed_impl(const opt_muon_hp* hpm, const opt_adamw_hp* hpa, const opt_tensor* tensors, int32_t n,
                      int32_t routing, void* workspace, size_t ws_bytes, void* stream_ptr,
                      const ClipPlan* clip = nullptr) {
  Split sp;
  opt_status st = split_tensors(tensors, n, routing, sp);
  if (st != OPT_OK) return st;
  bool any_adamw = false, any_muon = false;
  for (auto* t : sp.adamw) any_adamw |= (t->rows * t->cols) > 0;
  for (auto* t : sp.muon) any_muon |= (t->rows * t->cols) > 0;
  if (any_adamw && (st = check_adamw_hp(hpa)) != OPT_OK) return st;
  if (any_muon && (st = check_muon_hp(hpm)) != OPT_OK) return st;
  if (clip && !std::isfinite(clip->max_norm)) return OPT_ERR_INVALID_ARG;
  if (clip && ((reinterpret_cast<uintptr_t>(clip->user_norm) | reinterpret_cast<uintptr_t>(clip->user_scale)) & 3u))
    return OPT_ERR_MISALIGNED;
  if (!any_adamw && !any_muon) return OPT_OK;
  const bool clipping = clip && clip->max_norm > 0.f;   // max_norm <= 0: no clipping at all
  const std::vector<ShapeClass> classes = shape_classes(sp.muon);
  const size_t clip_region = clipping ? clip_bytes(sp) : 0;
  size_t need = min_bytes(classes);
  if (clipping) need = (need ? need : kHeaderBytes) + clip_region;
  if ((st = check_workspace(workspace, ws_bytes, need)) != OPT_OK) return st;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const float* grad_scale = nullptr;
  if (any_muon || clipping) {
    const cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderBytes, stream);
    if (e != cudaSuccess) return cuda_fail(e, "workspace header");
  }
  if (clipping) {
    if ((st = run_clip(sp, *clip, ws, stream)) != OPT_OK) return st;
    grad_scale = reinterpret_cast<const float*>(ws + kScaleSlot);
  }
  if (any_adamw && (st = run_adamw(hpa, sp.adamw, stream, grad_scale)) != OPT_OK) return st;
  if (any_muon) {
    uint32_t* status = reinterpret_cast<uint32_t*>(ws);
    const size_t off = kHeaderBytes + clip_region;
    const MuonPlanHp hp = plan_hp(*hpm, grad_scale);
    for (const ShapeClass& c : classes) {
      if ((st = run_muon_class(hp, c, ws + off, ws_bytes - off, status, stream, nullptr)) != OPT_OK) return st;
    }
  }
  return OPT_OK;
}

}  // namespace
}  // namespace mpopt

using namespace mpopt;

extern "C" {

size_t opt_workspace_size(const opt_tensor* tensors, int32_t n, int32_t routing) {
  const bool with_clip = (routing & OPT_WORKSPACE_CLIP) != 0;
  const bool all_grouped = (routing & OPT_WORKSPACE_GROUPED) != 0;
  routing &= ~(OPT_WORKSPACE_CLIP | OPT_WORKSPACE_GROUPED);
  if (routing != OPT_KIND_AUTO && routing != OPT_KIND_ADAMW && routing != OPT_KIND_MUON) return 0;
  Split sp;
  if (split_tensors(tensors, n, routing, sp) != OPT_OK) return 0;
  const size_t base = total_bytes(shape_classes(sp.muon), all_grouped);
  if (!with_clip) return base;
  return (base ? base : kHeaderBytes) + clip_bytes(sp);
}

opt_status opt_adamw_step(const opt_adamw_hp* hp, const opt_tensor* tensors, int32_t n, void* workspace,
                          size_t workspace_bytes, void* stream) {
  return mixed_impl(nullptr, hp, tensors, n, OPT_KIND_ADAMW, workspace, workspace_bytes, stream);
}

opt_status opt_muon_step(const opt_muon_hp* hp, const opt_tensor* t, void* workspace, size_t workspace_bytes,
                         void* stream) {
  if (!t) return OPT_ERR_INVALID_ARG;
  if (t->ndim != 2) return OPT_ERR_INVALID_ARG;
  return mixed_impl(hp, nullptr, t, 1, OPT_KIND_MUON, workspace, workspace_bytes, stream);
}

opt_status opt_mixed_step(const opt_muon_hp* hp_muon, const opt_adamw_hp* hp_adamw, const opt_tensor* tensors,
                          int32_t n, void* workspace, size_t workspace_bytes, void* stream) {
  return mixed_impl(hp_muon, hp_adamw, tensors, n, OPT_KIND_AUTO, workspace, workspace_bytes, stream);
}

opt_status opt_mixed_step_clipped(const opt_muon_hp* hp_muon, const opt_adamw_hp* hp_adamw, float max_norm,
                                  float* total_norm_out, float* clip_scale_out, const opt_tensor* tensors, int32_t n,
                                  void* workspace, size_t workspace_bytes, void* stream) {
  const ClipPlan clip{max_norm, total_norm_out, clip_scale_out};
  return mixed_impl(hp_muon, hp_adamw, tensors, n, OPT_KIND_AUTO, workspace, workspace_bytes, stream, &clip);
}

opt_status opt_shard_plan(const opt_tensor* tensors, int32_t n, int32_t routing, int32_t world_size,
                          int64_t align_elems, opt_shard_entry* entries, int64_t* rank_bounds,
                          double* rank_muon_work) {
  if (world_size < 1 || align_elems < 1 || (n > 0 && !entries) || !rank_bounds) return OPT_ERR_INVALID_ARG;
  if (routing != OPT_KIND_AUTO && routing != OPT_KIND_ADAMW && routing != OPT_KIND_MUON) return OPT_ERR_INVALID_ARG;
  if (n < 0 || (n > 0 && !tensors)) return OPT_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const opt_tensor& t = tensors[i];
    if (t.kind != OPT_KIND_AUTO && t.kind != OPT_KIND_ADAMW && t.kind != OPT_KIND_MUON) return OPT_ERR_INVALID_ARG;
    const opt_status st = check_shape(t, routes_to_muon(t, routing));   // shapes only: pointers may be null
    if (st != OPT_OK) return st;
  }
  // AdamW: one index space in list order, cut into aligned, near-equal ranges
  int64_t N = 0;
  std::vector<double> work(static_cast<size_t>(world_size), 0.0);
  std::vector<int32_t> muon_ids;
  for (int32_t i = 0; i < n; ++i) {
    const opt_tensor& t = tensors[i];
    entries[i] = opt_shard_entry{-1, 0, -1};
    const int64_t numel = t.rows * t.cols;
    if (routes_to_muon(t, routing)) {
      if (numel > 0) muon_ids.push_back(i);
    } else {
      // each tensor starts on an alignment boundary, so that every cut inside
      // it falls at a multiple of align_elems of its own elements
      N = (N + align_elems - 1) / align_elems * align_elems;
      entries[i].flat_begin = N;
      N += numel;
    }
  }
  rank_bounds[0] = 0;
  for (int32_t r = 1; r < world_size; ++r) {
    // r * N / world_size without overflow, then rounded up to the alignment
    const int64_t q = N / world_size, rem = N % world_size;
    const int64_t even = q * r + (rem * r) / world_size;
    int64_t b = (even + align_elems - 1) / align_elems * align_elems;
    if (b > N) b = N;
    if (b < rank_bounds[r - 1]) b = rank_bounds[r - 1];
    rank_bounds[r] = b;
  }
  rank_bounds[world_size] = N;
  // Muon: LPT on the Newton-Schulz work of one iteration, 2 (2 A^2 B + A^3)
  auto ns_work = [&](int32_t i) {
    const double R = static_cast<double>(tensors[i].rows), C = static_cast<double>(tensors[i].cols);
    const double A = R < C ? R : C, B = R < C ? C : R;
    return 2.0 * (2.0 * A * A * B + A * A * A);
  };
  std::stable_sort(muon_ids.begin(), muon_ids.end(),
                   [&](int32_t a, int32_t b) { return ns_work(a) > ns_work(b); });
  for (int32_t i : muon_ids) {
    int32_t best = 0;
    for (int32_t r = 1; r < world_size; ++r)
      if (work[static_cast<size_t>(r)] < work[static_cast<size_t>(best)]) best = r;
    entries[i].owner = best;
    work[static_cast<size_t>(best)] += ns_work(i);
  }
  if (rank_muon_work)
    for (int32_t r = 0; r < world_size; ++r) rank_muon_work[r] = work[static_cast<size_t>(r)];
  return OPT_OK;
}

opt_status opt_ns_plan(int64_t rows, int64_t cols, const opt_muon_hp* hp, int32_t* group_sizes, int32_t capacity,
                       int32_t* n_groups) {
  if (!group_sizes || !n_groups || rows < 1 || cols < 1) return OPT_ERR_INVALID_ARG;
  opt_status st = check_muon_hp(hp);
  if (st != OPT_OK) return st;
  const MuonPlanHp ph = plan_hp(*hp, nullptr);
  const int ns_steps = ph.no_ortho ? 0 : ph.ns_steps;
  if (capacity < ns_steps) return OPT_ERR_INVALID_ARG;
  int64_t A, B, Ap, Bp;
  shape_of(rows, cols, A, B, Ap, Bp);
  MuonScalars s{};
  fill_schedule(ph, s);
  const std::vector<int> sizes = fp16_safe_groups(ns_group_sizes(ns_steps, wants_grouped(ph, A, B)), s, ns_steps);
  for (size_t k = 0; k < sizes.size(); ++k) group_sizes[k] = sizes[k];
  *n_groups = static_cast<int32_t>(sizes.size());
  return OPT_OK;
}

opt_status opt_copy_from_host(void* dst, const void* src, size_t bytes, void* stream) {
  if (bytes == 0) return OPT_OK;
  if (!dst || !src) return OPT_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 3u) || (bytes & 3u))
    return OPT_ERR_MISALIGNED;
  cudaPointerAttributes sa{}, da{};
  if (cudaPointerGetAttributes(&sa, src) != cudaSuccess || cudaPointerGetAttributes(&da, dst) != cudaSuccess) {
    cudaGetLastError();
    return OPT_ERR_INVALID_ARG;
  }
  if (sa.type != cudaMemoryTypeHost || sa.devicePointer == nullptr) return OPT_ERR_INVALID_ARG;
  if (da.type != cudaMemoryTypeDevice && da.type != cudaMemoryTypeManaged) return OPT_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || da.device != dev) return OPT_ERR_INVALID_ARG;
  const cudaError_t e = launch_copy_from_host(dst, sa.devicePointer, bytes, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? OPT_OK : cuda_fail(e, "copy from host");
}

opt_status opt_reload_model_params(const opt_tensor* tensors, int32_t n, void* stream) {
  if (n < 0 || (n > 0 && !tensors)) return OPT_ERR_INVALID_ARG;
  for (int32_t i = 0; i < n; ++i) {
    const opt_tensor& t = tensors[i];
    if (t.rows < 0 || t.cols < 0) return OPT_ERR_INVALID_ARG;
    if (t.rows > 0 && t.cols > (INT64_MAX / t.rows)) return OPT_ERR_INVALID_ARG;
    if (t.rows * t.cols == 0 || !t.model_param) continue;
    if (!t.main_param) return OPT_ERR_INVALID_ARG;
    if (check_fp32_ptr(t.main_param) != OPT_OK || (reinterpret_cast<uintptr_t>(t.model_param) & 1u))
      return OPT_ERR_MISALIGNED;
  }
  static thread_local ReloadBatch batch;
  batch.n = 0;
  batch.total_chunks = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  for (int32_t i = 0; i <= n; ++i) {
    const bool flush = (i == n) || batch.n == kReloadBatch;
    if (flush && batch.n > 0) {
      const cudaError_t e = launch_reload(batch, s);
      if (e != cudaSuccess) return cuda_fail(e, "reload model params");
      batch.n = 0;
      batch.total_chunks = 0;
    }
    if (i == n) break;
    const opt_tensor& t = tensors[i];
    const int64_t numel = t.rows * t.cols;
    if (numel == 0 || !t.model_param) continue;
    batch.t[batch.n] = ReloadDesc{t.model_param, t.main_param, numel, batch.total_chunks};
    batch.total_chunks += (numel + kAdamwChunk - 1) / kAdamwChunk;
    ++batch.n;
  }
  return OPT_OK;
}

// opt_newton_schulz; `stall` is the self-test of the bounded device waits
static opt_status newton_schulz_impl(const float* G, float* O, int64_t rows, int64_t cols, int32_t ns_steps,
                                     float a, float b, float c, float eps, void* workspace, size_t workspace_bytes,
                                     void* stream, int stall) {
  if (rows < 0 || cols < 0 || ns_steps < 0 || ns_steps > 16) return OPT_ERR_INVALID_ARG;
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c) || !std::isfinite(eps) || eps < 0.f)
    return OPT_ERR_INVALID_ARG;
  if (rows > (int64_t(1) << 30) || cols > (int64_t(1) << 30)) return OPT_ERR_UNSUPPORTED;
  if (rows * cols == 0) return OPT_OK;
  if (!G || !O) return OPT_ERR_INVALID_ARG;
  if (check_fp32_ptr(G) != OPT_OK || check_fp32_ptr(O) != OPT_OK) return OPT_ERR_MISALIGNED;
  opt_tensor t{};
  t.main_param = O;
  t.main_grad = G;
  t.exp_avg = O;
  t.rows = rows;
  t.cols = cols;
  t.ndim = 2;
  t.kind = OPT_KIND_MUON;
  std::vector<const opt_tensor*> one{&t};
  const std::vector<ShapeClass> classes = shape_classes(one);
  opt_status st = check_workspace(workspace, workspace_bytes, min_bytes(classes));
  if (st != OPT_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaError_t e = cudaMemsetAsync(ws, 0, kHeaderBytes, s);
  if (e != cudaSuccess) return cuda_fail(e, "workspace header");
  MuonPlanHp hp{0.f, 0.f, 0.f, eps, a, b, c, 0.f, 0, ns_steps, 1};
  hp.stall = stall;
  float* outs[1] = {O};
  return run_muon_class(hp, classes[0], ws + kHeaderBytes, workspace_bytes - kHeaderBytes,
                        reinterpret_cast<uint32_t*>(ws), s, outs);
}

opt_status opt_newton_schulz(const float* G, float* O, int64_t rows, int64_t cols, int32_t ns_steps, float a,
                             float b, float c, float eps, void* workspace, size_t workspace_bytes, void* stream) {
  return newton_schulz_impl(G, O, rows, cols, ns_steps, a, b, c, eps, workspace, workspace_bytes, stream, 0);
}

opt_status opt_selftest_wait_timeout(const float* G, float* O, int64_t rows, int64_t cols, void* workspace,
                                     size_t workspace_bytes, void* stream) {
  return newton_schulz_impl(G, O, rows, cols, 5, 3.4445f, -4.7750f, 2.0315f, 1e-7f, workspace, workspace_bytes,
                            stream, 1);
}

opt_status opt_device_status(const void* workspace, void* stream) {
  if (!workspace) return OPT_ERR_WORKSPACE;
  uint32_t code = 0;
  cudaError_t e = cudaMemcpyAsync(&code, workspace, sizeof(code), cudaMemcpyDeviceToHost,
                                  static_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "device status");
  return code == 0 ? OPT_OK : OPT_ERR_DEVICE_TIMEOUT;
}

const char* opt_strerror(opt_status s) {
  switch (s) {
    case OPT_OK: return "ok";
    case OPT_ERR_INVALID_ARG: return "invalid argument";
    case OPT_ERR_UNSUPPORTED: return "unsupported case";
    case OPT_ERR_MISALIGNED: return "misaligned pointer";
    case OPT_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case OPT_ERR_CUDA: return "CUDA error";
    case OPT_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
  }
  return "unknown status";
}

const char* opt_last_cuda_error(void) { return g_last_cuda_error; }

opt_status opt_profile_launches(void* const* events, opt_launch_info* info, int32_t capacity, int32_t* count) {
  if (!events || !count) {
    g_prof = ProfState{};
    return OPT_OK;
  }
  if (capacity < 0 || (capacity > 0 && !info)) return OPT_ERR_INVALID_ARG;
  g_prof.events = reinterpret_cast<cudaEvent_t const*>(events);
  g_prof.info = info;
  g_prof.capacity = capacity;
  g_prof.count = count;
  g_prof.open = -1;
  return OPT_OK;
}

int32_t opt_abi_version(void) { return (2 << 16) | 0; }

}  // extern "C"

// ------------------------------------------------- allocation-free variant --
//
// opt_newton_schulz_noalloc: Newton-Schulz for callers that cannot allocate
// device memory and cannot hand the library a workspace -- for example code
// hosted by a runtime that owns every device allocation and gives extensions
// no allocator, or a path with a fixed memory budget where an allocation would
// fail or stall.  Its scratch is the file-scope device array below, sized for
// one matrix with min(rows, cols) <= 1024 and max(rows, cols) <= 4096 (padded
// Newton-Schulz buffers of 1024 x 4096 plus the 256-byte status header, 20 MiB).
// The array exists on every GPU that loads this library, from module load until
// the process exits.  In host code its name is a host-side stand-in, not a
// device address, so each device's address is taken once with
// cudaGetSymbolAddress (with that device current) and only that address is
// handed to kernels.

namespace mpopt {
namespace {

constexpr int64_t kNoallocMaxMin = 1024;   // largest min(rows, cols)
constexpr int64_t kNoallocMaxMax = 4096;   // largest max(rows, cols)

constexpr size_t noalloc_align(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }
// The same buffer layout as group_layout() for one kNoallocMaxMin x
// kNoallocMaxMax matrix (both already multiples of the 256 padding), after the
// status header.
constexpr size_t kNoallocScratchBytes =
    kHeaderBytes + 2 * noalloc_align(kNoallocMaxMin * kNoallocMaxMax * 2) +   // X x2 (ping-pong)
    2 * noalloc_align(kNoallocMaxMin * kNoallocMaxMin * 2) +                  // A fp16, C fp16
    noalloc_align(static_cast<size_t>(partials_per_matrix(kNoallocMaxMin, kNoallocMaxMax, kNoallocMaxMin,
                                                          kNoallocMaxMax)) * 4) +
    noalloc_align(kMatStats * 4);

}  // namespace

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

namespace {

constexpr int kNoallocMaxDevices = 64;
std::mutex g_noalloc_mu;
// Per device: the array's address and the id of the CUDA context it belongs
// to.  A context that is torn down (cudaDeviceReset) and created again gets a
// new id, and with it a new copy of the array at a possibly different address.
struct NoallocSlot {
  uint8_t* base;
  unsigned long long ctx_id;
};
NoallocSlot g_noalloc[kNoallocMaxDevices] = {};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the context current on this thread (driver entry points, so the
// library keeps linking only the runtime); 0 if there is none or the driver
// cannot tell.
unsigned long long current_context_id() {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

// Device address of the scratch array on the current device.  The address is
// looked up (under a lock) on the first call on each device, and again whenever
// the device's context has changed since -- after a cudaDeviceReset the old
// address is stale.  Without a context id from the driver it is looked up on
// every call.
opt_status noalloc_scratch(uint8_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "noalloc: current device");
  if (dev < 0 || dev >= kNoallocMaxDevices) return OPT_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  NoallocSlot& slot = g_noalloc[dev];
  const unsigned long long id = current_context_id();
  if (!slot.base || id == 0 || id != slot.ctx_id) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);   // creates the context if there is none yet
    if (e != cudaSuccess) return cuda_fail(e, "noalloc: scratch symbol address");
    if (reinterpret_cast<uintptr_t>(p) & 255u) return OPT_ERR_WORKSPACE;
    slot.base = static_cast<uint8_t*>(p);
    slot.ctx_id = id ? id : current_context_id();
  }
  *out = slot.base;
  return OPT_OK;
}

}  // namespace
}  // namespace mpopt

extern "C" opt_status opt_newton_schulz_noalloc(const float* G, float* O, int64_t rows, int64_t cols,
                                                 int32_t ns_steps, float a, float b, float c, float eps,
                                                 void* stream) {
  using namespace mpopt;
  if (rows < 0 || cols < 0 || ns_steps < 0 || ns_steps > 16) return OPT_ERR_INVALID_ARG;
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c) || !std::isfinite(eps) || eps < 0.f)
    return OPT_ERR_INVALID_ARG;
  if (rows * cols == 0) return OPT_OK;
  const int64_t mn = rows < cols ? rows : cols, mx = rows < cols ? cols : rows;
  if (mn > kNoallocMaxMin || mx > kNoallocMaxMax) {
    std::snprintf(g_last_cuda_error, sizeof(g_last_cuda_error),
                  "opt_newton_schulz_noalloc: %lldx%lld exceeds the built-in scratch (min side <= %lld, "
                  "max side <= %lld); use opt_newton_schulz with a workspace",
                  static_cast<long long>(rows), static_cast<long long>(cols),
                  static_cast<long long>(kNoallocMaxMin), static_cast<long long>(kNoallocMaxMax));
    return OPT_ERR_UNSUPPORTED;
  }
  if (!G || !O) return OPT_ERR_INVALID_ARG;
  if (check_fp32_ptr(G) != OPT_OK || check_fp32_ptr(O) != OPT_OK) return OPT_ERR_MISALIGNED;
  opt_tensor t{};
  t.main_param = O;
  t.main_grad = G;
  t.exp_avg = O;
  t.rows = rows;
  t.cols = cols;
  t.ndim = 2;
  t.kind = OPT_KIND_MUON;
  std::vector<const opt_tensor*> one{&t};
  const std::vector<ShapeClass> classes = shape_classes(one);
  if (kHeaderBytes + group_bytes(1, rows, cols, false) > kNoallocScratchBytes) return OPT_ERR_WORKSPACE;
  uint8_t* base = nullptr;
  opt_status st = noalloc_scratch(&base);
  if (st != OPT_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = cudaMemsetAsync(base, 0, kHeaderBytes, s);   // status word starts at zero
  if (e != cudaSuccess) return cuda_fail(e, "noalloc: status header");
  MuonPlanHp hp{0.f, 0.f, 0.f, eps, a, b, c, 0.f, 0, ns_steps, 1};
  hp.ns_order = OPT_MUON_NS_PER_ITERATION;   // the built-in scratch holds one iteration's buffers
  float* outs[1] = {O};
  return run_muon_class(hp, classes[0], base + kHeaderBytes, kNoallocScratchBytes - kHeaderBytes,
                        reinterpret_cast<uint32_t*>(base), s, outs);
}

extern "C" opt_status opt_noalloc_device_status(void* stream) {
  using namespace mpopt;
  uint8_t* base = nullptr;
  const opt_status st = noalloc_scratch(&base);
  if (st != OPT_OK) return st;
  return opt_device_status(base, stream);
}
