/*
 * mpopt.h -- C ABI of the GB300 mixed-precision optimizer step (libmpopt.so).
 *
 * One optimizer step over fp32 master weights ("main_param"), fp32 reduced
 * gradients ("main_grad") and fp32 optimizer state, ending with the bf16 copy
 * of every master weight written back to the model:
 *
 *   - AdamW for every tensor routed to it (opt_adamw_step), as defined in
 *     "02 · Optimizer：算法与 infra" §2 (Adam, bias correction, eps outside the
 *     square root) and §3 (decoupled weight decay, AdamW Algorithm 2);
 *   - Muon for 2-D hidden matrices (opt_muon_step), as defined in the same
 *     page §1 (momentum and Nesterov as lerp), §5.2 (Newton-Schulz quintic),
 *     §5.4 (decoupled decay, Eq. 3; update scaled by 0.2*sqrt(max(A, B)),
 *     Eq. 4), and in "优化器：AdamW、Muon 与分布式优化器", Muon section;
 *   - both at once with the routing rule of §5.5 / §14.2 (opt_mixed_step):
 *     a tensor is a Muon tensor when it is 2-D and not an embedding or an
 *     output (LM head) parameter; every other tensor goes to AdamW;
 *   - the bf16 writeback of §9.2 ("参数写回": master -> model copy), done in
 *     the same kernels, round-to-nearest-even.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every data pointer is a DEVICE pointer owned by the caller (for example
 *    torch.Tensor.data_ptr()).  The library allocates nothing and keeps no
 *    state between calls: optimizer state lives in the caller's buffers and
 *    scratch space in the caller's workspace.
 *  - Updates are in place.  Tensors are dense, row-major, element-contiguous.
 *    fp32 pointers must be 4-byte aligned and bf16 pointers 2-byte aligned;
 *    any other alignment is handled (unaligned heads and tails take a scalar
 *    path).  Tensors in one call must not overlap.
 *  - Work is enqueued on `stream` (a cudaStream_t; NULL is the legacy default
 *    stream) and runs asynchronously.  Argument errors are detected on the host
 *    before anything is enqueued and return a status; nothing runs then.
 *    A failed launch returns OPT_ERR_CUDA (the CUDA error text is available
 *    from opt_last_cuda_error()).
 *  - Device-side waits in the tensor-core kernels are bounded in time.  A wait
 *    that runs out records a code in the workspace header; opt_device_status()
 *    reads it.  Each step clears the header first.
 *  - Thread safety: calls that share a workspace must be serialised on one
 *    stream.
 */
#ifndef MPOPT_H
#define MPOPT_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MPOPT_API __attribute__((visibility("default")))
#else
#define MPOPT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OPT_OK = 0,
  OPT_ERR_INVALID_ARG = 1,   /* null pointer, bad size/shape/hyper-parameter  */
  OPT_ERR_UNSUPPORTED = 2,   /* a case this library does not implement        */
  OPT_ERR_MISALIGNED = 3,    /* fp32 pointer not 4-byte / bf16 not 2-byte aligned */
  OPT_ERR_WORKSPACE = 4,     /* workspace null, too small or not 256-B aligned */
  OPT_ERR_CUDA = 5,          /* a CUDA runtime/driver call or launch failed    */
  OPT_ERR_DEVICE_TIMEOUT = 6 /* a bounded device-side wait ran out (device status) */
} opt_status;

/* Routing of one tensor (opt_tensor.kind). */
enum {
  OPT_KIND_AUTO = 0,   /* opt_mixed_step decides: Muon iff ndim == 2 and not
                          flagged OPT_FLAG_EMBEDDING_OR_OUTPUT                  */
  OPT_KIND_ADAMW = 1,
  OPT_KIND_MUON = 2
};

/* opt_tensor.flags */
enum { OPT_FLAG_EMBEDDING_OR_OUTPUT = 1 };

/* OR into opt_workspace_size's `routing` to size a workspace for
   opt_mixed_step_clipped (adds one float per 16K gradient elements). */
enum { OPT_WORKSPACE_CLIP = 0x10 };
/* OR into opt_workspace_size's `routing` to size the Newton-Schulz buffers of
   every shape for grouped iterations (opt_muon_hp.flags OPT_MUON_NS_GROUPED);
   without it only the shapes grouped by default get their two extra buffers. */
enum { OPT_WORKSPACE_GROUPED = 0x20 };

/*
 * AdamW hyper-parameters for one step ("02 · Optimizer：算法与 infra" §2, §3).
 *   lr            eta, the step size
 *   beta1, beta2  EMA factors of the first and second raw moments, in [0, 1)
 *   eps           added OUTSIDE the square root: mhat / (sqrt(vhat) + eps)
 *   weight_decay  lambda, decoupled: theta <- theta * (1 - lr*lambda) - lr*update
 *   step          t >= 1, the number of this step (bias corrections 1 - beta^t)
 * The per-step scalars 1-beta1, 1-beta2, 1-beta1^t, 1-beta2^t and 1-lr*lambda are
 * formed in double precision from these values and rounded once to float; each
 * element is then evaluated in fp32 in the order written above, every operation
 * rounded to nearest (no fused multiply-add).
 */
typedef struct {
  float lr;
  float beta1;
  float beta2;
  float eps;
  float weight_decay;
  int32_t reserved;
  int64_t step;
} opt_adamw_hp;

/*
 * Muon hyper-parameters ("02 · Optimizer：算法与 infra" §1, §5.2, §5.4, §14.1,
 * §14.6).
 *   lr            eta
 *   momentum      mu in [0, 1): m <- lerp(m, g, 1 - mu)
 *   weight_decay  lambda, decoupled, applied to W_{t-1}
 *   eps           Newton-Schulz normalisation X = G / (||G||_F + eps); 1e-7
 *   nesterov      nonzero: Newton-Schulz input lerp(g, m, mu); zero: m
 *   ns_steps      number of quintic iterations, 0..16 (5 on the pages)
 *   ns_a, ns_b, ns_c  quintic coefficients, (3.4445, -4.7750, 2.0315), used
 *                 for every iteration unless ns_schedule is given
 *   scale_coeff   free factor k of the update scale (0.2 on the pages)
 *   scale_mode    OPT_SCALE_SPECTRAL: k * sqrt(max(m, n)) (the default, §5.4
 *                 Eq. 4); OPT_SCALE_SHAPE: k * sqrt(max(1, m / n));
 *                 OPT_SCALE_UNIT_RMS: k * sqrt(m / n) (§14.6), where
 *                 m = rows (fan_out) and n = cols (fan_in) of the parameter
 *   flags         OPT_MUON_NO_ORTHOGONALIZE: plain momentum SGD,
 *                 W <- W (1 - lr lambda) - lr * k * gtilde (§1), no Newton-Schulz;
 *                 evaluation order of the iterations (at most one of):
 *                 OPT_MUON_NS_PER_ITERATION: every iteration as printed
 *                 (A = X X^T, C = a I + b A + c A A, X <- C X);
 *                 OPT_MUON_NS_GROUPED: up to three consecutive iterations
 *                 share one X X^T and one C X.  Every C_k is a polynomial in
 *                 the group's first Gram matrix, so A_{k+1} = C_k (A_k C_k)
 *                 and X_{k+g} = (C_{k+g-1} ... C_k) X_k hold exactly; only
 *                 the rounding differs.  Used for every shape whose workspace
 *                 group has room for two more fp16 [A][A] buffers per matrix.
 *                 Neither flag (the default): grouped for the shapes where it
 *                 saves tensor-core work (padded max side >= 2 x padded min
 *                 side, min side >= 1024, e.g. 4096 x 14336), per iteration
 *                 otherwise
 *   ns_schedule   optional HOST array of ns_steps triples (a, b, c), one per
 *                 iteration in order (a coefficient schedule); NULL: ns_a..c
 */
typedef struct {
  float lr;
  float momentum;
  float weight_decay;
  float eps;
  int32_t nesterov;
  int32_t ns_steps;
  float ns_a;
  float ns_b;
  float ns_c;
  float scale_coeff;
  int32_t scale_mode;
  int32_t flags;
  const float* ns_schedule;
} opt_muon_hp;

enum { OPT_SCALE_SPECTRAL = 0, OPT_SCALE_SHAPE = 1, OPT_SCALE_UNIT_RMS = 2 };
enum { OPT_MUON_NO_ORTHOGONALIZE = 1, OPT_MUON_NS_PER_ITERATION = 2, OPT_MUON_NS_GROUPED = 4 };

/*
 * One parameter tensor.
 *   main_param   fp32 [rows*cols]   master weights, updated in place
 *   main_grad    fp32 [rows*cols]   this step's gradient, read only
 *   exp_avg      fp32 [rows*cols]   AdamW first moment m / Muon momentum buffer
 *   exp_avg_sq   fp32 [rows*cols]   AdamW second moment v; ignored for Muon
 *   model_param  bf16 [rows*cols]   written with the rounded master; NULL means
 *                                   the model parameter is itself fp32 (it IS
 *                                   main_param) and nothing is written back
 *   rows, cols   the shape; a 1-D tensor of n elements is rows = 1, cols = n,
 *                ndim = 1.  Muon requires ndim == 2, rows >= 1, cols >= 1.
 *                rows*cols == 0 is allowed and does nothing.
 *   ndim         the parameter's dimensionality (used by OPT_KIND_AUTO)
 *   kind, flags  routing, see above
 *   scale_rows, scale_cols  Muon only: the shape whose (fan_out, fan_in) set
 *                the update scale; 0, 0 means this tensor's own shape.  A block
 *                of a split parameter (QKV split, "02 · Optimizer：算法与 infra"
 *                §5.5 / §14.4: Q, K and V rows orthogonalised separately) is
 *                passed as its own row-block view with the whole parameter's
 *                shape here.
 */
typedef struct {
  float* main_param;
  const float* main_grad;
  float* exp_avg;
  float* exp_avg_sq;
  uint16_t* model_param;
  int64_t rows;
  int64_t cols;
  int32_t ndim;
  int32_t kind;
  int32_t flags;
  int32_t reserved;
  int64_t scale_rows;
  int64_t scale_cols;
} opt_tensor;

/*
 * Bytes of device workspace that opt_mixed_step (and the other steps) need for
 * this tensor list: a 256-byte status header and the Newton-Schulz buffers of
 * the largest group of same-shape Muon matrices (the fp16 iterate twice, as a
 * ping-pong pair, the fp16 Gram matrix, the fp16 polynomial a I + b A + c A A,
 * norm partials; for the shapes that take grouped iterations by default, two
 * more fp16 [A][A] buffers).  Shapes are padded to multiples of 256.
 * AdamW needs no workspace: 0 for a list without Muon tensors.
 * `routing` selects how kinds are interpreted: OPT_KIND_AUTO as in
 * opt_mixed_step, OPT_KIND_ADAMW treats every tensor as AdamW, OPT_KIND_MUON
 * every tensor as Muon.  Returns 0 if the list is invalid.
 * A smaller workspace is accepted by the Muon path as long as one matrix of
 * each shape fits without the grouped-iteration buffers; matrices are then
 * processed in smaller groups, and without grouped iterations when not even
 * one matrix fits with their buffers.
 */
MPOPT_API size_t opt_workspace_size(const opt_tensor* tensors, int32_t n, int32_t routing);

/*
 * AdamW step over a list of n tensors (n >= 0): a multi-tensor kernel over
 * 16K-element chunks whose tensor table travels in the kernel's parameter
 * space, one launch per 400 tensors.  kind/flags are ignored.  exp_avg_sq
 * must be non-null.  No workspace is needed (workspace may be NULL).
 */
MPOPT_API opt_status opt_adamw_step(const opt_adamw_hp* hp, const opt_tensor* tensors, int32_t n,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * Muon step for one 2-D matrix t (t->ndim must be 2): momentum, Nesterov,
 * Newton-Schulz on the wide orientation (transposed when rows > cols),
 * W <- W (1 - lr*lambda) - lr * scale_coeff * sqrt(max(rows, cols)) * O, and
 * bf16 writeback.  exp_avg is the momentum buffer; exp_avg_sq is ignored.
 */
MPOPT_API opt_status opt_muon_step(const opt_muon_hp* hp, const opt_tensor* t,
                         void* workspace, size_t workspace_bytes, void* stream);

/*
 * The whole mixed step: routes each tensor (kind/flags), runs one AdamW
 * launch over all AdamW tensors, and Muon over all Muon matrices, batching
 * matrices of the same (min, max) shape into shared tensor-core launches.
 * hp_muon may be NULL when no tensor routes to Muon, hp_adamw when none
 * routes to AdamW.
 */
MPOPT_API opt_status opt_mixed_step(const opt_muon_hp* hp_muon, const opt_adamw_hp* hp_adamw,
                          const opt_tensor* tensors, int32_t n,
                          void* workspace, size_t workspace_bytes, void* stream);

/*
 * opt_mixed_step with global gradient-norm clipping fused in front
 * ("02 · Optimizer：算法与 infra" §11.1; §11.4: one norm over the gradients of
 * both optimizer groups):
 *   total_norm = sqrt(sum over every tensor of ||main_grad||^2)
 *   clip_coeff = max_norm / (total_norm + 1e-6)
 *   every gradient is multiplied by clip_coeff when clip_coeff < 1.
 * The factor is computed on the device (fp32 sums of squares per 16K-element
 * chunk, added in double in a fixed order) and applied by the AdamW and Muon
 * kernels as they load each gradient; main_grad itself is not rewritten.
 * max_norm <= 0 disables clipping (no norm pass, outputs untouched).
 * total_norm_out and clip_scale_out are optional 4-byte-aligned DEVICE fp32
 * pointers receiving the norm and the factor applied.  Workspace:
 * opt_workspace_size(tensors, n, OPT_KIND_AUTO | OPT_WORKSPACE_CLIP).
 */
MPOPT_API opt_status opt_mixed_step_clipped(const opt_muon_hp* hp_muon, const opt_adamw_hp* hp_adamw, float max_norm,
                                            float* total_norm_out, float* clip_scale_out, const opt_tensor* tensors,
                                            int32_t n, void* workspace, size_t workspace_bytes, void* stream);

/*
 * main_param <- fp32(model_param) for every tensor that has a bf16 model copy
 * ("02 · Optimizer：算法与 infra" §9.2 reload_model_params: refresh the masters
 * after the model copy was changed from outside; "支持FP32优化器" §9.3-§9.4:
 * the plain-checkpoint and model-only restore branches).  Exact (bf16 widens
 * to fp32 without rounding).  fp32-native tensors (model_param NULL) are left
 * alone.  Only main_param, model_param and the shape are read; no workspace.
 * Note the fp32 tail the masters had is not recoverable this way: a resume
 * that must continue bit for bit restores main_param itself.
 */
MPOPT_API opt_status opt_reload_model_params(const opt_tensor* tensors, int32_t n, void* stream);

/*
 * Data-parallel sharding of one optimizer step over `world_size` ranks
 * ("02 · Optimizer：算法与 infra" §12.1-§12.2 and §14.3; "优化器：AdamW、Muon 与
 * 分布式优化器", distributed Muon, scheme ③).  Host-only: no device work, no
 * CUDA call; every rank computes the same plan from the same tensor list.
 *
 *   - AdamW tensors (the routing of opt_mixed_step, with `routing` as in
 *     opt_workspace_size) are laid end to end, in list order, in one index
 *     space of N elements, each starting at a multiple of `align_elems` (>= 1;
 *     the gaps belong to no tensor), which is cut into world_size contiguous
 *     ranges, ZeRO-1 style: rank r owns [rank_bounds[r], rank_bounds[r+1]).
 *     The cuts ignore tensor boundaries (a tensor may span ranks); every inner
 *     cut is a multiple of `align_elems`, so it falls at a multiple of
 *     `align_elems` of the tensor's own elements, and the ranges are as equal
 *     as that allows: rank_bounds[r] = min(N, round_up(r * N / world_size,
 *     align_elems)).
 *     Rank r steps only the elements it owns, with fp32 master, m and v of
 *     that size, and then every rank receives the bf16 values of the rest.
 *   - Muon tensors stay whole (Newton-Schulz needs the whole matrix): each has
 *     one owner rank, assigned by LPT bin-packing on its Newton-Schulz work
 *     2 (2 A^2 B + A^3) per iteration (largest first; each goes to the rank
 *     with the least work so far, the lowest rank on ties; equal sizes keep
 *     list order), so the plan is deterministic.
 *
 * Output, caller-owned host memory:
 *   entries[n]            per tensor: owner = the owning rank (Muon) or -1
 *                         (AdamW; and for empty tensors); flat_begin = the
 *                         tensor's first index in the AdamW index space
 *                         (AdamW) or -1 (Muon)
 *   rank_bounds[world_size + 1]   the AdamW ranges (rank_bounds[0] = 0,
 *                         rank_bounds[world_size] = N)
 *   rank_muon_work[world_size]    optional (NULL: not written): the
 *                         Newton-Schulz flops per iteration each rank owns
 * Only shapes, kinds and flags are read: the tensors' pointers may be null
 * (on a sharded rank the master and state of what it does not own need not
 * exist).  Errors: OPT_ERR_INVALID_ARG for world_size < 1, align_elems < 1,
 * null outputs, or a shape or kind opt_mixed_step would reject.
 */
typedef struct {
  int32_t owner;
  int32_t reserved;
  int64_t flat_begin;
} opt_shard_entry;

MPOPT_API opt_status opt_shard_plan(const opt_tensor* tensors, int32_t n, int32_t routing, int32_t world_size,
                                    int64_t align_elems, opt_shard_entry* entries, int64_t* rank_bounds,
                                    double* rank_muon_work);

/*
 * How opt_muon_step / opt_mixed_step evaluate the Newton-Schulz iterations of
 * one rows x cols matrix under `hp` (host only: nothing is launched, no GPU is
 * needed).  Writes the size of each group of consecutive iterations that
 * share one X X^T and one C X, in order (all 1: every iteration as written),
 * into group_sizes[0 .. *n_groups) and their count into *n_groups; the sizes
 * add up to hp->ns_steps.  The plan assumes a workspace from
 * opt_workspace_size (with OPT_WORKSPACE_GROUPED when hp->flags has
 * OPT_MUON_NS_GROUPED): a workspace without room for the grouped buffers
 * evaluates every iteration as written.
 * Grouping follows hp->flags (see opt_muon_hp), in groups of at most three,
 * and splits a group into single iterations when the product of its
 * polynomials could leave fp16's range: each iteration's largest |a + b l +
 * c l^2| over the squared singular values it can reach (from [0, 1] after the
 * normalisation, through the per-singular-value form of the iteration,
 * "02 · Optimizer：算法与 infra" §5.2) is multiplied over the group, and
 * groups above 4096 are split (the printed coefficients give about 42).
 * Errors: OPT_ERR_INVALID_ARG for a null pointer, an invalid hp, rows or cols
 * below 1, or capacity below hp->ns_steps.
 */
MPOPT_API opt_status opt_ns_plan(int64_t rows, int64_t cols, const opt_muon_hp* hp, int32_t* group_sizes,
                                 int32_t capacity, int32_t* n_groups);

/*
 * Copies `bytes` from page-locked host memory `src` (cudaHostAlloc, or
 * registered with cudaHostRegister) to device memory `dst` of the current
 * device, enqueued on `stream`, with a kernel whose threads load the host
 * buffer over the CPU-GPU link and store to device memory (32 CTAs, no
 * shared memory: it runs beside the optimizer's kernels on another stream
 * and leaves most SMs to them).  No counterpart on the pages: it serves callers whose gradients
 * arrive in host memory.  On GB300 hosts the copy engines' host-to-device
 * rate (cudaMemcpyAsync) from page-locked memory varies with the pages and
 * over time, down to 13-40 GB/s on some buffers of some hosts, while loads by
 * the SMs keep about 210 GB/s.
 *   dst, src  4-byte aligned (16-byte aligned for the vector path), not
 *             overlapping; bytes a multiple of 4.
 * Errors: OPT_ERR_INVALID_ARG for null pointers, a src that is not
 * page-locked host memory, or a dst that is not device memory of the current
 * device; OPT_ERR_MISALIGNED for the alignment rules; OPT_ERR_CUDA if the
 * launch fails.  bytes == 0 does nothing.
 */
MPOPT_API opt_status opt_copy_from_host(void* dst, const void* src, size_t bytes, void* stream);

/*
 * Newton-Schulz orthogonalisation alone ("02 · Optimizer：算法与 infra" §5.2):
 * O = NS_steps(G) for one fp32 rows x cols matrix G, same fp16 tensor-core
 * path as opt_muon_step.  G and O are device fp32 [rows*cols]; O may alias G.
 * Workspace: opt_workspace_size of a one-matrix Muon list of that shape.
 */
MPOPT_API opt_status opt_newton_schulz(const float* G, float* O, int64_t rows, int64_t cols,
                             int32_t ns_steps, float a, float b, float c, float eps,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * opt_newton_schulz without a workspace, for callers that cannot allocate
 * device memory: code hosted by a runtime that owns every device allocation
 * and gives extensions no allocator, or a path whose memory budget is fixed in
 * advance.  No counterpart on the pages: this is an interface convenience, the
 * arithmetic is opt_newton_schulz's with every iteration evaluated as written
 * (as with OPT_MUON_NS_PER_ITERATION): the built-in scratch holds the buffers
 * of one iteration, not those of grouped iterations.
 *   - Scratch is a 20 MiB array of device memory built into the library (a
 *     static __device__ array).  Every GPU that loads the library holds it until
 *     the process exits.  This entry point calls no cudaMalloc, cudaFree or
 *     other allocating routine.
 *   - Size limit: min(rows, cols) <= 1024 and max(rows, cols) <= 4096; larger
 *     matrices return OPT_ERR_UNSUPPORTED (text in opt_last_cuda_error()).
 *   - The first call on each device looks up the array's device address there
 *     (cudaGetSymbolAddress with that device current), and so does the first
 *     call after the device's CUDA context was destroyed and created again
 *     (cudaDeviceReset): the library remembers the context's id with the
 *     address.  Make such a first call before any stream capture.
 *   - Every call on a device shares the one array, and the array keeps the last
 *     call's contents (the status word is cleared at the start of each call).
 *     Calls whose work overlaps on the GPU -- on different streams, or from
 *     different threads -- race on it: serialise them on one stream.
 *   - A device-side timeout is recorded in the array's header: read it with
 *     opt_noalloc_device_status() after the call.
 */
MPOPT_API opt_status opt_newton_schulz_noalloc(const float* G, float* O, int64_t rows, int64_t cols,
                                               int32_t ns_steps, float a, float b, float c, float eps,
                                               void* stream);

/*
 * Status of the last opt_newton_schulz_noalloc call on the current device:
 * synchronises `stream` and returns OPT_ERR_DEVICE_TIMEOUT if a kernel of
 * that call recorded a device-side timeout in the built-in array's header,
 * else OPT_OK (OPT_ERR_CUDA if the copy or the synchronisation fails).  Like
 * the call itself, no counterpart on the pages.
 */
MPOPT_API opt_status opt_noalloc_device_status(void* stream);

/*
 * Synchronises `stream` and reports whether a kernel of the last step on this
 * workspace recorded a device-side timeout (OPT_ERR_DEVICE_TIMEOUT) or not
 * (OPT_OK).  Returns OPT_ERR_CUDA if the synchronisation itself fails.
 */
MPOPT_API opt_status opt_device_status(const void* workspace, void* stream);

/*
 * Self-test of the bounded device-side waits (for tests of the failure path).
 * Runs opt_newton_schulz on G (rows x cols; 5 iterations with the quintic
 * coefficients of "02 · Optimizer：算法与 infra" §5.2, eps 1e-7) with one TMA
 * stage of the first X X^T launch withheld: the even CTA of the first CTA pair
 * never signals it, so the MMA issuer's wait for that stage runs out after
 * about 2 s.  The kernel then records the timeout in the workspace header,
 * every role of the CTA pair leaves its loop (each of their waits is bounded
 * too), and the remaining launches run to completion on whatever the buffers
 * hold.  Nothing faults, and the CUDA context and the workspace stay usable:
 * opt_device_status() returns OPT_ERR_DEVICE_TIMEOUT, and the next call on
 * the same workspace clears the header and runs normally.  O receives
 * unspecified values.  Arguments, workspace size (opt_workspace_size of one
 * OPT_KIND_MUON tensor of this shape) and host-side errors are those of
 * opt_newton_schulz.
 */
MPOPT_API opt_status opt_selftest_wait_timeout(const float* G, float* O, int64_t rows, int64_t cols,
                                               void* workspace, size_t workspace_bytes, void* stream);

/*
 * Optional launch instrumentation (off by default).  After
 *   opt_profile_launches(events, info, capacity, &count)
 * every kernel this library launches from the calling thread is bracketed by
 * cudaEventRecord(events[2*i]) and cudaEventRecord(events[2*i+1]) on the
 * launch's stream, and info[i] describes it, for i = count, count+1, ...
 * while count < capacity (count is incremented by the library, also past
 * capacity, so the caller learns how many launches there were).  `events`
 * holds 2*capacity cudaEvent_t created by the caller; `info` and `count` are
 * host memory owned by the caller and must stay valid until
 * opt_profile_launches(NULL, NULL, 0, NULL) switches it off.
 */
typedef struct {
  int32_t kernel;   /* OPT_KERNEL_* */
  int32_t count;    /* matrices (Newton-Schulz, Muon stages) or tensors (AdamW) */
  int64_t a;        /* Newton-Schulz: A = min(rows, cols); AdamW: elements */
  int64_t b;        /* Newton-Schulz: B = max(rows, cols) */
} opt_launch_info;

enum {
  OPT_KERNEL_NS_GRAM = 0,      /* A = X X^T, fp16 tensor cores                   */
  OPT_KERNEL_NS_POLY = 1,      /* C = a I + b A + c A A, fp16 tensor cores       */
  OPT_KERNEL_NS_BX = 2,        /* X' = C X, fp16 tensor cores (last one updates W) */
  OPT_KERNEL_ADAMW = 3,
  OPT_KERNEL_MUON_PREP = 4,    /* momentum, Nesterov, norm partials (and, with
                                  Newton-Schulz, the fp16 iterate)              */
  OPT_KERNEL_MUON_NORM = 5,
  OPT_KERNEL_MUON_APPLY = 6,   /* ns_steps == 0 only                             */
  OPT_KERNEL_MUON_OPERANDS = 7, /* fix-up: normalised fp16 X0 rewritten for the
                                  matrices whose iterate left fp16's range       */
  OPT_KERNEL_GRAD_NORM = 8,     /* clipping: sums of squares of the gradients      */
  OPT_KERNEL_CLIP_FINALIZE = 9, /* clipping: total norm and factor                 */
  OPT_KERNEL_MUON_SAMPLE = 10,  /* per-matrix power-of-two scale of the iterate    */
  OPT_KERNEL_NS_SYM = 11        /* grouped iterations: product of two commuting
                                   symmetric [A][A] matrices, fp16 tensor cores  */
};

MPOPT_API opt_status opt_profile_launches(void* const* events, opt_launch_info* info, int32_t capacity,
                                          int32_t* count);

/* Static text for a status code. */
MPOPT_API const char* opt_strerror(opt_status status);

/* Text of the last CUDA error seen by this thread's calls ("" if none). */
MPOPT_API const char* opt_last_cuda_error(void);

/* ABI version: (major << 16) | minor (2.0: Muon variants, scale shapes, clipping). */
MPOPT_API int32_t opt_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MPOPT_H */
