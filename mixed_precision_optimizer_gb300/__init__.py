"""GB300 mixed-precision optimizer step: Python binding of ``libmpopt.so``.

This module only marshals arguments: it checks dtypes, devices and layouts of
PyTorch tensors, packs their device pointers into the C structs of
``include/mpopt.h`` and calls the library on the current CUDA stream.  Every
step of the optimizer runs in the library's CUDA kernels.  If the library has
not been built, importing works but every call raises ``MpoptUnavailable``.

Entry points (same names as the C ABI, without the ``opt_`` prefix):

* ``adamw_step``      -- AdamW over a list of tensors
* ``muon_step``       -- Muon for one 2-D matrix
* ``mixed_step``      -- both, with the Muon/AdamW routing rule
* ``newton_schulz``   -- Newton-Schulz orthogonalisation alone
* ``workspace_size``  -- device scratch bytes a call needs
* ``ns_plan``         -- how a matrix's Newton-Schulz iterations are grouped
* ``device_status``   -- reads the device-side status word of a workspace
* ``sharded.shard_plan`` -- opt_shard_plan: the data-parallel sharding plan
  (``sharded`` also holds the per-rank views and the bf16 exchange)
"""

from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional, Sequence

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmpopt.so")

OPT_OK = 0
OPT_ERR_INVALID_ARG = 1
OPT_ERR_MISALIGNED = 3
OPT_ERR_DEVICE_TIMEOUT = 6
STATUS_NAMES = {0: "OPT_OK", 1: "OPT_ERR_INVALID_ARG", 2: "OPT_ERR_UNSUPPORTED", 3: "OPT_ERR_MISALIGNED",
                4: "OPT_ERR_WORKSPACE", 5: "OPT_ERR_CUDA", 6: "OPT_ERR_DEVICE_TIMEOUT"}
KIND_AUTO, KIND_ADAMW, KIND_MUON = 0, 1, 2
SCALE_MODES = {"spectral": 0, "shape_scaling": 1, "unit_rms_norm": 2}
MUON_NO_ORTHOGONALIZE = 1
MUON_NS_PER_ITERATION = 2
MUON_NS_GROUPED = 4
NS_ORDERS = {"auto": 0, "per_iteration": MUON_NS_PER_ITERATION, "grouped": MUON_NS_GROUPED}
FLAG_EMBEDDING_OR_OUTPUT = 1
NS_COEFFS = (3.4445, -4.7750, 2.0315)


class MpoptUnavailable(RuntimeError):
    """The compiled library is missing or failed to load."""


class MpoptError(RuntimeError):
    def __init__(self, status, where, detail=""):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}"
                         + (f" ({detail})" if detail else ""))


class OptTensor(ctypes.Structure):
    _fields_ = [("main_param", ctypes.c_void_p), ("main_grad", ctypes.c_void_p),
                ("exp_avg", ctypes.c_void_p), ("exp_avg_sq", ctypes.c_void_p),
                ("model_param", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ndim", ctypes.c_int32), ("kind", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("reserved", ctypes.c_int32), ("scale_rows", ctypes.c_int64), ("scale_cols", ctypes.c_int64)]


class OptAdamwHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float), ("beta2", ctypes.c_float),
                ("eps", ctypes.c_float), ("weight_decay", ctypes.c_float), ("reserved", ctypes.c_int32),
                ("step", ctypes.c_int64)]


class OptMuonHP(ctypes.Structure):
    _fields_ = [("lr", ctypes.c_float), ("momentum", ctypes.c_float), ("weight_decay", ctypes.c_float),
                ("eps", ctypes.c_float), ("nesterov", ctypes.c_int32), ("ns_steps", ctypes.c_int32),
                ("ns_a", ctypes.c_float), ("ns_b", ctypes.c_float), ("ns_c", ctypes.c_float),
                ("scale_coeff", ctypes.c_float), ("scale_mode", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("ns_schedule", ctypes.POINTER(ctypes.c_float))]


_lib = None

EXPORTED = ("opt_workspace_size", "opt_adamw_step", "opt_muon_step", "opt_mixed_step", "opt_mixed_step_clipped",
            "opt_newton_schulz", "opt_newton_schulz_noalloc", "opt_noalloc_device_status",
            "opt_reload_model_params", "opt_device_status", "opt_shard_plan", "opt_ns_plan",
            "opt_copy_from_host",
            "opt_selftest_wait_timeout", "opt_profile_launches",
            "opt_strerror",
            "opt_last_cuda_error", "opt_abi_version")

KERNEL_NAMES = {0: "ns_gram", 1: "ns_poly", 2: "ns_bx", 3: "adamw", 4: "muon_momentum", 5: "muon_norm",
                6: "muon_apply", 7: "muon_fixup", 8: "grad_norm", 9: "clip_finalize", 10: "muon_sample",
                11: "ns_sym"}
WORKSPACE_CLIP = 0x10
WORKSPACE_GROUPED = 0x20


class OptShardEntry(ctypes.Structure):
    _fields_ = [("owner", ctypes.c_int32), ("reserved", ctypes.c_int32), ("flat_begin", ctypes.c_int64)]


class OptLaunchInfo(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("count", ctypes.c_int32), ("a", ctypes.c_int64),
                ("b", ctypes.c_int64)]


def lib():
    """The loaded library (loads it on first use)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise MpoptUnavailable(f"{LIB_PATH} is not built; run mixed_precision_optimizer_gb300.build_lib")
    try:
        L = ctypes.CDLL(LIB_PATH)
    except OSError as e:
        raise MpoptUnavailable(str(e)) from e
    vp, sz, i32, i64, f32 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
    T = ctypes.POINTER(OptTensor)
    L.opt_workspace_size.argtypes = [T, i32, i32]
    L.opt_workspace_size.restype = sz
    L.opt_adamw_step.argtypes = [ctypes.POINTER(OptAdamwHP), T, i32, vp, sz, vp]
    L.opt_adamw_step.restype = ctypes.c_int
    L.opt_muon_step.argtypes = [ctypes.POINTER(OptMuonHP), T, vp, sz, vp]
    L.opt_muon_step.restype = ctypes.c_int
    L.opt_mixed_step.argtypes = [ctypes.POINTER(OptMuonHP), ctypes.POINTER(OptAdamwHP), T, i32, vp, sz, vp]
    L.opt_mixed_step.restype = ctypes.c_int
    L.opt_mixed_step_clipped.argtypes = [ctypes.POINTER(OptMuonHP), ctypes.POINTER(OptAdamwHP), f32, vp, vp, T, i32,
                                         vp, sz, vp]
    L.opt_mixed_step_clipped.restype = ctypes.c_int
    L.opt_newton_schulz.argtypes = [vp, vp, i64, i64, i32, f32, f32, f32, f32, vp, sz, vp]
    L.opt_newton_schulz.restype = ctypes.c_int
    L.opt_newton_schulz_noalloc.argtypes = [vp, vp, i64, i64, i32, f32, f32, f32, f32, vp]
    L.opt_newton_schulz_noalloc.restype = ctypes.c_int
    L.opt_shard_plan.argtypes = [T, i32, i32, i32, i64, ctypes.POINTER(OptShardEntry), ctypes.POINTER(i64),
                                 ctypes.POINTER(ctypes.c_double)]
    L.opt_shard_plan.restype = ctypes.c_int
    L.opt_ns_plan.argtypes = [i64, i64, ctypes.POINTER(OptMuonHP), ctypes.POINTER(i32), i32, ctypes.POINTER(i32)]
    L.opt_ns_plan.restype = ctypes.c_int
    L.opt_copy_from_host.argtypes = [vp, vp, sz, vp]
    L.opt_copy_from_host.restype = ctypes.c_int
    L.opt_noalloc_device_status.argtypes = [vp]
    L.opt_noalloc_device_status.restype = ctypes.c_int
    L.opt_reload_model_params.argtypes = [T, i32, vp]
    L.opt_reload_model_params.restype = ctypes.c_int
    L.opt_device_status.argtypes = [vp, vp]
    L.opt_device_status.restype = ctypes.c_int
    L.opt_selftest_wait_timeout.argtypes = [vp, vp, i64, i64, vp, sz, vp]
    L.opt_selftest_wait_timeout.restype = ctypes.c_int
    L.opt_profile_launches.argtypes = [vp, ctypes.POINTER(OptLaunchInfo), i32, ctypes.POINTER(i32)]
    L.opt_profile_launches.restype = ctypes.c_int
    L.opt_strerror.argtypes = [ctypes.c_int]
    L.opt_strerror.restype = ctypes.c_char_p
    L.opt_last_cuda_error.argtypes = []
    L.opt_last_cuda_error.restype = ctypes.c_char_p
    L.opt_abi_version.argtypes = []
    L.opt_abi_version.restype = i32
    _lib = L
    return L


def _check(status, where):
    if status != OPT_OK:
        detail = lib().opt_last_cuda_error().decode() if status == 5 else ""
        raise MpoptError(status, where, detail)


# --------------------------------------------------------------------------
# tensor marshalling
# --------------------------------------------------------------------------

def _ptr(t, dtype, what, numel):
    import torch
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{what} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{what} must be {dtype}, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{what} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{what} must be contiguous")
    if t.numel() != numel:
        raise ValueError(f"{what} has {t.numel()} elements, expected {numel}")
    return t.data_ptr() if numel else None


@dataclasses.dataclass
class Param:
    """One parameter's buffers.  ``model`` is the bf16 model copy (None: the
    parameter is fp32-native and ``main_param`` is the model parameter).
    ``exp_avg_sq`` is only used by AdamW.  ``kind`` forces the route
    ("adamw" or "muon"); by default 2-D tensors that are not embeddings or
    output heads go to Muon."""
    main_param: object
    main_grad: object
    exp_avg: object
    exp_avg_sq: object = None
    model: object = None
    embedding_or_output: bool = False
    kind: Optional[str] = None
    scale_shape: Optional[tuple] = None   # Muon: shape setting the update scale (split blocks)

    def to_c(self, force=None):
        import torch
        p = self.main_param
        shape = tuple(p.shape)
        ndim = len(shape)
        if ndim == 2:
            rows, cols = shape
        else:
            rows, cols = 1, p.numel()
        n = rows * cols
        kind = force or self.kind
        ct = OptTensor()
        ct.main_param = _ptr(p, torch.float32, "main_param", n)
        ct.main_grad = _ptr(self.main_grad, torch.float32, "main_grad", n)
        ct.exp_avg = _ptr(self.exp_avg, torch.float32, "exp_avg", n)
        ct.exp_avg_sq = _ptr(self.exp_avg_sq, torch.float32, "exp_avg_sq", n)
        ct.model_param = _ptr(self.model, torch.bfloat16, "model", n)
        ct.rows, ct.cols, ct.ndim = rows, cols, ndim
        ct.kind = {None: KIND_AUTO, "adamw": KIND_ADAMW, "muon": KIND_MUON}[kind]
        ct.flags = FLAG_EMBEDDING_OR_OUTPUT if self.embedding_or_output else 0
        if self.scale_shape is not None:
            ct.scale_rows, ct.scale_cols = (int(x) for x in self.scale_shape)
        return ct

    def split_rows(self, sizes):
        """Row-block views of a 2-D parameter (QKV split: the blocks are
        orthogonalised separately, the update scale stays the whole
        parameter's).  No copies: every block writes into this parameter."""
        import torch
        shape = tuple(self.main_param.shape)
        if len(shape) != 2 or sum(sizes) != shape[0]:
            raise ValueError("split sizes must add up to the number of rows")
        out, r0 = [], 0
        for n in sizes:
            sl = lambda t: None if t is None else t[r0:r0 + n]
            out.append(Param(sl(self.main_param), sl(self.main_grad), sl(self.exp_avg), sl(self.exp_avg_sq),
                             sl(self.model), self.embedding_or_output, "muon", shape))
            r0 += n
        return out


class Prepared:
    """A parameter list marshalled once into the C descriptor array, for
    callers that step the same tensors many times (the pointers must stay
    valid: keep the tensors alive and do not reallocate them)."""

    def __init__(self, params: Sequence[Param], force=None):
        self.params = list(params)
        self.force = force
        self.array = (OptTensor * max(1, len(self.params)))()
        for i, p in enumerate(self.params):
            self.array[i] = p.to_c(force)

    def __len__(self):
        return len(self.params)


def prepare(params: Sequence[Param], force=None) -> Prepared:
    return Prepared(params, force)


def _array(params, force=None):
    if isinstance(params, Prepared):
        return params.array
    arr = (OptTensor * max(1, len(params)))()
    for i, p in enumerate(params):
        arr[i] = p.to_c(force)
    return arr


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def adamw_hp(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, step=1):
    return OptAdamwHP(lr, beta1, beta2, eps, weight_decay, 0, int(step))


def muon_hp(lr=0.02, momentum=0.95, weight_decay=0.0, eps=1e-7, nesterov=True, ns_steps=5,
            coeffs=NS_COEFFS, scale_coeff=0.2, scale_mode="spectral", orthogonalize=True, schedule=None,
            ns_order="auto"):
    """schedule: optional list of ns_steps (a, b, c) triples, one per iteration.
    ns_order: "auto", "per_iteration" or "grouped" (opt_muon_hp.flags)."""
    a, b, c = coeffs
    flags = (0 if orthogonalize else MUON_NO_ORTHOGONALIZE) | NS_ORDERS[ns_order]
    hp = OptMuonHP(lr, momentum, weight_decay, eps, 1 if nesterov else 0, int(ns_steps), a, b, c, scale_coeff,
                   SCALE_MODES[scale_mode], flags, None)
    if schedule is not None:
        flat = [float(x) for trip in schedule for x in trip]
        hp._schedule_buf = (ctypes.c_float * len(flat))(*flat)   # kept alive with the struct
        hp.ns_schedule = ctypes.cast(hp._schedule_buf, ctypes.POINTER(ctypes.c_float))
    return hp


def workspace_size(params: Sequence[Param], routing="auto", clip=False, ns_order="auto") -> int:
    """ns_order="grouped" sizes every Muon shape for grouped iterations."""
    r = {"auto": KIND_AUTO, "adamw": KIND_ADAMW, "muon": KIND_MUON}[routing]
    arr = _array(params)
    r |= (WORKSPACE_CLIP if clip else 0) | (WORKSPACE_GROUPED if ns_order == "grouped" else 0)
    return int(lib().opt_workspace_size(arr, len(params), r))


def copy_from_host(dst, src, stream=None):
    """dst (CUDA tensor) <- src (page-locked CPU tensor) by SM loads of the
    host buffer (opt_copy_from_host), enqueued on `stream`; both contiguous,
    with the same number of bytes."""
    import torch
    if not (dst.is_cuda and dst.is_contiguous() and not src.is_cuda and src.is_contiguous()):
        raise ValueError("copy_from_host: dst must be a contiguous CUDA tensor and src a contiguous CPU tensor")
    nbytes = src.numel() * src.element_size()
    if dst.numel() * dst.element_size() != nbytes:
        raise ValueError("copy_from_host: dst and src differ in size")
    _check(lib().opt_copy_from_host(ctypes.c_void_p(dst.data_ptr()), ctypes.c_void_p(src.data_ptr()), nbytes,
                                    _stream(stream)), "opt_copy_from_host")


def ns_plan(rows, cols, hp: OptMuonHP):
    """Sizes of the groups of Newton-Schulz iterations opt_muon_step uses for
    a rows x cols matrix under hp (opt_ns_plan; host only)."""
    cap = max(int(hp.ns_steps), 1)
    out = (ctypes.c_int32 * cap)()
    n = ctypes.c_int32(0)
    _check(lib().opt_ns_plan(rows, cols, ctypes.byref(hp), out, cap, ctypes.byref(n)), "opt_ns_plan")
    return list(out[:n.value])


def alloc_workspace(nbytes, device=None):
    """Device scratch from the PyTorch caching allocator (256-byte aligned)."""
    import torch
    if nbytes == 0:
        return None
    return torch.empty(int(nbytes), dtype=torch.uint8, device=device or "cuda")


def _ws(workspace):
    if workspace is None:
        return None, 0
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def adamw_step(params, hp: OptAdamwHP, workspace=None, stream=None):
    """params: a list of Param or a Prepared list (marshalled once)."""
    arr = _array(params, "adamw")
    w, nb = _ws(workspace)
    _check(lib().opt_adamw_step(ctypes.byref(hp), arr, len(params), w, nb, _stream(stream)), "opt_adamw_step")


def muon_step(param: Param, hp: OptMuonHP, workspace, stream=None):
    arr = _array([param], "muon")
    w, nb = _ws(workspace)
    _check(lib().opt_muon_step(ctypes.byref(hp), arr, w, nb, _stream(stream)), "opt_muon_step")


def mixed_step(params, hp_muon: Optional[OptMuonHP], hp_adamw: Optional[OptAdamwHP],
               workspace, stream=None):
    arr = _array(params)
    w, nb = _ws(workspace)
    _check(lib().opt_mixed_step(ctypes.byref(hp_muon) if hp_muon is not None else None,
                                ctypes.byref(hp_adamw) if hp_adamw is not None else None,
                                arr, len(params), w, nb, _stream(stream)), "opt_mixed_step")


def mixed_step_clipped(params, hp_muon: Optional[OptMuonHP], hp_adamw: Optional[OptAdamwHP],
                       max_norm: float, workspace, total_norm_out=None, clip_scale_out=None, stream=None):
    """mixed_step with global gradient-norm clipping; the optional outputs are
    1-element fp32 CUDA tensors receiving the norm and the factor applied."""
    import torch
    arr = _array(params)
    w, nb = _ws(workspace)
    tn = _ptr(total_norm_out, torch.float32, "total_norm_out", 1) if total_norm_out is not None else None
    cs = _ptr(clip_scale_out, torch.float32, "clip_scale_out", 1) if clip_scale_out is not None else None
    _check(lib().opt_mixed_step_clipped(ctypes.byref(hp_muon) if hp_muon is not None else None,
                                        ctypes.byref(hp_adamw) if hp_adamw is not None else None,
                                        float(max_norm), tn, cs, arr, len(params), w, nb, _stream(stream)),
           "opt_mixed_step_clipped")


def reload_model_params(params: Sequence[Param], stream=None):
    """main_param <- fp32(model) for every parameter with a bf16 model copy."""
    arr = _array(params)
    _check(lib().opt_reload_model_params(arr, len(params), _stream(stream)), "opt_reload_model_params")


def newton_schulz(G, out, steps=5, coeffs=NS_COEFFS, eps=1e-7, workspace=None, stream=None):
    import torch
    if G.dim() != 2:
        raise ValueError("G must be 2-D")
    rows, cols = G.shape
    gp = _ptr(G, torch.float32, "G", rows * cols)
    op = _ptr(out, torch.float32, "out", rows * cols)
    w, nb = _ws(workspace)
    a, b, c = coeffs
    _check(lib().opt_newton_schulz(gp, op, rows, cols, int(steps), a, b, c, eps, w, nb, _stream(stream)),
           "opt_newton_schulz")


def newton_schulz_workspace_size(rows, cols):
    ct = OptTensor()
    ct.rows, ct.cols, ct.ndim, ct.kind = rows, cols, 2, KIND_MUON
    ct.main_param = ct.main_grad = ct.exp_avg = 256   # any aligned non-null value: sizing only
    arr = (OptTensor * 1)(ct)
    return int(lib().opt_workspace_size(arr, 1, KIND_MUON))


def device_status(workspace, stream=None) -> int:
    if workspace is None:
        return OPT_OK
    return int(lib().opt_device_status(ctypes.c_void_p(workspace.data_ptr()), _stream(stream)))


def selftest_wait_timeout(G, out, workspace, stream=None):
    """Newton-Schulz on G with one TMA stage withheld, so that a bounded
    device-side wait runs out (about 2 s): device_status() then reports
    OPT_ERR_DEVICE_TIMEOUT and the workspace stays usable.  For tests of the
    failure path; `out` receives unspecified values."""
    import torch
    if G.dim() != 2:
        raise ValueError("G must be 2-D")
    rows, cols = G.shape
    gp = _ptr(G, torch.float32, "G", rows * cols)
    op = _ptr(out, torch.float32, "out", rows * cols)
    w, nb = _ws(workspace)
    _check(lib().opt_selftest_wait_timeout(gp, op, rows, cols, w, nb, _stream(stream)), "opt_selftest_wait_timeout")


class LaunchProfiler:
    """Records a CUDA event pair around every kernel the library launches
    from this thread (opt_profile_launches), up to ``capacity`` launches.

        with LaunchProfiler(4096) as prof:
            ... library calls ...
        torch.cuda.synchronize()
        for rec in prof.records(): rec["kernel"], rec["ms"], rec["count"], ...
    """

    def __init__(self, capacity=4096):
        import torch
        self.capacity = int(capacity)
        self._events = [torch.cuda.Event(enable_timing=True) for _ in range(2 * self.capacity)]
        for e in self._events:           # materialise the cudaEvent_t handles
            e.record()
        self._handles = (ctypes.c_void_p * (2 * self.capacity))(*[e.cuda_event for e in self._events])
        self._info = (OptLaunchInfo * self.capacity)()
        self._count = ctypes.c_int32(0)

    def __enter__(self):
        self._count.value = 0
        _check(lib().opt_profile_launches(self._handles, self._info, self.capacity, ctypes.byref(self._count)),
               "opt_profile_launches")
        return self

    def __exit__(self, *exc):
        lib().opt_profile_launches(None, None, 0, None)
        return False

    @property
    def count(self):
        return int(self._count.value)

    def records(self):
        out = []
        for i in range(min(self.count, self.capacity)):
            inf = self._info[i]
            ms = self._events[2 * i].elapsed_time(self._events[2 * i + 1])
            out.append(dict(kernel=KERNEL_NAMES.get(inf.kernel, str(inf.kernel)), count=int(inf.count),
                            a=int(inf.a), b=int(inf.b), ms=float(ms)))
        return out
