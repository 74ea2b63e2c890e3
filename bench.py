#!/usr/bin/env python3
"""Benchmark of the mixed-precision optimizer step on one GB300 (or N replicas).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama16_mixed|tiny_mixed|adamw_8m|muon_8m_skewed|adamw_sweep_10k]
                    [--shard] [--clip MAX_NORM] [--no-sweep] [--clock-log DIR]

A step is one full optimizer step over the workload: AdamW over every
AdamW-routed tensor, Muon (momentum, Nesterov, five Newton-Schulz iterations,
scaled update) over every 2-D hidden matrix, and the bf16 writeback of every
parameter.  The default workload is the Llama-like 16-layer parameter set
(3.49e9 Muon + 1.05e9 AdamW parameters), the only one that exercises the
whole path at scale.  Inputs are seeded synthetic tensors drawn on the GPU;
the per-step inputs (~100 GB resident) are far larger than L2.

Prints ONE JSON line on rank 0.  With --impl reference the line times the
CPU oracle (numpy, fp64 Newton-Schulz) on a fixed sample of one step of the
same workload instead.  Under torchrun (N > 1) every rank by default runs an
independent replica of the whole step on its own GPU, and the process group
carries only barriers and the max-over-ranks time (weak scaling).  With
--shard the ranks share one step (ZeRO-1 AdamW ranges, one owner per Muon
matrix, the bf16 pieces exchanged by broadcasts; strong scaling).  After the
main line's measurements the 10,000-tensor AdamW sweep reports GB/s per size
decade (--no-sweep skips it).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synthetic as S  # noqa: E402

METRIC = "optimizer-step params/s; AdamW HBM GB/s; Muon Newton-Schulz TFLOPS"
UNIT = "params/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
ADAMW_BYTES_PER_PARAM = 30     # read p, g, m, v (16 B); write p, m, v (12 B) and bf16 (2 B)
NOMINAL_HBM_GBS = 8000.0       # GB300 HBM3e, nominal (the measured copy bandwidth is the roofline's peak)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama16_mixed", choices=sorted(S.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps of the end-to-end leg; its time includes filling and draining the copy pipeline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--compare-cublas", action="store_true",
                    help="also time cuBLAS (torch.bmm, fp16) on the Newton-Schulz GEMM shapes of the largest "
                         "Muon group, back to back for a few seconds each, for comparison only")
    ap.add_argument("--clip", type=float, default=0.0,
                    help="max_norm of global grad-norm clipping fused into the step (0: off)")
    ap.add_argument("--shard", action="store_true",
                    help="data-parallel sharded step over the ranks (ZeRO-1 AdamW ranges, one owner per Muon "
                         "matrix, bf16 exchange by broadcasts); total work fixed as N grows (strong scaling)")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the AdamW size sweep (10,000 tensors, GB/s per size decade) after the main workload")
    ap.add_argument("--ns-order", choices=["auto", "per_iteration", "grouped"], default="auto",
                    help="evaluation order of the Newton-Schulz iterations (opt_muon_hp.flags)")
    ap.add_argument("--clock-log", default=None, help="directory for the nvidia-smi clock samples (default: temp)")
    return ap.parse_args()


# ------------------------------------------------------------------ peaks --

def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


# ----------------------------------------------------------------- clocks --

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap,"
             "clocks.mem,temperature.gpu")

    log_dir = None   # --clock-log DIR keeps the samples there; otherwise a temporary file

    def __init__(self, index, tag=""):
        self.index = index
        self.proc = None
        self.tag = tag

    def __enter__(self):
        try:
            if ClockSampler.log_dir:
                os.makedirs(ClockSampler.log_dir, exist_ok=True)
                self.path = os.path.join(ClockSampler.log_dir, f"clocks{self.tag}_gpu{self.index}.csv")
            else:
                fd, self.path = tempfile.mkstemp(prefix=f"mpopt_clocks{self.tag}_", suffix=".csv")
                os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.3)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()
        return False

    def summary(self):
        if self.proc is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    extra = [float(x) for x in parts[9:11]] if len(parts) >= 11 else [float("nan")] * 2
                    rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9], *extra))
                except ValueError:
                    continue
        if not ClockSampler.log_dir:
            try:
                os.unlink(self.path)
            except OSError:
                pass
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[3]) if v.lower() == "active"})
        loaded = [r for r in rows if r[2] > 200.0] or rows
        out = {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
               "power_w_max": max(r[2] for r in rows), "samples": len(rows), "reasons": reasons}
        if all(r[4] == r[4] for r in rows):
            out["mem_mhz"] = statistics.median(r[4] for r in loaded)
            out["temp_c_max"] = max(r[5] for r in rows)
        return out


def smi_index(cuda_index):
    """nvidia-smi's index of a CUDA device (CUDA_VISIBLE_DEVICES remaps)."""
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    parts = [p.strip() for p in vis.split(",") if p.strip()]
    if cuda_index < len(parts) and parts[cuda_index].isdigit():
        return int(parts[cuda_index])
    return cuda_index


# ------------------------------------------------------------ distributed --

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch
            import torch.distributed as dist
            backend = "nccl" if torch.cuda.is_available() else "gloo"
            if backend == "nccl":
                torch.cuda.set_device(self.local)
            dist.init_process_group(backend)
            self.pg = dist

    def barrier(self):
        if self.pg is not None:
            self.pg.barrier()

    def max(self, x: float) -> float:
        """Max over ranks (timing only; no optimizer data crosses ranks)."""
        if self.pg is None:
            return x
        import torch
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        t = torch.tensor([x], dtype=torch.float64, device=dev)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg is not None:
            self.pg.destroy_process_group()


# ---------------------------------------------------------------- workload --

def is_muon(w: S.Workload, spec: S.TensorSpec) -> bool:
    """The routing rule the library applies ("02 · Optimizer：算法与 infra" §5.5):
    2-D and not an embedding/output -> Muon; used here only to decide whether
    a tensor needs a second-moment buffer."""
    return (not w.force_adamw) and len(spec.shape) == 2 and not spec.embedding_or_output


FLAT_ALIGN = 64   # elements: every tensor of a flat buffer starts 256 B (fp32) / 128 B (bf16) aligned


def flat_layout(numels):
    """Element offsets of consecutive tensors in one flat buffer, each start
    rounded up to FLAT_ALIGN elements; and the buffer's length."""
    offs, o = [], 0
    for n in numels:
        offs.append(o)
        o += -(-int(n) // FLAT_ALIGN) * FLAT_ALIGN
    return offs, max(o, FLAT_ALIGN)


def flat_views(flat, offs, shapes):
    return [flat[o:o + int(math.prod(sh))].view(sh) for o, sh in zip(offs, shapes)]


def step_groups(w: S.Workload):
    """The tensors in the groups the library steps them in: one group per Muon
    shape class (smallest first), then the AdamW tensors.  [(kind, indices)]."""
    classes, adamw = {}, []
    for i, sp in enumerate(w.tensors):
        if is_muon(w, sp):
            classes.setdefault(tuple(sorted(sp.shape)), []).append(i)
        else:
            adamw.append(i)
    out = [("muon", ids) for ids in sorted(classes.values(), key=lambda ids: sum(w.tensors[i].numel for i in ids))]
    if adamw:
        out.append(("adamw", adamw))
    return out


def build_device_workload(w: S.Workload, device):
    """Parameters, optimizer state and gradients of the workload on the
    device.  As in a mixed-precision trainer, every main_grad is a view of one
    contiguous fp32 gradient buffer and every bf16 model copy a view of one
    contiguous bf16 buffer (same element offsets), so the e2e leg moves each
    direction's data with one copy per step group.  The buffers hold the
    tensors group by group (step_groups), so each group is one contiguous
    segment."""
    import torch
    import mixed_precision_optimizer_gb300 as mp
    shapes = [spec.shape for spec in w.tensors]
    groups = step_groups(w)
    order = [i for _, ids in groups for i in ids]
    offs_in_order, n_flat = flat_layout(w.tensors[i].numel for i in order)
    offs = [0] * len(w.tensors)
    for i, o in zip(order, offs_in_order):
        offs[i] = o
    segments, pos = [], 0
    for kind, ids in groups:
        start = offs_in_order[pos]
        pos += len(ids)
        end = offs_in_order[pos] if pos < len(order) else n_flat
        segments.append((kind, ids, start, end))
    grad_flat = torch.empty(n_flat, dtype=torch.float32, device=device)
    model_flat = torch.empty(n_flat, dtype=torch.bfloat16, device=device)
    grads, models = flat_views(grad_flat, offs, shapes), flat_views(model_flat, offs, shapes)
    params, n_muon, n_adamw = [], 0, 0
    for i, spec in enumerate(w.tensors):
        p = torch.empty(spec.shape, dtype=torch.float32, device=device)
        S.torch_init_(p, spec, i)
        g = grads[i]
        S.torch_grad_(g, spec, i, 1)
        m = torch.zeros_like(p)
        muon = is_muon(w, spec)
        v = None if muon else torch.zeros_like(p)
        model = models[i]
        model.copy_(p)
        params.append(mp.Param(p, g, m, v, model, embedding_or_output=spec.embedding_or_output,
                               kind="adamw" if w.force_adamw else None))
        if muon:
            n_muon += spec.numel
        else:
            n_adamw += spec.numel
    flat = {"offsets": offs, "shapes": shapes, "grad": grad_flat, "model": model_flat, "segments": segments}
    return params, n_muon, n_adamw, flat


def hyper(w: S.Workload, ns_order="auto"):
    import mixed_precision_optimizer_gb300 as mp
    hm = None
    if w.muon is not None:
        hm = mp.muon_hp(lr=w.muon.lr, momentum=w.muon.momentum, weight_decay=w.muon.weight_decay,
                        nesterov=w.muon.nesterov, ns_steps=w.muon.ns_steps, ns_order=ns_order)

    def ha(t):
        if w.adamw is None:
            return None
        return mp.adamw_hp(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
                           weight_decay=w.adamw.weight_decay, step=t)
    return hm, ha


NS_KERNELS = ("ns_gram", "ns_poly", "ns_sym", "ns_bx")


def iteration_flops(A, B):
    """Flops of one Newton-Schulz iteration on one matrix as the pages count
    them (dense products): 2 (2 A^2 B + A^3), the pages' 4 m^2 n + 2 m^3."""
    return 2.0 * (2.0 * A * A * B + A * A * A)


def annotate_iterations(recs):
    """Marks each C X launch with the iterations it completes: the polynomial
    launches since the previous C X (one per iteration; grouped iterations
    share one C X).  Records are in launch order."""
    polys = 0
    for r in recs:
        if r["kernel"] == "ns_poly":
            polys += 1
        elif r["kernel"] == "ns_bx":
            r["iters"] = polys
            polys = 0
    return recs


def gemm_pages_flops(rec):
    """The pages' dense count of the iterations a launch completes, all put
    on the C X that ends them: 2 (2 A^2 B + A^3) per iteration and matrix."""
    if rec["kernel"] != "ns_bx":
        return 0.0
    return rec["count"] * rec.get("iters", 1) * iteration_flops(rec["a"], rec["b"])


def gemm_method_flops(rec):
    """Flops of one launch's own products, the symmetric ones at their
    triangle: X X^T A^2 B, A A and the products of grouped iterations A^3,
    C X 2 A^2 B.  This is the roofline's algorithmic count.  Per-iteration
    evaluation does 3 A^2 B + A^3 per iteration; a group of g iterations
    does 3 A^2 B + (4 g - 3) A^3."""
    A, B, c = rec["a"], rec["b"], rec["count"]
    k = rec["kernel"]
    if k == "ns_gram":
        return c * 1.0 * A * A * B
    if k in ("ns_poly", "ns_sym"):
        return c * 1.0 * A * A * A
    return c * 2.0 * A * A * B


def gemm_executed_flops(rec):
    """Flops the tensor cores actually execute: padded shapes, and only the
    on-or-below-diagonal 256x256 blocks of the symmetric products."""
    Ap = -(-rec["a"] // 256) * 256
    Bp = -(-rec["b"] // 256) * 256
    T = Ap // 256
    c = rec["count"]
    if rec["kernel"] == "ns_gram":
        return c * T * (T + 1) * 2.0 * 128 * 256 * Bp
    if rec["kernel"] in ("ns_poly", "ns_sym"):
        return c * T * (T + 1) * 2.0 * 128 * 256 * Ap
    return c * 2.0 * Ap * Ap * Bp


def kernels_by_shape(recs, peak):
    """Per Newton-Schulz GEMM stage and Muon shape class (A x B, matrices per
    launch): launches, ms per launch, TFLOP/s by the launch's own algorithmic
    count (the roofline's) and as executed by the tensor cores; the executed
    rate as a fraction of `peak`."""
    out = {}
    for r in recs:
        if r["kernel"] not in NS_KERNELS:
            continue
        k = out.setdefault(f"{r['kernel']} {r['a']}x{r['b']} x{r['count']}",
                           dict(launches=0, ms=0.0, method=0.0, ex=0.0))
        k["launches"] += 1
        k["ms"] += r["ms"]
        k["method"] += gemm_method_flops(r)
        k["ex"] += gemm_executed_flops(r)
    res = {}
    for name, k in sorted(out.items()):
        sec = k["ms"] * 1e-3
        res[name] = {"launches": k["launches"], "ms_per_launch": round(k["ms"] / k["launches"], 4),
                     "tflops_method": round(k["method"] / sec / 1e12, 1),
                     "tflops_executed": round(k["ex"] / sec / 1e12, 1),
                     "executed_frac": round(k["ex"] / sec / 1e12 / peak, 3)}
    return res


def cublas_same_shapes(w, seconds=3.0):
    """cuBLAS (torch.bmm, fp16 in and out, fp32 accumulation) on the three GEMMs
    of one Newton-Schulz iteration of the largest Muon group, each run back to
    back for `seconds` and timed with CUDA events; the symmetric products are
    computed in full, as a library GEMM does.  For comparison only: this is
    not the optimizer step."""
    import torch
    groups = {}
    for sp in w.tensors:
        if is_muon(w, sp):
            A, B = sorted(sp.shape)
            groups[(A, B)] = groups.get((A, B), 0) + 1
    if not groups:
        return None
    (A, B), n = max(groups.items(), key=lambda kv: kv[1] * kv[0][0] * kv[0][0] * kv[0][1])
    n = min(n, 64)
    g = torch.Generator(device="cuda")
    g.manual_seed(0)
    X = (torch.randn(n, A, B, device="cuda", generator=g) * 0.01).half()
    C = (torch.randn(n, A, A, device="cuda", generator=g) * 0.01).half()
    out_x = torch.empty(n, A, B, device="cuda", dtype=torch.half)
    out_a = torch.empty(n, A, A, device="cuda", dtype=torch.half)
    res = {"shape": f"{n} x ({A} x {B})", "note": "full products; fp16 operands and output"}
    for name, fn, flops in (("C X", lambda: torch.bmm(C, X, out=out_x), 2.0 * n * A * A * B),
                            ("X X^T", lambda: torch.bmm(X, X.transpose(1, 2), out=out_a), 2.0 * n * A * A * B),
                            ("A A", lambda: torch.bmm(C, C, out=out_a), 2.0 * n * A * A * A)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        k, t0 = 0, time.perf_counter()
        e0.record()
        while time.perf_counter() - t0 < seconds:
            fn()
            k += 1
            if k % 4 == 0:
                torch.cuda.synchronize()
        e1.record()
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / k
        res[name] = {"ms_per_launch": round(ms, 3), "tflops": round(flops / (ms * 1e-3) / 1e12, 1)}
    del X, C, out_x, out_a
    torch.cuda.empty_cache()
    return res


def source_sha(name):
    """sha256 prefix of a kernel source file: a profile row applies only while
    the source it was captured from is unchanged."""
    path = os.path.join(ROOT, "mixed_precision_optimizer_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def profile_row(key):
    """The row `key` of profiles/rows.json (figures taken from committed ncu
    captures) if the kernel source it names still has the sha256 prefix it was
    captured from; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "rows.json"), encoding="utf-8") as f:
            rows = json.load(f)
    except (OSError, ValueError):
        return None
    row = rows.get(key)
    if not isinstance(row, dict):
        return None
    try:
        if source_sha(row["source"]) != row["sha256_16"]:
            return None
    except (OSError, KeyError):
        return None
    return row


# ------------------------------------------------------------ CPU oracle --

MUON_SAMPLE_FLOPS = 1.5e11   # a shape class is run through the oracle when one matrix's NS is at most this


def cpu_oracle_sample(w: S.Workload):
    """Time the oracle (as it stands) on a fixed sample of one step of the
    workload and extrapolate to the whole step.  The same sample serves the
    cpu_baseline of our arm and every step of --impl reference, so the two
    report one measurement:

      AdamW  the fp32 oracle over min(AdamW elements, 2^24) elements, scaled
             per element to every AdamW parameter;
      Muon   one fp64 oracle step on one matrix of every shape class whose
             Newton-Schulz is at most MUON_SAMPLE_FLOPS (at least the
             smallest class), scaled by the count of its class; larger classes
             extrapolated by Newton-Schulz flop count at the best fp64 rate
             the sampled classes reached.

    Returns (seconds per step, description dict)."""
    import numpy as np
    from oracle import adamw as OA
    from oracle import muon as OM
    rng = np.random.default_rng(0)
    t_total = 0.0
    sampled, extrapolated = [], []
    adamw_n = sum(s.numel for s in w.tensors if not is_muon(w, s))
    if adamw_n:
        n = min(adamw_n, 1 << 24)
        p = rng.standard_normal(n, dtype=np.float32)
        g = (rng.standard_normal(n, dtype=np.float32) * 1e-3).astype(np.float32)
        m = np.zeros(n, np.float32)
        v = np.zeros(n, np.float32)
        t0 = time.perf_counter()
        OA.adamw_step_fp32(p, g, m, v, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, t=1)
        dt = time.perf_counter() - t0
        t_total += dt / n * adamw_n
        sampled.append(f"AdamW fp32 oracle on {n} elements")
        if n < adamw_n:
            extrapolated.append(f"AdamW scaled per element to {adamw_n}")
    shapes = {}
    for sp in w.tensors:
        if is_muon(w, sp):
            key = tuple(sorted(sp.shape))
            shapes[key] = shapes.get(key, 0) + 1
    if shapes:
        measured = {}
        for key in sorted(shapes, key=lambda k: OM.ns_flops(*k)):
            if measured and OM.ns_flops(*key) > MUON_SAMPLE_FLOPS:
                break
            A, B = key
            W = rng.standard_normal((A, B)) * 0.02
            gg = rng.standard_normal((A, B)) * 1e-3
            t0 = time.perf_counter()
            OM.muon_step(W, gg, np.zeros_like(W), lr=0.02, momentum=0.95)
            measured[key] = (time.perf_counter() - t0, OM.ns_flops(*key))
            sampled.append(f"Muon fp64 oracle step on one {A}x{B} matrix")
        rate = max(f / t for t, f in measured.values())     # fp64 flop/s of the best-measured shape
        for key, cnt in shapes.items():
            if key in measured:
                t_total += cnt * measured[key][0]
                if cnt > 1:
                    extrapolated.append(f"{key[0]}x{key[1]} x{cnt} from one matrix")
            else:
                t_total += cnt * OM.ns_flops(*key) / rate
                extrapolated.append(f"{key[0]}x{key[1]} x{cnt} by Newton-Schulz flops at {rate / 1e9:.1f} GFLOP/s")
    desc = {"sampled": sampled, "extrapolated": bool(extrapolated), "extrapolation": extrapolated,
            "threads": f"Newton-Schulz matmuls: BLAS on up to {cpu_threads()} threads; AdamW and the Muon "
                       "elementwise steps: numpy on 1 thread"}
    return t_total, desc


def cpu_baseline_entry(w, t_step, desc, total):
    return {"value": round(total / t_step, 1), "unit": UNIT, "cores": cpu_threads(), "kind": "oracle",
            "sample": "; ".join(desc["sampled"]) + " (one step of the workload, extrapolated to all of it)",
            "extrapolated": desc["extrapolated"], "extrapolation": desc["extrapolation"],
            "cores_detail": desc["threads"], "seconds_per_step": round(t_step, 3)}


def workload_config(w: S.Workload, clip: float):
    """The workload as both arms name it (identical dicts)."""
    n_muon = sum(s.numel for s in w.tensors if is_muon(w, s))
    total = w.numel
    return {"workload": w.name, "params": total, "muon_params": n_muon, "adamw_params": total - n_muon,
            "tensors": len(w.tensors), "grad_clip_max_norm": clip if clip > 0 else None,
            "l2": "inputs larger than L2 (all state resident, ~18 B/param touched per step)"
            if total * 14 > 4 * 129e6 else "L2 not flushed: workload smaller than L2"}


def cpu_threads():
    n = os.cpu_count() or 1
    for var in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS"):
        if os.environ.get(var, "").isdigit():
            n = min(n, int(os.environ[var]))
    return n


# --------------------------------------------------------------- our arm --

def run_ours(args, dist: Dist):
    import torch
    import mixed_precision_optimizer_gb300 as mp
    from mixed_precision_optimizer_gb300 import build_lib
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    build_lib.build()
    device = torch.device("cuda", dist.local)
    torch.cuda.set_device(device)
    w = S.WORKLOADS[args.workload]()
    params, n_muon, n_adamw, flat = build_device_workload(w, device)
    total = n_muon + n_adamw
    hm, ha = hyper(w, args.ns_order)
    if args.shard:
        # this rank keeps the replicated main_grad and bf16 model of every
        # tensor, and master/state only for what the plan gives it
        from mixed_precision_optimizer_gb300 import sharded as sh
        if args.clip > 0:
            raise SystemExit("--shard with --clip is not supported (the norm would need a cross-rank sum)")
        plan = sh.shard_plan(params, dist.world)
        state = sh.RankState.empty(plan, dist.rank, device)
        state.load(plan, params)
        params = [mp.Param(None, p.main_grad, None, None, p.model, p.embedding_or_output, p.kind) for p in params]
        torch.cuda.empty_cache()

        def prepare_set(plist):
            return plist, mp.prepare(sh.rank_params(plist, plan, state))

        prepared = prepare_set(params)
        ws = mp.alloc_workspace(mp.workspace_size(prepared[1].params), device)

        def step(t, pset=None):
            pset = prepared if pset is None else pset
            sh.sharded_step(pset[0], plan, state, hm, ha(t), ws, prepared=pset[1])
    else:
        prepare_set = mp.prepare
        ws = mp.alloc_workspace(mp.workspace_size(params, clip=args.clip > 0, ns_order=args.ns_order), device)
        prepared = mp.prepare(params)

        def step(t, plist=None):
            plist = prepared if plist is None else plist
            if args.clip > 0:
                mp.mixed_step_clipped(plist, hm, ha(t), args.clip, ws)
            else:
                mp.mixed_step(plist, hm, ha(t), ws)

    def group_step(t, plist, kind):
        """One step group through the public API (the e2e leg without clipping
        or sharding): opt_adamw_step for the AdamW tensors, opt_mixed_step for
        a Muon shape class."""
        if kind == "adamw":
            mp.adamw_step(plist, ha(t))
        else:
            mp.mixed_step(plist, hm, None, ws)

    stream = torch.cuda.current_stream()
    t = 1
    for _ in range(args.warmup):
        step(t)
        t += 1
    torch.cuda.synchronize()
    if mp.device_status(ws) != mp.OPT_OK:
        raise SystemExit("device-side timeout during warm-up")

    # ---- timed region: K steps, inputs resident in HBM
    prof = mp.LaunchProfiler(capacity=max(256, 100 * args.steps))
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(smi_index(device.index)) as clocks:
        dist.barrier()
        torch.cuda.synchronize()
        start.record(stream)
        host_ms = []
        with prof:
            for _ in range(args.steps):
                h0 = time.perf_counter()
                step(t)
                host_ms.append((time.perf_counter() - h0) * 1e3)
                t += 1
        end.record(stream)
        torch.cuda.synchronize()
        dist.barrier()
    elapsed_ms = dist.max(start.elapsed_time(end))
    if mp.device_status(ws) != mp.OPT_OK:
        raise SystemExit("device-side timeout in the timed region")
    recs = prof.records()
    launches = prof.count

    # ---- per-kernel breakdown from the events around each launch
    peaks, peak_src = load_peaks()
    line = measured_line(args, w, recs, launches, elapsed_ms, total, dist, peaks, peak_src)
    # host time of each step call: the first starts on an empty launch queue;
    # later ones block only once the queue holds more launches than it takes
    line["host_enqueue_ms"] = {"first_step": round(host_ms[0], 3), "median": round(statistics.median(host_ms), 3),
                               "max": round(max(host_ms), 3), "launches_per_step": launches // args.steps}

    # ---- end to end through the public API with host buffers
    grouped = None if (args.shard or args.clip > 0) else group_step
    line["e2e"] = run_e2e(args, step, prepare_set, params, flat, t, total, dist, grouped,
                          step_ms=elapsed_ms / args.steps)
    t += args.e2e_steps
    line["clocks"] = clocks.summary()
    if args.compare_cublas and dist.rank == 0:
        with ClockSampler(smi_index(device.index), "_cublas") as cclocks:
            line["cublas_same_shapes"] = cublas_same_shapes(w)
        if line["cublas_same_shapes"] is not None:
            line["cublas_same_shapes"]["clocks"] = cclocks.summary()

    # ---- AdamW GB/s by size decade: the 10,000-tensor sweep, on the device
    # once this workload's buffers are released
    del step, group_step, grouped, params, flat, prepared, ws
    import gc
    gc.collect()
    torch.cuda.empty_cache()
    if w.name == "adamw_sweep_10k" or not args.no_sweep:
        line["adamw_gbs_by_size"] = run_sweep(device, peaks)
    if dist.rank == 0 and dist.world == 1 and not args.no_cpu_baseline:
        t_cpu, desc = cpu_oracle_sample(w)
        line["cpu_baseline"] = cpu_baseline_entry(w, t_cpu, desc, total)
    return line


def measured_line(args, w, recs, launches, elapsed_ms, total, dist, peaks, peak_src):
    """The JSON line's measured part: value, per-kernel times, the roofline of
    the dominant kernel and AdamW's bandwidth."""
    kernels = {}
    annotate_iterations(recs)
    for r in recs:
        k = kernels.setdefault(r["kernel"], dict(launches=0, ms=0.0, flops=0.0, method=0.0, executed=0.0, elems=0))
        k["launches"] += 1
        k["ms"] += r["ms"]
        if r["kernel"] in NS_KERNELS:
            k["flops"] += gemm_pages_flops(r)
            k["method"] += gemm_method_flops(r)
            k["executed"] += gemm_executed_flops(r)
        if r["kernel"] == "adamw":
            k["elems"] += r["a"]
    busy = sum(k["ms"] for k in kernels.values()) or 1.0
    kern_out = {}
    for name, k in kernels.items():
        e = dict(launches=k["launches"], ms_total=round(k["ms"], 3), share=round(k["ms"] / busy, 4))
        if k["method"]:
            sec = k["ms"] * 1e-3
            e["tflops_method"] = round(k["method"] / sec / 1e12, 1)
            e["tflops_executed"] = round(k["executed"] / sec / 1e12, 1)
        if k["elems"]:
            e["gbs"] = round(k["elems"] * ADAMW_BYTES_PER_PARAM / (k["ms"] * 1e-3) / 1e9, 1)
        kern_out[name] = e
    # dominant kernel: the fp16 tensor-core GEMM (X X^T, A A, the grouped
    # iterations' products and C X are one kernel)
    ns = NS_KERNELS
    gemm_ms = sum(kernels.get(n, {}).get("ms", 0.0) for n in ns)
    adamw_ms = kernels.get("adamw", {}).get("ms", 0.0)
    sustained = peaks["bf16_tflops_sustained"]
    if gemm_ms >= adamw_ms and gemm_ms > 0:
        sec = gemm_ms * 1e-3
        fl = sum(kernels.get(n, {}).get("flops", 0.0) for n in ns)
        me = sum(kernels.get(n, {}).get("method", 0.0) for n in ns)
        ex = sum(kernels.get(n, {}).get("executed", 0.0) for n in ns)
        nl = sum(kernels.get(n, {}).get("launches", 0) for n in ns)
        achieved = me / sec / 1e12
        # fp16 and bf16 share the dense tensor rate (nominal ratio 1), so the
        # measured bf16 figure is the fp16 peak
        row = profile_row("ns_gemm_traffic") or {}
        pipe = profile_row("ns_gemm_tensor_pipe")
        roofline = {"bound": "tensor",
                    "kernel": "ns_gemm_kernel (fp16 x fp16 -> fp32: X X^T, A A, grouped-iteration products, C X)",
                    "achieved": round(achieved, 1), "peak": sustained, "unit": "TFLOP/s",
                    "frac": round(achieved / sustained, 4), "traffic": row.get("bytes_per_launch"),
                    "count": "each launch's own products, symmetric ones at their triangle: X X^T A^2 B, A A and "
                             "the grouped iterations' products A^3, C X 2 A^2 B (per iteration 3 A^2 B + A^3; "
                             "a group of g iterations 3 A^2 B + (4 g - 3) A^3)",
                    "peak_source": f"{peak_src} bf16_tflops_sustained (of measured) x nominal fp16/bf16 ratio 1",
                    "per_launch_flops": round(me / nl), "avg_launch_ms": round(gemm_ms / nl, 4),
                    "executed_tflops": round(ex / sec / 1e12, 1),
                    "executed_frac": round(ex / sec / 1e12 / sustained, 4),
                    "executed_count": "padded to 256, every 256 x 256 block on or below the diagonal in full",
                    "pages_count_tflops": round(fl / sec / 1e12, 1),
                    "pages_count": "iteration-equivalent rate: 2 (2 A^2 B + A^3) per iteration and matrix (the "
                                   "pages' 4 m^2 n + 2 m^3, dense products) over the GEMM time; grouped iterations "
                                   "do fewer flops, so this is not a tensor-pipe rate",
                    "burst_frac": round(achieved / peaks["bf16_tflops"], 4),
                    "traffic_source": row.get("how"),
                    "tensor_pipe_active_pct": pipe.get("pct") if pipe else None}
    else:
        k = kernels["adamw"]
        achieved = k["elems"] * ADAMW_BYTES_PER_PARAM / (k["ms"] * 1e-3) / 1e9
        peak = peaks["hbm_gbs"]
        row = profile_row("adamw_traffic") or {}
        roofline = {"bound": "hbm", "kernel": "adamw_mta_kernel", "achieved": round(achieved, 1), "peak": peak,
                    "unit": "GB/s", "frac": round(achieved / peak, 4), "traffic": row.get("bytes_per_launch"),
                    "peak_source": f"{peak_src} hbm_gbs (of measured)",
                    "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                    "per_launch_bytes": round(k["elems"] * ADAMW_BYTES_PER_PARAM / k["launches"]),
                    "avg_launch_ms": round(k["ms"] / k["launches"], 4)}
    roofline_adamw = None
    if "adamw" in kernels:
        k = kernels["adamw"]
        gbs = kern_out["adamw"]["gbs"]
        row = profile_row("adamw_traffic") or {}
        roofline_adamw = {"bound": "hbm", "kernel": "adamw_mta_kernel", "achieved": gbs,
                          "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                          "frac_of_nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4),
                          "traffic": row.get("bytes_per_launch"), "peak_source": f"{peak_src} hbm_gbs (of measured)",
                          "per_launch_bytes": round(k["elems"] * ADAMW_BYTES_PER_PARAM / k["launches"])}
    shard = getattr(args, "shard", False)
    # replicas: every rank steps the whole workload; sharded: the ranks
    # together step it once per step
    value = total * args.steps * (1 if shard else dist.world) / (elapsed_ms * 1e-3)
    cfg = workload_config(w, args.clip)
    return {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(elapsed_ms / args.steps, 3), "higher_is_better": True,
        "scaling": "strong" if shard else "weak", "vs_baseline": None, "dtype": "f32",
        "dtype_detail": "fp32 master weights, gradients, state and AdamW arithmetic; Newton-Schulz GEMMs take fp16 "
                        "operands with fp32 accumulation on the tensor cores; bf16 model writeback",
        "data": "synthetic (seeded, drawn on the GPU)",
        "config": cfg,
        "parallelism": (f"sharded x{dist.world} (ZeRO-1 AdamW, one owner per Muon matrix)" if shard
                        else f"replicas x{dist.world}" if dist.world > 1 else "1 GPU"),
        "ns_order": getattr(args, "ns_order", "auto"),
        "adamw_gbs": kern_out.get("adamw", {}).get("gbs"),
        "ns_tflops_method": roofline.get("achieved") if roofline["bound"] == "tensor" else None,
        "roofline": roofline,
        "roofline_adamw": roofline_adamw,
        "kernels": kern_out,
        "kernels_by_shape": kernels_by_shape(recs, sustained),
        "gpu_launches": launches,
    }


def run_sweep(device, peaks):
    """AdamW GB/s by size decade on the 10,000-tensor sweep (sizes log-uniform
    in [1, 2^24), ~1.0e10 parameters, 18 B/param resident).  All tensors at
    once when the device has room; otherwise five seeded groups of 2,000
    tensors, one after another, their per-decade times added.  Every array is
    a view of one flat buffer per kind (p, g, m, v, bf16 copy)."""
    import torch
    import mixed_precision_optimizer_gb300 as mp
    w = S.adamw_sweep_10k()
    specs = list(w.tensors)
    need = w.numel * 18 * 1.03 + 4e9
    free, _ = torch.cuda.mem_get_info()
    if free >= need:
        groups, mode = [list(range(len(specs)))], "all 10,000 tensors resident"
    else:
        import numpy as np
        perm = np.random.default_rng([S.INIT_SEED, 5]).permutation(len(specs))
        groups, mode = [sorted(perm[k::5].tolist()) for k in range(5)], "5 seeded groups of 2,000 tensors"
    hp = mp.adamw_hp(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
                     weight_decay=w.adamw.weight_decay, step=1)
    acc = {}
    for ids in groups:
        numels = [specs[i].numel for i in ids]
        offs, n_flat = flat_layout(numels)
        flats = [torch.empty(n_flat, dtype=torch.float32, device=device) for _ in range(4)]
        model = torch.empty(n_flat, dtype=torch.bfloat16, device=device)
        shp = [specs[i].shape for i in ids]
        P, G, M, V = (flat_views(f, offs, shp) for f in flats)
        Bv = flat_views(model, offs, shp)
        M_flat, V_flat = flats[2], flats[3]
        M_flat.zero_()
        V_flat.zero_()
        params = []
        for k, i in enumerate(ids):
            S.torch_init_(P[k], specs[i], i)
            S.torch_grad_(G[k], specs[i], i, 1)
            params.append(mp.Param(P[k], G[k], M[k], V[k], Bv[k], kind="adamw"))
        for key, rec in adamw_buckets(params, hp).items():
            a = acc.setdefault(key, dict(tensors=0, params=0, launches=0, ms=0.0))
            for f in ("tensors", "params", "launches"):
                a[f] += rec[f]
            a["ms"] += rec["kernel_ms"]
        del params, P, G, M, V, Bv, flats, model, M_flat, V_flat
        torch.cuda.empty_cache()
    out = {"mode": mode, "bytes_per_param": ADAMW_BYTES_PER_PARAM, "peak_gbs": peaks["hbm_gbs"], "buckets": {}}
    for key, a in sorted(acc.items(), key=lambda kv: float(kv[0].split("-")[0])):
        gbs = a["params"] * ADAMW_BYTES_PER_PARAM / (a["ms"] * 1e-3) / 1e9
        out["buckets"][key] = {"tensors": a["tensors"], "params": a["params"], "launches": a["launches"],
                               "kernel_ms": round(a["ms"], 4), "gbs": round(gbs, 1),
                               "frac": round(gbs / peaks["hbm_gbs"], 4)}
    tp = sum(a["params"] for a in acc.values())
    tm = sum(a["ms"] for a in acc.values())
    out["all"] = {"params": tp, "kernel_ms": round(tm, 3),
                  "gbs": round(tp * ADAMW_BYTES_PER_PARAM / (tm * 1e-3) / 1e9, 1)}
    return out


class PinnedHostArena:
    """Page-locked host memory for every per-tensor host buffer of the e2e
    leg: one allocation from CUDA's pinned-host allocator (cudaHostAlloc,
    through torch's pinned memory), carved into per-tensor views at 256-byte
    boundaries.

    On the GB300 hosts (64 KiB base pages) the copy engines are fast only on
    memory the driver pinned itself or on transparent huge pages: one
    cudaHostRegister of a numpy array per tensor (294 for the 147-tensor model)
    copied at 10-30 GB/s, and a registered mapping advised MADV_HUGEPAGE copied
    at 190-210 GB/s only while the kernel could back all of it with huge pages
    (with 79 % backed, H2D fell to 13 GB/s).  cudaHostAlloc memory copies at
    190-210 GB/s in both directions whatever the state of host memory."""

    ALIGN = 256

    def __init__(self, counts_dtypes):
        import torch
        offsets, o = [], 0
        for n, dt in counts_dtypes:
            offsets.append(o)
            o += (n * torch.empty(0, dtype=dt).element_size() + self.ALIGN - 1) // self.ALIGN * self.ALIGN
        self.nbytes = max(o, self.ALIGN)
        self._raw = torch.empty(self.nbytes, dtype=torch.uint8, pin_memory=True)
        if not self._raw.is_pinned():
            raise SystemExit("e2e: the pinned host allocation is not page-locked")
        self.views = [self._raw[off:off + n * torch.empty(0, dtype=dt).element_size()].view(dt)
                      for off, (n, dt) in zip(offsets, counts_dtypes)]

    def close(self):
        self.views, self._raw = [], None


def adamw_buckets(params, hp, reps=5):
    """AdamW throughput (GB/s at 30 B/param) for the tensors of each size
    decade [10^k, 10^(k+1)), each decade stepped as its own multi-tensor list
    (marshalled once) and timed on the device by the library's launch events
    (kernel time only)."""
    import math as _m
    import torch
    import mixed_precision_optimizer_gb300 as mp
    groups = {}
    for p in params:
        n = p.main_param.numel()
        groups.setdefault(int(_m.log10(n)) if n > 0 else 0, []).append(p)
    out = {}
    for k in sorted(groups):
        g = mp.prepare(groups[k], "adamw")
        n = sum(p.main_param.numel() for p in groups[k])
        mp.adamw_step(g, hp)
        prof = mp.LaunchProfiler(capacity=64 * reps)
        with prof:
            for _ in range(reps):
                mp.adamw_step(g, hp)
        torch.cuda.synchronize()
        recs = prof.records()
        ms = sum(r["ms"] for r in recs) / reps
        out[f"1e{k}-1e{k + 1}"] = {"tensors": len(groups[k]), "params": n, "launches": len(recs) // reps,
                                   "kernel_ms": round(ms, 4),
                                   "gbs": round(n * ADAMW_BYTES_PER_PARAM / (ms * 1e-3) / 1e9, 1)}
    return out


def h2d_sm_share(r_sm, r_ce, t_budget_ms, need_bytes):
    """Share of a step's H2D bytes for the SM loads, the rest going to the
    copy engines, from each path's rate (bytes per ms) on an earlier step:
    the copy engines take what they move in 0.9 of the time budget; when that
    would leave the SM loads the longer of the two, the shares are set for
    both to finish together.  Kept within [0.05, 0.95]."""
    ce_first = 1.0 - 0.9 * r_ce * t_budget_ms / need_bytes
    balanced = r_sm / (r_sm + r_ce)
    return min(max(min(ce_first, balanced), 0.05), 0.95)


def run_e2e(args, step_fn, prepare_set, params, flat, t, total, dist: Dist, group_step=None, step_ms=None):
    """The same step through the public API, with main_grad arriving from
    pinned host memory and the bf16 model parameters read back to host
    memory, every step, inside the timed region.

    The gradients of all tensors form one contiguous buffer, and so do the
    bf16 model copies, laid out group by group (build_device_workload).  With
    `group_step` each step is one library call per step group (a Muon shape
    class, or the AdamW tensors), and each group's gradients are one
    host-to-device segment (shared between the copy engines and SM loads,
    below) and its model copies one device-to-host copy: a group's compute
    starts as soon as its own gradients have landed, and its model copy
    leaves while the next group computes.  Without it (sharded or
    clipped steps, whose calls span every tensor) a step is one call and each
    direction one copy.  The copies are pipelined across steps too: both
    buffers are double-buffered on the device, step k uses set k % 2, and
    events order every reuse of a buffer set."""
    import torch
    import mixed_precision_optimizer_gb300 as mp
    if args.e2e_steps <= 0:
        return None
    K = args.e2e_steps
    n_flat = flat["grad"].numel()
    arena = PinnedHostArena([(n_flat, torch.float32), (n_flat, torch.bfloat16)])
    g_host, b_host = arena.views
    g_host.copy_(flat["grad"])
    if not (g_host.is_pinned() and b_host.is_pinned()):
        raise SystemExit("e2e: host buffers are not page-locked")
    # second device set of gradients and model copies, same layout
    grad2, model2 = torch.empty_like(flat["grad"]), torch.empty_like(flat["model"])
    g2 = flat_views(grad2, flat["offsets"], flat["shapes"])
    b2 = flat_views(model2, flat["offsets"], flat["shapes"])
    sets = [params, [mp.Param(p.main_param, g, p.exp_avg, p.exp_avg_sq, b, p.embedding_or_output, p.kind)
                     for p, g, b in zip(params, g2, b2)]]
    flats = [(flat["grad"], flat["model"]), (grad2, model2)]
    # step groups: (calls per set, flat segment); one group = the whole step
    if group_step is not None:
        groups = []
        for kind, ids, a, b in flat["segments"]:
            preps = [mp.prepare([st[i] for i in ids], "adamw" if kind == "adamw" else None) for st in sets]
            groups.append((lambda tt, si, preps=preps, kind=kind: group_step(tt, preps[si], kind), a, b))
    else:
        preps = [prepare_set(x) for x in sets]
        groups = [(lambda tt, si: step_fn(tt, preps[si]), 0, n_flat)]
    G = len(groups)
    compute = torch.cuda.current_stream()
    # H2D by two paths at once: the copy engines on one stream and SM loads of
    # the pinned buffers (opt_copy_from_host) on another, each taking a share
    # of every segment.  On these hosts either path's host-to-device rate can
    # drop, with the pages, over time and from host to host, and the two share
    # one limit of about 200 GB/s.  The copies need only keep up with the
    # compute, and the SM loads slow the compute more than the copy engines
    # do.  Each step uses the rates the two paths reached on earlier steps
    # (the step two back is finished by then): the copy engines get what they
    # move in 0.9 of the device-resident step time and the SM loads the rest;
    # when that would leave the SM loads the longer of the two, the shares are
    # set for both paths to finish together instead.  At least 5 % each, so
    # that both rates stay measured.  D2H: the copy engines.
    s_sm, s_ce, s_out = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    sm_copy = lambda dst, src, st: mp.copy_from_host(dst, src, stream=st)
    ce_copy = lambda dst, src, st: dst.copy_(src, non_blocking=True)
    # untimed: one pass of each copy direction over every host buffer; the
    # first pass of each H2D path is timed on its own (the SM pass beside the
    # first D2H, then the copy-engine pass) to show this host's copy rates
    # with no compute running, and to set the first step's shares
    E = lambda: torch.cuda.Event(enable_timing=True)
    warm = [E() for _ in range(6)]
    for st in (s_sm, s_ce, s_out):
        st.wait_stream(compute)
    for i, (gd, bd) in enumerate(flats):
        with torch.cuda.stream(s_sm):
            if i == 0:
                warm[0].record(s_sm)
            sm_copy(gd, g_host, s_sm)
            if i == 0:
                warm[1].record(s_sm)
        with torch.cuda.stream(s_ce):
            s_ce.wait_stream(s_sm)
            if i == 0:
                warm[4].record(s_ce)
            ce_copy(gd, g_host, s_ce)
            if i == 0:
                warm[5].record(s_ce)
        with torch.cuda.stream(s_out):
            if i == 0:
                warm[2].record(s_out)
            b_host.copy_(bd, non_blocking=True)
            if i == 0:
                warm[3].record(s_out)
    start = E()
    torch.cuda.synchronize()
    nb_g = g_host.numel() * g_host.element_size()
    idle_gbs = {"h2d": round(nb_g / (warm[0].elapsed_time(warm[1]) * 1e6), 1),
                "d2h": round(b_host.numel() * b_host.element_size() / (warm[2].elapsed_time(warm[3]) * 1e6), 1),
                "h2d_copy_engine": round(nb_g / (warm[4].elapsed_time(warm[5]) * 1e6), 1)}
    need = sum(b - a for _, a, b in groups) * g_host.element_size()
    # first shares from the idle rates; later ones from each path's slowest
    # rate over its last three measured steps (a path's rate can swing several
    # fold from step to step with the pages it reads, and a step lasts as long
    # as its slower path)
    hist = [[idle_gbs["h2d"] * 1e6], [idle_gbs["h2d_copy_engine"] * 1e6]]     # bytes per ms
    ctl = {"f_sm": h2d_sm_share(hist[0][0], hist[1][0], step_ms, need) if step_ms else 0.5, "t": t}

    def rates(run, j):
        """Bytes per ms of each H2D path on step j of a run (finished)."""
        out = []
        for b_ev, e_ev, part in ((run["sm_b"], run["sm_e"], 0), (run["ce_b"], run["ce_e"], 1)):
            tt = sum(b_ev[j][g].elapsed_time(e_ev[j][g]) for g in range(G))
            n = sum((run["cuts"][j][g][1] - run["cuts"][j][g][0]) if part == 0 else
                    (run["cuts"][j][g][2] - run["cuts"][j][g][1]) for g in range(G)) * g_host.element_size()
            out.append(n / tt if tt > 0 and n > 0 else None)
        return out

    def run_steps(n):
        """Enqueues n pipelined steps (H2D on two paths, compute, D2H); the
        shares follow the rates of earlier steps, carried over between runs."""
        ev = lambda: [[E() for _ in range(G)] for _ in range(n)]
        run = {k: ev() for k in ("sm_b", "sm_e", "ce_b", "ce_e", "step_done", "d2h_begin", "d2h_done")}
        run.update(step_begin=[E() for _ in range(n)], cuts=[[None] * G for _ in range(n)], shares=[],
                   host_ms=[0.0, 0.0, 0.0, 0.0])
        sm_b, sm_e, ce_b, ce_e = run["sm_b"], run["sm_e"], run["ce_b"], run["ce_e"]
        step_done, d2h_begin, d2h_done, step_begin = run["step_done"], run["d2h_begin"], run["d2h_done"], \
            run["step_begin"]
        host_ms = run["host_ms"]
        for k in range(n):
            hw = time.perf_counter()
            if k >= 2:
                # at most two steps in flight: step k-2's compute (and so its
                # copies) has finished, and its copy rates set this step's shares
                step_done[k - 2][G - 1].synchronize()
                r_now = rates(run, k - 2)
                if r_now[0] and r_now[1]:
                    for h, r in zip(hist, r_now):
                        h.append(r)
                    t_budget = step_ms if step_ms else step_begin[k - 2].elapsed_time(step_done[k - 2][G - 1])
                    ctl["f_sm"] = h2d_sm_share(min(hist[0][-3:]), min(hist[1][-3:]), t_budget, need)
            h0 = time.perf_counter()
            host_ms[3] += (h0 - hw) * 1e3
            f_sm = ctl["f_sm"]
            run["shares"].append(f_sm)
            gd, bd = flats[k % 2]
            for g, (_, a, b) in enumerate(groups):     # gradients of step k, group by group
                m = a + int((b - a) * f_sm) // 64 * 64
                run["cuts"][k][g] = (a, m, b)
                for st, b_ev, e_ev, lo, hi, copy in ((s_sm, sm_b, sm_e, a, m, sm_copy),
                                                     (s_ce, ce_b, ce_e, m, b, ce_copy)):
                    with torch.cuda.stream(st):
                        if k >= 2:
                            st.wait_event(step_done[k - 2][g])   # step k-2 finished reading this segment
                        b_ev[k][g].record(st)
                        if hi > lo:
                            copy(gd[lo:hi], g_host[lo:hi], st)
                        e_ev[k][g].record(st)
            h1 = time.perf_counter()
            h_step = 0.0
            for g, (call, a, b) in enumerate(groups):
                compute.wait_event(sm_e[k][g])
                compute.wait_event(ce_e[k][g])
                if k >= 2:
                    compute.wait_event(d2h_done[k - 2][g])   # model copy of this segment of set k % 2 read back
                if g == 0:
                    step_begin[k].record(compute)
                c0 = time.perf_counter()
                call(ctl["t"], k % 2)
                h_step += time.perf_counter() - c0
                step_done[k][g].record(compute)
                with torch.cuda.stream(s_out):             # model parameters of this group
                    s_out.wait_event(step_done[k][g])
                    d2h_begin[k][g].record(s_out)
                    b_host[a:b].copy_(bd[a:b], non_blocking=True)
                    d2h_done[k][g].record(s_out)
            ctl["t"] += 1
            h3 = time.perf_counter()
            host_ms[0] += (h1 - h0) * 1e3
            host_ms[1] += h_step * 1e3
            host_ms[2] += ((h3 - h1) - h_step) * 1e3
        return run

    # untimed: as many e2e steps as the bench's warm-up, through the same
    # pipeline, so that the copies and the shares settle before timing
    if args.warmup > 0:
        for st in (s_sm, s_ce, s_out):
            st.wait_stream(compute)
        run_steps(args.warmup)
        torch.cuda.synchronize()
    clocks = ClockSampler(smi_index(torch.cuda.current_device()), "_e2e").__enter__()
    dist.barrier()
    torch.cuda.synchronize()
    t_wall = time.perf_counter()
    start.record(compute)
    for st in (s_sm, s_ce, s_out):
        st.wait_event(start)
    run = run_steps(K)
    sm_b, sm_e, ce_b, ce_e = run["sm_b"], run["sm_e"], run["ce_b"], run["ce_e"]
    step_done, d2h_begin, d2h_done, step_begin = run["step_done"], run["d2h_begin"], run["d2h_done"], \
        run["step_begin"]
    host_ms, shares = run["host_ms"], run["shares"]
    torch.cuda.synchronize()
    wall_ms = (time.perf_counter() - t_wall) * 1e3
    clocks.__exit__(None, None, None)
    dist.barrier()
    ms = dist.max(start.elapsed_time(d2h_done[-1][-1]))
    # untimed: the idle copy rates once more, after the loop (one H2D pass
    # of each path with no compute running), to tell a host whose copies are
    # slow throughout from copies slowed while the loop runs
    after = [E() for _ in range(4)]
    with torch.cuda.stream(s_sm):
        after[0].record(s_sm)
        sm_copy(flats[0][0], g_host, s_sm)
        after[1].record(s_sm)
    with torch.cuda.stream(s_ce):
        s_ce.wait_stream(s_sm)
        after[2].record(s_ce)
        ce_copy(flats[0][0], g_host, s_ce)
        after[3].record(s_ce)
    torch.cuda.synchronize()
    idle_after = {"h2d": round(nb_g / (after[0].elapsed_time(after[1]) * 1e6), 1),
                  "h2d_copy_engine": round(nb_g / (after[2].elapsed_time(after[3]) * 1e6), 1)}
    # a step's H2D spans from the first start to the last end of its parts
    # (the two streams run staggered, so per-segment spans would overlap)
    at = lambda e: start.elapsed_time(e)
    span = [max(max(at(sm_e[k][g]), at(ce_e[k][g])) for g in range(G)) -
            min(min(at(sm_b[k][g]), at(ce_b[k][g])) for g in range(G)) for k in range(K)]
    seg_bytes = [(b - a) * g_host.element_size() for _, a, b in groups]
    step_gbs = sorted(sum(seg_bytes) / (span[k] * 1e6) for k in range(K))
    path_gbs = [[r / 1e6 if r else None for r in rates(run, k)] for k in range(K)]
    med = lambda xs: round(statistics.median(xs), 1) if xs else None
    # device time of each phase per step: the H2D span above, the D2H copies
    # summed over the groups, the step from its first group's start to its
    # last group's end
    phase = {"h2d": round(sum(span) / K, 3),
             "step": round(sum(step_begin[k].elapsed_time(step_done[k][-1]) for k in range(K)) / K, 3),
             "d2h": round(sum(d2h_begin[k][g].elapsed_time(d2h_done[k][g]) for k in range(K) for g in range(G)) / K, 3)}
    h2d = sum((b - a) for _, a, b in groups) * g_host.element_size()
    d2h = sum((b - a) for _, a, b in groups) * b_host.element_size()
    del g_host, b_host
    arena.close()
    per_step = total * (1 if getattr(args, "shard", False) else dist.world)
    return {"value": round(per_step * K / (ms * 1e-3), 1), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "steps": K, "warmup_steps": max(args.warmup, 0), "ms_per_step": round(ms / K, 3),
            "calls_per_step": G,
            "pipelined": ("one library call per step group (each Muon shape class, the AdamW tensors), each "
                          "group's gradients one H2D copy and its bf16 model copies one D2H copy" if G > 1 else
                          "one library call per step; main_grad and bf16 model buffers one copy per direction") +
                         "; buffers double-buffered; H2D, compute and D2H on three streams; the first step's "
                         "first H2D and the last step's last D2H are not overlapped and are included",
            "h2d_by": "two paths at once, each a share of every segment: the copy engines and SM loads of the "
                      "pinned host buffers (opt_copy_from_host), on two streams; the SM share is "
                      "min(1 - 0.9 r_ce T / bytes, r_sm / (r_sm + r_ce)), T the device-resident step time, r each "
                      "path's slowest rate over its last three measured steps (the newest two back; first steps: "
                      "idle rates; 5-95 %, at most two steps in flight); D2H by the copy engines",
            "h2d_paths": {"sm_share": {"first": round(shares[0], 3), "median": round(statistics.median(shares), 3),
                                       "min": round(min(shares), 3), "max": round(max(shares), 3)},
                          "sm_gbs_median": med([r[0] for r in path_gbs if r[0]]),
                          "copy_engine_gbs_median": med([r[1] for r in path_gbs if r[1]]),
                          "by_step": [[round(f, 3), round(r[0] or 0, 1), round(r[1] or 0, 1)]
                                      for f, r in zip(shares, path_gbs)],
                          "by_step_fields": ["sm_share", "sm_gbs", "copy_engine_gbs"]},
            "host_buffers": f"one cudaHostAlloc arena of {arena.nbytes} bytes (torch pinned memory); "
                            "copies warmed once before timing",
            "host_wall_ms_per_step": round(wall_ms / K, 3),
            "host_enqueue_ms_per_step": {"h2d": round(host_ms[0] / K, 3), "step": round(host_ms[1] / K, 3),
                                         "d2h": round(host_ms[2] / K, 3)},
            "host_wait_ms_per_step": round(host_ms[3] / K, 3),
            "device_ms_per_step": phase,
            "h2d_gbs": round(h2d / (phase["h2d"] * 1e6), 1) if phase["h2d"] > 0 else None,
            "d2h_gbs": round(d2h / (phase["d2h"] * 1e6), 1) if phase["d2h"] > 0 else None,
            "copy_gbs_before_timing": idle_gbs,
            "h2d_gbs_after_timing": idle_after,
            "h2d_gbs_per_step": {"min": round(step_gbs[0], 1), "median": round(statistics.median(step_gbs), 1),
                                 "max": round(step_gbs[-1], 1)},
            "clocks": clocks.summary()}


# --------------------------------------------------------- reference arm --

def run_reference(args, dist: Dist):
    """The oracle, as it stands, on this host's cores: every step is one run of
    the fixed sample of cpu_oracle_sample (the same sample as our arm's
    cpu_baseline), extrapolated to the whole workload."""
    w = S.WORKLOADS[args.workload]()
    total = w.numel
    for _ in range(args.warmup):
        cpu_oracle_sample(w)
    times, desc = [], None
    for _ in range(args.steps):
        t, desc = cpu_oracle_sample(w)
        times.append(t)
    t_step = statistics.mean(times)
    value = total / t_step
    base = cpu_baseline_entry(w, t_step, desc, total)
    return {"metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": dist.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(t_step * 1e3, 1), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "dtype_detail": "CPU oracle: fp32 AdamW in literal operation order, fp64 Muon and Newton-Schulz",
            "data": "synthetic (seeded)", "impl": "reference",
            "config": workload_config(w, args.clip), "parallelism": "CPU oracle on rank 0",
            "cpu_baseline": base,
            "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    if args.steps < 1 or args.warmup < 0:
        raise SystemExit("--steps >= 1, --warmup >= 0")
    ClockSampler.log_dir = args.clock_log
    dist = Dist()
    try:
        if args.impl == "reference":
            if dist.rank != 0:
                return
            line = run_reference(args, dist)
        else:
            line = run_ours(args, dist)
        if dist.rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
