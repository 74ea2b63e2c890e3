"""Host logic of bench.py on the CPU: replica timing over a world-size-2 gloo
group, clock-log parsing, the flop accounting of the roofline, and the
reference (oracle) arm's JSON line on the small workload."""

import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from oracle import muon as OM  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    d = bench.Dist()
    d.barrier()
    q.put((rank, d.max(10.0 + rank)))
    d.close()


def test_max_over_ranks_gloo_world_2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_clock_summary_parsing(tmp_path):
    cs = bench.ClockSampler(0)
    cs.path = str(tmp_path / "c.csv")
    with open(cs.path, "w") as f:
        f.write("0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active\n")
        f.write("0, 1950, 2070, 1000.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
        f.write("0, 300, 2070, 100.0, 0x0, Not Active, Not Active, Not Active, Not Active\n")
    cs.proc = object()
    s = cs.summary()
    assert s["sm_mhz"] == 1925.0 and s["sm_max_mhz"] == 2070.0 and s["reasons"] == ["sw_power_cap"]
    assert "mem_mhz" not in s
    # with the memory clock and temperature columns
    with open(cs.path, "w") as f:
        f.write("0, 1900, 2070, 900.5, 0x0, Not Active, Not Active, Not Active, Active, 3996, 61\n")
        f.write("0, 1700, 2070, 1000.0, 0x0, Not Active, Active, Not Active, Not Active, 3996, 74\n")
    s = cs.summary()
    assert s["sm_mhz"] == 1800.0 and s["mem_mhz"] == 3996.0 and s["temp_c_max"] == 74.0
    assert s["reasons"] == ["hw_thermal_slowdown", "sw_power_cap"]


def test_smi_index(monkeypatch):
    monkeypatch.setenv("CUDA_VISIBLE_DEVICES", "3,5")
    assert bench.smi_index(1) == 5
    monkeypatch.delenv("CUDA_VISIBLE_DEVICES")
    assert bench.smi_index(2) == 2


def test_gemm_flop_accounting_matches_pages_formula():
    """One Newton-Schulz iteration's three launches add up to the pages'
    4 m^2 n + 2 m^3 per matrix (dense count, put on the C X that completes the
    iteration); the launches' own count (the roofline's) takes the symmetric
    products at their triangle, 3 m^2 n + m^3; the executed count lies between
    the two for large shapes."""
    for A, B in ((1024, 4096), (4096, 14336), (256, 512)):
        recs = bench.annotate_iterations([dict(kernel=k, count=3, a=A, b=B) for k in ("ns_gram", "ns_poly", "ns_bx")])
        pages = sum(bench.gemm_pages_flops(r) for r in recs)
        assert pages == 3 * OM.ns_flops(A, B, 1)
        assert sum(bench.gemm_method_flops(r) for r in recs) == 3 * (3 * A * A * B + A ** 3)
        ex = sum(bench.gemm_executed_flops(r) for r in recs)
        assert sum(bench.gemm_method_flops(r) for r in recs) <= ex <= pages
        # executed below the dense count for the symmetric stage
        assert bench.gemm_executed_flops(recs[0]) < 2.0 * 3 * A * A * B or A == 256


def test_grouped_iteration_accounting():
    """A group of g iterations is one X X^T, g polynomials, 3 (g - 1) more
    symmetric [A][A] products and one C X: its own count is 3 A^2 B +
    (4 g - 3) A^3 per matrix, and the pages' count of its g iterations lands on
    the C X.  Five iterations as groups of 3 and 2 count the pages' five."""
    A, B, n = 4096, 14336, 48
    recs = []
    for g in (3, 2):
        recs.append(dict(kernel="ns_gram", count=n, a=A, b=B))
        recs.append(dict(kernel="ns_poly", count=n, a=A, b=B))
        for _ in range(g - 1):
            recs += [dict(kernel="ns_sym", count=n, a=A, b=B), dict(kernel="ns_sym", count=n, a=A, b=B),
                     dict(kernel="ns_poly", count=n, a=A, b=B), dict(kernel="ns_sym", count=n, a=A, b=B)]
        recs.append(dict(kernel="ns_bx", count=n, a=A, b=B))
    bench.annotate_iterations(recs)
    assert [r["iters"] for r in recs if r["kernel"] == "ns_bx"] == [3, 2]
    assert sum(bench.gemm_pages_flops(r) for r in recs) == n * OM.ns_flops(A, B, 5)
    me = sum(bench.gemm_method_flops(r) for r in recs)
    assert me == n * sum(3 * A * A * B + (4 * g - 3) * A ** 3 for g in (3, 2))
    per_iteration = n * 5 * (3 * A * A * B + A ** 3)
    assert 0.6 < me / per_iteration < 0.65          # 39 % fewer flops for this shape


def _run_bench(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run_bench("--impl", "reference", "--workload", "tiny_mixed", "--steps", "1", "--warmup", "0")
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["cpu_baseline"]["value"] == d["value"] and d["cpu_baseline"]["extrapolated"] is False
    # the same config dict as our arm builds for the workload
    assert d["config"] == bench.workload_config(bench.S.tiny_mixed(), 0.0)


def test_cpu_sample_is_shared_and_fixed():
    """Both arms time one fixed sample: the Muon classes whose Newton-Schulz
    is small enough run through the oracle, larger ones are extrapolated and
    say so."""
    w = bench.S.llama16_mixed()
    t, desc = bench.cpu_oracle_sample(bench.S.scaled_copy(bench.S.muon_8m_skewed(), "two", [(64, 128), (128, 64)]))
    assert t > 0 and desc["extrapolated"] is True        # two matrices of one class, timed on one
    classes = {tuple(sorted(sp.shape)) for sp in w.tensors if bench.is_muon(w, sp)}
    runs = sorted(c for c in classes if OM.ns_flops(*c) <= bench.MUON_SAMPLE_FLOPS)
    assert runs == [(1024, 4096)]


def test_profile_rows_apply_only_to_their_source(tmp_path, monkeypatch):
    """traffic and tensor-pipe rows are used only while the kernel source has the
    sha256 prefix they were captured from."""
    import hashlib
    csrc = tmp_path / "mixed_precision_optimizer_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    (csrc / "ns_gemm.cu").write_bytes(b"kernel v1")
    (csrc / "adamw.cu").write_bytes(b"adamw v1")
    sha = hashlib.sha256(b"kernel v1").hexdigest()[:16]
    rows = {"ns_gemm_traffic": {"source": "ns_gemm.cu", "sha256_16": sha, "bytes_per_launch": 1.5e9},
            "adamw_traffic": {"source": "adamw.cu", "sha256_16": "0000000000000000", "bytes_per_launch": 3e9},
            "ns_gemm_tensor_pipe": {"source": "ns_gemm.cu", "sha256_16": sha,
                                    "pct": {"gram": 70.5, "poly": 60.0, "bx": 85.25}}}
    (tmp_path / "profiles" / "rows.json").write_text(json.dumps(rows))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profile_row("ns_gemm_traffic")["bytes_per_launch"] == 1.5e9
    assert bench.profile_row("adamw_traffic") is None          # captured from another source
    assert bench.profile_row("ns_gemm_tensor_pipe")["pct"]["bx"] == 85.25
    (csrc / "ns_gemm.cu").write_bytes(b"kernel v2")       # source changed since the capture
    assert bench.profile_row("ns_gemm_traffic") is None and bench.profile_row("ns_gemm_tensor_pipe") is None


def test_kernels_by_shape_groups_stages_and_classes():
    recs = [dict(kernel="ns_gram", count=48, a=4096, b=14336, ms=7.5),
            dict(kernel="ns_gram", count=48, a=4096, b=14336, ms=7.3),
            dict(kernel="ns_bx", count=32, a=1024, b=4096, ms=0.2),
            dict(kernel="adamw", count=2, a=1000, b=0, ms=5.0)]
    out = bench.kernels_by_shape(recs, 1700.0)
    assert set(out) == {"ns_gram 4096x14336 x48", "ns_bx 1024x4096 x32"}
    g = out["ns_gram 4096x14336 x48"]
    assert g["launches"] == 2 and g["ms_per_launch"] == 7.4
    # the launch's own count A^2 B per matrix; executed: 136 of the 256 blocks
    assert g["tflops_method"] == round(48 * 1.0 * 4096 ** 2 * 14336 / 7.4e-3 / 1e12, 1)
    ex = 48 * 136 * 2.0 * 256 * 256 * 14336 / 7.4e-3 / 1e12
    assert g["tflops_executed"] == round(ex, 1) and g["executed_frac"] == round(ex / 1700.0, 3)


def test_measured_line_roofline_follows_from_the_kernels():
    """frac = the launches' own flops / their event time / the sustained peak;
    the executed count and the pages' iteration-equivalent rate beside it."""
    class A:
        steps, clip, warmup = 2, 0.0, 1
    class D:
        world = 1
    recs = []
    for _ in range(2):
        for k, ms in (("ns_gram", 7.0), ("ns_poly", 2.0), ("ns_bx", 14.0)):
            recs.append(dict(kernel=k, count=48, a=4096, b=14336, ms=ms))
        recs.append(dict(kernel="adamw", count=35, a=1_000_000, b=0, ms=0.01))
    peaks = {"hbm_gbs": 6787.2, "bf16_tflops": 1875.3, "bf16_tflops_sustained": 1708.2}
    w = bench.S.llama_mlp_1layer()
    line = bench.measured_line(A, w, recs, len(recs), 50.0, w.numel, D, peaks, "measured")
    r = line["roofline"]
    me = sum(bench.gemm_method_flops(x) for x in recs if x["kernel"] != "adamw")
    ms = sum(x["ms"] for x in recs if x["kernel"] != "adamw")
    assert r["achieved"] == round(me / (ms * 1e-3) / 1e12, 1)
    assert r["frac"] == round(me / (ms * 1e-3) / 1e12 / 1708.2, 4)
    assert r["executed_frac"] > r["frac"] and r["pages_count_tflops"] > r["executed_tflops"]
    assert r["pages_count_tflops"] == round(2 * 48 * OM.ns_flops(4096, 14336, 1) / (ms * 1e-3) / 1e12, 1)
    a = line["roofline_adamw"]
    assert a["frac_of_nominal_8tbs"] == round(a["achieved"] / 8000.0, 4)


def test_flat_buffers_hold_step_groups_contiguously():
    """The e2e leg copies one segment of the flat gradient and model buffers
    per step group: every tensor of a group lies inside its group's segment,
    the segments tile the buffer in order, and the groups are each Muon shape
    class (smallest first) and then the AdamW tensors."""
    import torch
    w = bench.S.scaled_copy(bench.S.tiny_mixed(), "groups",
                            [(64, 96), (7,), (96, 64), (40, 40), (300,), (40, 40), (3, 5, 2)])
    params, n_muon, n_adamw, flat = bench.build_device_workload(w, torch.device("cpu"))
    segs = flat["segments"]
    assert [k for k, *_ in segs] == ["muon", "muon", "adamw"]
    assert sorted(map(tuple, (segs[0][1], segs[1][1]))) == [(0, 2), (3, 5)]
    assert segs[0][1] == [3, 5]                           # 40 x 40 class (3200) before 64 x 96 (12288)
    assert segs[0][2] == 0 and segs[-1][3] == flat["grad"].numel()
    assert all(a[3] == b[2] for a, b in zip(segs, segs[1:]))
    base = flat["grad"].data_ptr()
    for kind, ids, a, b in segs:
        for i in ids:
            off = (params[i].main_grad.data_ptr() - base) // 4
            assert a <= off and off + params[i].main_grad.numel() <= b
            assert (params[i].model.data_ptr() - flat["model"].data_ptr()) // 2 == off
    assert n_muon + n_adamw == w.numel


def test_h2d_share_rule():
    """The e2e leg's split of each step's gradients between the copy engines
    and SM loads: copy engines first while they keep up with the step,
    balanced when neither path alone does, never below 5 % for either."""
    need, T = 18.2e9, 118.0                              # bytes per step, ms
    assert bench.h2d_sm_share(200e6, 200e6, T, need) == 0.05         # copy engines cover the step
    f = bench.h2d_sm_share(200e6, 30e6, T, need)                      # slow copy engines
    assert abs(f - (1 - 0.9 * 30e6 * T / need)) < 1e-12
    assert (1 - f) * need / 30e6 <= 0.9 * T + 1e-9 and f * need / 200e6 < 0.9 * T
    f = bench.h2d_sm_share(100e6, 50e6, T, need)                      # both slow: finish together
    assert abs(f - 100 / 150) < 1e-12
    assert abs(f * need / 100e6 - (1 - f) * need / 50e6) < 1e-6
    assert bench.h2d_sm_share(200e6, 1e3, T, need) == 0.95            # copy engines all but stalled
