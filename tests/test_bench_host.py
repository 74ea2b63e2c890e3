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
    4 m^2 n + 2 m^3 (per matrix)."""
    for A, B in ((1024, 4096), (4096, 14336), (256, 512)):
        recs = [dict(kernel=k, count=3, a=A, b=B) for k in ("ns_gram", "ns_poly", "ns_bx")]
        assert sum(bench.gemm_flops(r) for r in recs) == 3 * OM.ns_flops(A, B, 1)
        # executed <= algorithmic for the symmetric stages
        assert bench.gemm_executed_flops(recs[0]) < bench.gemm_flops(recs[0]) or A == 256


def test_reference_arm_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_mixed", "--steps", "1", "--warmup", "0"], capture_output=True, text=True,
                       timeout=600, env=dict(os.environ, WORLD_SIZE="1"))
    assert r.returncode == 0, r.stderr
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "params/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0


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
    (tmp_path / "profiles" / "dram_traffic_llama16_mixed.md").write_text(f"| ns_gemm | {sha} | 1.5e9 |\n| adamw | 0000000000000000 | 3e9 |\n")
    (tmp_path / "profiles" / "ns_gemm_llama_mlp_1layer.md").write_text(f"| tensor_pipe | {sha} | 70.5 | 60.0 | 85.25 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.kernel_traffic("ns_gemm") == 1.5e9
    assert bench.kernel_traffic("adamw") is None          # captured from another source
    tp = bench.tensor_pipe_active()
    assert (tp["gram"], tp["poly"], tp["bx"]) == (70.5, 60.0, 85.25)
    (csrc / "ns_gemm.cu").write_bytes(b"kernel v2")       # source changed since the capture
    assert bench.kernel_traffic("ns_gemm") is None and bench.tensor_pipe_active() is None


def test_kernels_by_shape_groups_stages_and_classes():
    recs = [dict(kernel="ns_gram", count=48, a=4096, b=14336, ms=7.5),
            dict(kernel="ns_gram", count=48, a=4096, b=14336, ms=7.3),
            dict(kernel="ns_bx", count=32, a=1024, b=4096, ms=0.2),
            dict(kernel="adamw", count=2, a=1000, b=0, ms=5.0)]
    out = bench.kernels_by_shape(recs)
    assert set(out) == {"ns_gram 4096x14336 x48", "ns_bx 1024x4096 x32"}
    g = out["ns_gram 4096x14336 x48"]
    assert g["launches"] == 2 and g["ms_per_launch"] == 7.4
    # algorithmic 2 A^2 B per matrix; executed: 136 of the 256 blocks
    assert g["tflops_algorithmic"] == round(48 * 2.0 * 4096 ** 2 * 14336 / 7.4e-3 / 1e12, 1)
    assert g["tflops_executed"] == round(48 * 136 * 2.0 * 256 * 256 * 14336 / 7.4e-3 / 1e12, 1)
