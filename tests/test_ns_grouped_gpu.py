"""Grouped Newton-Schulz iterations on the GPU, through the C ABI, against the
fp64 oracle's iteration as printed ("02 · Optimizer：算法与 infra" §5.2;
"优化器：AdamW、Muon 与分布式优化器", newton_schulz in the Muon section).

Every polynomial C_k = a I + b A_k + c A_k A_k of an iteration is a polynomial
in the Gram matrix A_k0 of the group's first iterate, so the factors commute
and, exactly, A_{k+1} = C_k A_k C_k and X_{k0+g} = C_{k0+g-1} ... C_k0 X_k0.
A group of g iterations therefore needs one X X^T and one C X.  Grouped and
per-iteration evaluation differ only in rounding, so both meet the bar of
every Muon test: the update within 2e-2 relative Frobenius error of the
oracle; on rectangular matrices every singular value of the output in
[0.6, 1.3]; on square ones the sorted singular values within 0.05 of the
oracle's and none above 1.3.

Each test reads back the launches its call made (opt_profile_launches), so
that it checks the evaluation order it asks for is the one that ran: a group
of g iterations launches one X X^T, g polynomials, 3 (g - 1) products of
symmetric [A][A] matrices and one C X.
"""

import numpy as np
import pytest

from gpu_helpers import assert_square_spectrum, bf16_host, dev, host, require_gpu, singular_values, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
from oracle import muon as OM
import synthetic as S

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def group_sizes(steps):
    """The library's split of `steps` iterations: ceil(steps / 3) groups as
    equal as possible, the larger first."""
    n = -(-steps // 3)
    return [steps // n + (1 if k < steps % n else 0) for k in range(n)]


def expected_launches(steps, grouped):
    sizes = group_sizes(steps) if grouped else [1] * steps
    return {"ns_gram": len(sizes), "ns_poly": steps, "ns_sym": sum(3 * (g - 1) for g in sizes),
            "ns_bx": len(sizes)}


def muon_step_gpu(W, g, m, hp, ns_order, ws_order=None):
    """One Muon step on the device; returns the new master, momentum, bf16
    copy and the launch count of each Newton-Schulz GEMM stage."""
    Wd, gd, md = dev(W), dev(g), dev(m)
    Wb = torch.zeros(W.shape, dtype=torch.bfloat16, device="cuda")
    p = mp.Param(Wd, gd, md, None, Wb)
    ws = mp.alloc_workspace(mp.workspace_size([p], "muon", ns_order=ws_order or ns_order))
    with mp.LaunchProfiler(256) as prof:
        mp.muon_step(p, hp, ws)
    torch.cuda.synchronize()
    assert mp.device_status(ws) == mp.OPT_OK
    counts = {}
    for r in prof.records():
        counts[r["kernel"]] = counts.get(r["kernel"], 0) + 1
    stages = {k: counts.get(k, 0) for k in ("ns_gram", "ns_poly", "ns_sym", "ns_bx")}
    return host(Wd), host(md), bf16_host(Wb), stages


def check_update(shape, W, W1, Wn, lr):
    """The update within NS_TOL of the oracle's.  Its singular values lie in
    [0.6, 1.3] wherever the oracle's do; where even the exact iteration leaves
    some below 0.6 (square matrices, or a rank-8 component that dominates the
    norm of a 1024 x 2048 gradient), the sorted singular values match the
    oracle's within 0.05 and none exceeds 1.3."""
    s = lr * OM.update_scale(*shape)
    upd = (W.astype(np.float64) - W1) / s
    want = (W.astype(np.float64) - Wn) / s
    assert rel(upd, want) < NS_TOL
    if min(shape) > 1:
        sw = singular_values(want)
        if 0.6 <= sw.min() and sw.max() <= 1.3:
            sv = singular_values(upd)
            assert 0.6 <= sv.min() and sv.max() <= 1.3, (sv.min(), sv.max())
        else:
            assert_square_spectrum(upd, want, f"grouped {shape}")


@pytest.mark.parametrize("shape", [(300, 700), (700, 300), (127, 257), (256, 512), (512, 1536), (96, 96),
                                   (512, 512), (1, 64), (64, 1), (1, 1)])
def test_grouped_muon_step_matches_oracle(shape):
    """Forced grouping (two groups of 3 and 2 iterations) on ragged, tall,
    wide, square and degenerate shapes."""
    rng = np.random.default_rng(shape[0] * 13 + shape[1])
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    lr, mu = 0.02, 0.95
    W1, m1, Wb, stages = muon_step_gpu(W, g, m, mp.muon_hp(lr=lr, momentum=mu, ns_order="grouped"), "grouped")
    assert stages == expected_launches(5, True)
    Wn, mn, _ = OM.muon_step(W, g, m, lr=lr, momentum=mu)
    check_update(shape, W, W1, Wn, lr)
    assert np.allclose(m1, mn, rtol=1e-5, atol=1e-9)
    assert np.array_equal(Wb, OA.bf16_rne(W1))


@pytest.mark.parametrize("steps", [2, 3, 4, 6, 7, 8])
def test_grouped_step_counts(steps):
    """Every split of the iterations into groups of at most three."""
    shape = (300, 700)
    rng = np.random.default_rng(100 + steps)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = np.zeros(shape, np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    hp = mp.muon_hp(ns_steps=steps, ns_order="grouped")
    W1, _, _, stages = muon_step_gpu(W, g, m, hp, "grouped")
    assert stages == expected_launches(steps, True)
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95, ns_steps=steps)
    check_update(shape, W, W1, Wn, 0.02)


def test_grouped_coefficient_schedule():
    """A different (a, b, c) in every iteration: each polynomial of a group
    takes its own iteration's coefficients.  The schedule keeps the iteration
    bounded on every singular value in [0, 1] (each quintic maps the range
    the previous ones reach back into [0, 1.22]), so the plan keeps both
    groups; a schedule that lets singular values near 1 grow without bound
    is split into single iterations (test_abi_host.py)."""
    shape = (384, 1000)
    sched = [(3.4445, -4.7750, 2.0315), (3.2, -4.4, 1.9), (3.0, -4.0, 1.7), (2.8, -3.6, 1.55), (2.2, -2.1, 0.9)]
    assert mp.ns_plan(*shape, mp.muon_hp(schedule=sched, ns_order="grouped")) == [3, 2]
    rng = np.random.default_rng(7)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = np.zeros(shape, np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    W1, _, _, stages = muon_step_gpu(W, g, m, mp.muon_hp(schedule=sched, ns_order="grouped"), "grouped")
    assert stages == expected_launches(5, True)
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95, coeffs=sched)
    assert rel(W.astype(np.float64) - W1, W.astype(np.float64) - Wn) < NS_TOL


@pytest.mark.parametrize("shape,default_grouped", [((1024, 4096), True), ((4096, 1024), True),
                                                   ((1024, 2048), True), ((768, 2048), False),
                                                   ((1024, 1024), False)])
def test_default_order_and_per_iteration_agree(shape, default_grouped):
    """The default groups the shapes where it saves tensor-core work (padded
    max side >= 2 x padded min side, min side >= 1024) and evaluates the
    others per iteration; OPT_MUON_NS_PER_ITERATION never groups.  Both
    orders meet the bar on the skewed workload gradient (rank-8 component of
    10x the noise RMS)."""
    spec = S.TensorSpec("w", shape, "normal", 0.02, 1e-3, lowrank=8, lowrank_rms=1e-2)
    W = S.init_value(spec, 0)
    g = S.grad_value(spec, 0, 1)
    m = np.zeros(shape, np.float32)
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)
    out = {}
    for order in ("auto", "per_iteration"):
        W1, _, _, stages = muon_step_gpu(W, g, m, mp.muon_hp(ns_order=order), order)
        assert stages == expected_launches(5, order == "auto" and default_grouped), order
        check_update(shape, W, W1, Wn, 0.02)
        out[order] = W1
    if default_grouped:
        # two roundings of the same polynomial: close to each other as well
        assert rel(W.astype(np.float64) - out["auto"], W.astype(np.float64) - out["per_iteration"]) < NS_TOL


def test_grouping_falls_back_without_room():
    """Forced grouping in a workspace sized for per-iteration buffers only
    (one matrix's worth): the step evaluates per iteration and still meets
    the bar."""
    shape = (300, 700)
    rng = np.random.default_rng(5)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = np.zeros(shape, np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    W1, _, _, stages = muon_step_gpu(W, g, m, mp.muon_hp(ns_order="grouped"), "grouped", ws_order="auto")
    assert stages == expected_launches(5, False)
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)
    check_update(shape, W, W1, Wn, 0.02)


def test_grouped_three_consecutive_steps_batched_both_orientations():
    """Three Muon steps of a group of same-shape matrices in both
    orientations (one batched launch per stage), momentum carried across
    steps, against the oracle step by step."""
    shapes = [(1024, 2048), (2048, 1024), (1024, 2048)]
    rng = np.random.default_rng(9)
    Ws = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    params, hW, hm = [], [w.astype(np.float64) for w in Ws], [np.zeros(s) for s in shapes]
    for w, s in zip(Ws, shapes):
        params.append(mp.Param(dev(w), torch.zeros(s, device="cuda"), torch.zeros(s, device="cuda"), None,
                               torch.zeros(s, dtype=torch.bfloat16, device="cuda")))
    ws = mp.alloc_workspace(mp.workspace_size(params, "muon"))
    hp = mp.muon_hp()
    for step in range(3):
        gs = [(rng.standard_normal(s) * 1e-2).astype(np.float32) for s in shapes]
        for p, gh in zip(params, gs):
            p.main_grad.copy_(torch.from_numpy(gh))
        W0 = [host(p.main_param).copy() for p in params]
        with mp.LaunchProfiler(256) as prof:
            mp.mixed_step(params, hp, None, ws)
        torch.cuda.synchronize()
        assert mp.device_status(ws) == mp.OPT_OK
        kinds = [r["kernel"] for r in prof.records()]
        assert kinds.count("ns_sym") == 9 and kinds.count("ns_bx") == 2   # one batched group, [3, 2]
        for i, (p, gh) in enumerate(zip(params, gs)):
            Wn, mn, _ = OM.muon_step(W0[i], gh, hm[i], lr=0.02, momentum=0.95)
            hm[i] = host(p.exp_avg).astype(np.float64)
            assert rel(W0[i].astype(np.float64) - host(p.main_param), W0[i].astype(np.float64) - Wn) < NS_TOL
            assert np.allclose(hm[i], mn, rtol=1e-5, atol=1e-9)
            assert np.array_equal(bf16_host(p.model), OA.bf16_rne(host(p.main_param)))


@pytest.mark.parametrize("case", ["default_wide", "default_square", "forced", "per_iteration", "split"])
def test_launches_follow_the_plan(case):
    """The GEMM launches of a step are the ones opt_ns_plan reports for the
    matrix (host only), including a group split because its product could
    leave fp16's range: two iterations that multiply every singular value by
    70 bound the pair by about 4998 > 4096, so they run one at a time (the
    result is 4900 X0, as in the oracle)."""
    shape, hp, ws_order = {
        "default_wide": ((1024, 2048), mp.muon_hp(), "auto"),
        "default_square": ((512, 512), mp.muon_hp(), "auto"),
        "forced": ((300, 700), mp.muon_hp(ns_order="grouped", ns_steps=7), "grouped"),
        "per_iteration": ((1024, 4096), mp.muon_hp(ns_order="per_iteration"), "auto"),
        "split": ((300, 700), mp.muon_hp(ns_order="grouped", ns_steps=2, schedule=[(70.0, 0.0, 0.0)] * 2),
                  "grouped"),
    }[case]
    plan = mp.ns_plan(*shape, hp)
    rng = np.random.default_rng(len(case))
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = np.zeros(shape, np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    W1, _, _, stages = muon_step_gpu(W, g, m, hp, ws_order)
    assert stages == {"ns_gram": len(plan), "ns_poly": sum(plan), "ns_sym": sum(3 * (k - 1) for k in plan),
                      "ns_bx": len(plan)}, (plan, stages)
    if case == "split":
        assert plan == [1, 1]
    coeffs = [(hp.ns_schedule[3 * i], hp.ns_schedule[3 * i + 1], hp.ns_schedule[3 * i + 2])
              for i in range(hp.ns_steps)] if hp.ns_schedule else OM.NS_COEFFS
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95, ns_steps=hp.ns_steps, coeffs=coeffs)
    assert rel(W.astype(np.float64) - W1, W.astype(np.float64) - Wn) < NS_TOL


@pytest.mark.parametrize("case", ["more_than_64", "workspace_for_two"])
def test_grouped_batches(case):
    """A class of 70 matrices runs as batches of at most 64; a workspace with
    room for the grouped buffers of two matrices runs five matrices two at a
    time.  Every matrix matches the oracle, and the launches show the batches."""
    shape = (96, 200)
    n = 70 if case == "more_than_64" else 5
    rng = np.random.default_rng(n)
    Ws = [(rng.standard_normal(shape) * 0.02).astype(np.float32) for _ in range(n)]
    gs = [(rng.standard_normal(shape) * 1e-2).astype(np.float32) for _ in range(n)]
    params = [mp.Param(dev(W), dev(g), torch.zeros(shape, device="cuda"), None,
                       torch.zeros(shape, dtype=torch.bfloat16, device="cuda")) for W, g in zip(Ws, gs)]
    hp = mp.muon_hp(ns_order="grouped")
    if case == "more_than_64":
        nbytes = mp.workspace_size(params, "muon", ns_order="grouped")
        batches = [64, 6]
    else:
        nbytes = mp.workspace_size(params[:2], "muon", ns_order="grouped")
        batches = [2, 2, 1]
    ws = mp.alloc_workspace(nbytes)
    with mp.LaunchProfiler(1024) as prof:
        mp.mixed_step(params, hp, None, ws)
    torch.cuda.synchronize()
    assert mp.device_status(ws) == mp.OPT_OK
    bx = [r["count"] for r in prof.records() if r["kernel"] == "ns_bx"]
    assert bx == [b for b in batches for _ in range(2)]          # two groups of iterations per batch
    for W, g, p in zip(Ws, gs, params):
        Wn, _, _ = OM.muon_step(W, g, np.zeros(shape, np.float32), lr=0.02, momentum=0.95)
        check_update(shape, W, host(p.main_param), Wn, 0.02)
