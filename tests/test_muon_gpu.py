"""Muon parity on the GPU, through the C ABI, against the fp64 oracle.

Tolerance (the bar for the Muon update): the update, and the Newton-Schulz
output, within 2e-2 relative Frobenius error of the oracle's fp64
Newton-Schulz; on rectangular matrices every singular value of the output
in [0.6, 1.3]; on square matrices the sorted singular values of the output
within 0.05 of the oracle's and none above 1.3 (gpu_helpers).  The momentum buffer is fp32 arithmetic on the same inputs:
within 1e-5 relative per element (a few fp32 roundings).  The bf16 model copy
is bit-exact against round-to-nearest-even of the GPU's own master weights.
"""

import math

import numpy as np
import pytest

from gpu_helpers import assert_square_spectrum, bf16_host, dev, host, require_gpu, singular_values, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
from oracle import muon as OM
import oracle_pins as PINS
import synthetic as S

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def ns_gpu(G: np.ndarray, steps=5):
    Gd = dev(G.astype(np.float32))
    out = torch.empty_like(Gd)
    ws = mp.alloc_workspace(mp.newton_schulz_workspace_size(*G.shape))
    mp.newton_schulz(Gd, out, steps=steps, workspace=ws)
    assert mp.device_status(ws) == mp.OPT_OK
    return host(out).astype(np.float64)


# ----------------------------------------------------------- Newton-Schulz --

@pytest.mark.parametrize("shape", [(8, 16), (16, 8), (127, 257), (257, 127), (256, 512), (300, 200),
                                   (512, 512), (1, 64), (64, 1), (1, 1), (1000, 3000)])
@pytest.mark.parametrize("steps", [1, 5])
def test_newton_schulz_gaussian(shape, steps):
    rng = np.random.default_rng(hash(shape) % 2 ** 32 + steps)
    G = rng.standard_normal(shape).astype(np.float32)
    want = OM.newton_schulz(G.astype(np.float64), steps)
    got = ns_gpu(G, steps)
    assert rel(got, want) < NS_TOL


@pytest.mark.parametrize("shape", [(1024, 4096), (4096, 1024)])
def test_newton_schulz_skewed_spectrum_workload_shapes(shape):
    spec = S.TensorSpec("w", shape, "normal", 0.02, 1e-3, lowrank=8, lowrank_rms=1e-2)
    G = S.grad_value(spec, 0, 1)
    want = OM.newton_schulz(G.astype(np.float64))
    got = ns_gpu(G)
    assert rel(got, want) < NS_TOL
    sv = np.linalg.svd(got, compute_uv=False)
    assert 0.6 <= sv.min() and sv.max() <= 1.3


def test_newton_schulz_printed_spectrum():
    """The orthogonalize.py input of "优化器：AdamW、Muon 与分布式优化器"
    (256 x 1024, spectrum logspace(0, -2)); the GPU output reproduces the
    printed 5-step ranges to the printed two decimals (min within 0.01)."""
    rng = np.random.default_rng(0)
    U = PINS.random_orthonormal(rng, 256, 256)
    V = PINS.random_orthonormal(rng, 1024, 256)
    S_ = np.logspace(0, -2, 256)
    G = (U * S_) @ V.T
    got = ns_gpu(G.astype(np.float32), 5)
    want = OM.newton_schulz(G, 5)
    assert rel(got, want) < NS_TOL
    s = np.linalg.svd(got, compute_uv=False)
    assert abs(s.min() - 0.68) < 0.015 and abs(s.max() - 1.20) < 0.015
    frac = np.mean((s > 0.7) & (s < 1.2))
    assert abs(frac - 0.89) < 0.03


def test_newton_schulz_zero_steps_is_normalisation():
    rng = np.random.default_rng(3)
    G = rng.standard_normal((40, 70)).astype(np.float32)
    got = ns_gpu(G, 0)
    want = G.astype(np.float64) / (np.linalg.norm(G.astype(np.float64)) + 1e-7)
    assert rel(got, want) < 1e-6


def test_newton_schulz_diagonal_special_case():
    """A diagonal input: the iteration acts on each diagonal entry with the
    scalar quintic (the per-singular-value form)."""
    d = np.linspace(0.1, 1.0, 64)
    G = np.zeros((64, 128))
    G[np.arange(64), np.arange(64)] = d
    got = ns_gpu(G.astype(np.float32), 5)
    want = np.zeros_like(G)
    want[np.arange(64), np.arange(64)] = PINS.phi_iterate(d / (np.linalg.norm(d) + 1e-7), 5)
    assert rel(got, want) < NS_TOL


@pytest.mark.parametrize("shape,kind", [((96, 96), "gaussian"), ((512, 512), "gaussian"),
                                        ((1024, 1024), "gaussian"), ((512, 512), "skewed"),
                                        ((257, 257), "gaussian")])
def test_newton_schulz_square_spectrum(shape, kind):
    """Square matrices are not transposed, and their near-zero singular values
    stay small after five steps: the output's sorted singular values match the
    fp64 oracle's (each within 0.05) and none exceeds 1.3 ("02 · Optimizer：
    算法与 infra" §5.2: the iteration acts on each singular value with the
    quintic)."""
    rng = np.random.default_rng(shape[0] * 3 + (kind == "skewed"))
    if kind == "gaussian":
        G = rng.standard_normal(shape).astype(np.float32)
    else:
        spec = S.TensorSpec("w", shape, "normal", 0.02, 1e-3, lowrank=8, lowrank_rms=1e-2)
        G = S.grad_value(spec, 0, 1)
    want = OM.newton_schulz(G.astype(np.float64))
    got = ns_gpu(G)
    assert rel(got, want) < NS_TOL
    assert_square_spectrum(got, want, f"{shape} {kind}")


# -------------------------------------------------------------- Muon step --

def muon_case(shape, rng, *, weight_decay=0.0, nesterov=True, ns_steps=5, lr=0.02, mu=0.95, model=True,
              steps=1):
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    Wd, md = dev(W), dev(m)
    Wb = torch.zeros(shape, dtype=torch.bfloat16, device="cuda") if model else None
    hp = mp.muon_hp(lr=lr, momentum=mu, weight_decay=weight_decay, nesterov=nesterov, ns_steps=ns_steps)
    for _ in range(steps):
        g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
        W0, m0 = host(Wd).copy(), host(md).copy()
        gd = dev(g)
        p = mp.Param(Wd, gd, md, None, Wb)
        ws = mp.alloc_workspace(mp.workspace_size([p], "muon"))
        mp.muon_step(p, hp, ws)
        assert mp.device_status(ws) == mp.OPT_OK
        W1, m1 = host(Wd), host(md)
        Wn, mn, O = OM.muon_step(W0, g, m0, lr=lr, momentum=mu, weight_decay=weight_decay,
                                 nesterov=nesterov, ns_steps=ns_steps)
        upd_gpu = W0.astype(np.float64) * (1 - lr * weight_decay) - W1
        upd_want = W0.astype(np.float64) * (1 - lr * weight_decay) - Wn
        assert rel(upd_gpu, upd_want) < NS_TOL
        assert np.allclose(m1, mn, rtol=1e-5, atol=1e-9)
        if model:
            assert np.array_equal(bf16_host(Wb), OA.bf16_rne(W1))
    return upd_gpu, upd_want, lr * OM.update_scale(*shape)


@pytest.mark.parametrize("shape", [(256, 512), (512, 256), (300, 200), (96, 96), (512, 512), (1, 40), (40, 1)])
def test_muon_step_shapes(shape):
    upd, want, s = muon_case(shape, np.random.default_rng(shape[0] * 7 + shape[1]), steps=2)
    if 1 < shape[0] != shape[1] > 1:
        sv = singular_values(upd / s)
        assert 0.6 <= sv.min() and sv.max() <= 1.3
    elif shape[0] == shape[1] > 1:
        assert_square_spectrum(upd / s, want / s, f"update {shape}")


@pytest.mark.parametrize("kw", [dict(weight_decay=0.1), dict(nesterov=False), dict(ns_steps=1),
                                dict(ns_steps=0), dict(ns_steps=8), dict(model=False), dict(mu=0.0)])
def test_muon_step_options(kw):
    muon_case((200, 328), np.random.default_rng(11), **kw)


@pytest.mark.parametrize("case", ["aligned_wide", "aligned_tall", "unaligned_wide", "unaligned_tall",
                                  "bf16_pitch_8_bytes_off", "pitch_100_floats_no_model"])
def test_muon_update_memory_layouts(case):
    """The last Newton-Schulz GEMM updates W and its bf16 copy through TMA when
    the bases are 16-byte aligned and the row pitches multiples of 16 bytes,
    and through plain loads and stores otherwise (a view one element into its
    buffer; 100 columns, whose bf16 rows are 200 bytes apart).  Both give the
    oracle's update and a bf16 copy equal to the rounding of the new master."""
    shape = {"aligned_wide": (96, 160), "aligned_tall": (160, 96), "unaligned_wide": (96, 160),
             "unaligned_tall": (160, 96), "bf16_pitch_8_bytes_off": (64, 100),
             "pitch_100_floats_no_model": (64, 100)}[case]
    model = case != "pitch_100_floats_no_model"
    rng = np.random.default_rng(23)
    R, C = shape
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    if case.startswith("unaligned"):
        Wd = torch.zeros(R * C + 1, dtype=torch.float32, device="cuda")[1:].view(R, C)
        Wd.copy_(torch.from_numpy(W).cuda())
        Wb = torch.zeros(R * C + 1, dtype=torch.bfloat16, device="cuda")[1:].view(R, C)
    else:
        Wd = dev(W)
        Wb = torch.zeros(shape, dtype=torch.bfloat16, device="cuda") if model else None
    md, gd = dev(m), dev(g)
    lr, mu = 0.02, 0.95
    hp = mp.muon_hp(lr=lr, momentum=mu)
    p = mp.Param(Wd, gd, md, None, Wb)
    ws = mp.alloc_workspace(mp.workspace_size([p], "muon"))
    mp.muon_step(p, hp, ws)
    assert mp.device_status(ws) == mp.OPT_OK
    W1 = host(Wd)
    Wn, mn, _ = OM.muon_step(W, g, m, lr=lr, momentum=mu, weight_decay=0.0, nesterov=True, ns_steps=5)
    assert rel(W.astype(np.float64) - W1, W.astype(np.float64) - Wn) < NS_TOL
    assert np.allclose(host(md), mn, rtol=1e-5, atol=1e-9)
    if Wb is not None:
        assert np.array_equal(bf16_host(Wb), OA.bf16_rne(W1))


@pytest.mark.parametrize("scale", [1e-6, 1e-3, 1e3])
def test_newton_schulz_scale_invariance(scale):
    """The normalisation makes the iteration independent of the gradient's
    scale; the fp16 operands are formed after it, so tiny and large
    gradients keep the same accuracy."""
    rng = np.random.default_rng(31)
    G = (rng.standard_normal((384, 1000)) * scale).astype(np.float32)
    want = OM.newton_schulz(G.astype(np.float64))
    assert rel(ns_gpu(G), want) < NS_TOL


@pytest.mark.parametrize("case", ["outlier", "sparse_tiny", "outlier_tall", "zeros"])
def test_newton_schulz_iterate_outside_fp16_range(case):
    """The one-pass prologue writes fp16(gtilde * x_scale) with x_scale a power
    of two set from a strided sample of |gtilde|.  An element far beyond the
    sampled maximum (here 2000 times it, at a position the sample skips)
    would overflow fp16, and a gradient whose sampled elements are all zero
    and whose others are tiny would lose fp16 precision: such matrices take
    the fix-up, which rewrites X0 normalised from g and m.  Either way the
    output is the oracle's; an all-zero gradient gives zeros."""
    rng = np.random.default_rng(41)
    shape = (1000, 384) if case == "outlier_tall" else (384, 1000)
    if case in ("outlier", "outlier_tall"):
        G = rng.standard_normal(shape).astype(np.float32)
        G.reshape(-1)[1] = 1e4            # index 1: the sample's stride is n // 4096 = 93
    elif case == "sparse_tiny":
        G = np.zeros(shape, np.float32)
        idx = rng.choice(G.size, 500, replace=False)
        idx = idx[idx % 93 != 0]            # none at a sampled position
        G.reshape(-1)[idx] = (rng.standard_normal(idx.size) * 1e-3).astype(np.float32)
    else:
        G = np.zeros(shape, np.float32)
    got = ns_gpu(G)
    if case == "zeros":
        assert np.array_equal(got, np.zeros(shape))
        return
    want = OM.newton_schulz(G.astype(np.float64))
    assert rel(got, want) < NS_TOL


def test_muon_step_fixup_keeps_momentum_single_update():
    """A Muon step whose gradient takes the fix-up: the momentum buffer is
    updated exactly once (the fix-up reads the new m, it does not update it
    again) and the update matches the oracle."""
    rng = np.random.default_rng(43)
    shape = (256, 640)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g.reshape(-1)[5] = 1e3                  # 1e5 times the gradient's scale, off the sample
    Wd, md = dev(W), dev(m)
    p = mp.Param(Wd, dev(g), md, None, None)
    mp.muon_step(p, mp.muon_hp(), mp.alloc_workspace(mp.workspace_size([p], "muon")))
    Wn, mn, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)
    assert np.allclose(host(md), mn, rtol=1e-5, atol=1e-9)
    assert rel(W.astype(np.float64) - host(Wd), W.astype(np.float64) - Wn) < NS_TOL


def test_non_finite_gradient_propagates():
    """A NaN in the gradient is not skipped ("02 · Optimizer：算法与 infra"
    §10: bf16 training has no loss scaler): its momentum element becomes NaN,
    the Frobenius norm is NaN, and so is every element of the update, as in
    the oracle; the other momentum elements are unaffected and the call ends
    normally."""
    rng = np.random.default_rng(47)
    shape = (192, 320)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    m = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    g[3, 5] = np.nan
    Wd, md = dev(W), dev(m)
    p = mp.Param(Wd, dev(g), md, None, None)
    ws = mp.alloc_workspace(mp.workspace_size([p], "muon"))
    mp.muon_step(p, mp.muon_hp(), ws)
    assert mp.device_status(ws) == mp.OPT_OK
    Wn, mn, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)
    assert np.isnan(Wn).all() and np.isnan(host(Wd)).all()
    m1 = host(md)
    assert np.isnan(m1[3, 5]) and np.isnan(mn[3, 5])
    ok = ~np.isnan(mn)
    assert np.isnan(m1).sum() == 1 and np.allclose(m1[ok], mn[ok], rtol=1e-5, atol=1e-9)


def test_newton_schulz_many_steps():
    rng = np.random.default_rng(32)
    G = rng.standard_normal((256, 512)).astype(np.float32)
    for steps in (8, 16):
        assert rel(ns_gpu(G, steps), OM.newton_schulz(G.astype(np.float64), steps)) < NS_TOL


def test_tiny_mixed_workload_10_steps():
    """The tiny mixed workload through opt_mixed_step: one 256x512 Muon
    matrix and one 512-vector under AdamW, 10 steps.  Each step is checked
    from the state the GPU started it with (AdamW bit-exact; Muon within
    the Newton-Schulz tolerance)."""
    w = S.tiny_mixed()
    specs = w.tensors
    Wm, vec = specs
    dW = dev(S.init_value(Wm, 0))
    dv = dev(S.init_value(vec, 1))
    mW = torch.zeros_like(dW)
    mv = torch.zeros_like(dv)
    vv = torch.zeros_like(dv)
    bW = torch.zeros(Wm.shape, dtype=torch.bfloat16, device="cuda")
    bv = torch.zeros(vec.shape, dtype=torch.bfloat16, device="cuda")
    gW = torch.zeros_like(dW)
    gv = torch.zeros_like(dv)
    params = [mp.Param(dW, gW, mW, None, bW), mp.Param(dv, gv, mv, vv, bv)]
    ws = mp.alloc_workspace(mp.workspace_size(params))
    hm = mp.muon_hp(lr=w.muon.lr, momentum=w.muon.momentum, weight_decay=w.muon.weight_decay,
                    nesterov=w.muon.nesterov, ns_steps=w.muon.ns_steps)
    ah = dict(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
              weight_decay=w.adamw.weight_decay)
    for t in range(1, w.steps + 1):
        g0, g1 = S.grad_value(Wm, 0, t), S.grad_value(vec, 1, t)
        gW.copy_(dev(g0))
        gv.copy_(dev(g1))
        W0, m0 = host(dW).copy(), host(mW).copy()
        hv = [host(x).copy() for x in (dv, mv, vv)]
        mp.mixed_step(params, hm, mp.adamw_hp(step=t, **ah), ws)
        assert mp.device_status(ws) == mp.OPT_OK
        # AdamW vector: bit-exact
        OA.adamw_step_fp32(hv[0], g1, hv[1], hv[2], t=t, **ah)
        for got, want in zip((dv, mv, vv), hv):
            assert np.array_equal(host(got).view(np.uint32), want.view(np.uint32))
        assert np.array_equal(bf16_host(bv), OA.bf16_rne(hv[0]))
        # Muon matrix
        Wn, mn, _ = OM.muon_step(W0, g0, m0, lr=w.muon.lr, momentum=w.muon.momentum,
                                 weight_decay=w.muon.weight_decay)
        assert rel(W0 - host(dW).astype(np.float64), W0 - Wn) < NS_TOL
        assert np.allclose(host(mW), mn, rtol=1e-5, atol=1e-9)
        assert np.array_equal(bf16_host(bW), OA.bf16_rne(host(dW)))
        sv = np.linalg.svd((W0 - host(dW).astype(np.float64)) / (w.muon.lr * OM.update_scale(256, 512)),
                           compute_uv=False)
        assert 0.6 <= sv.min() and sv.max() <= 1.3


def test_muon_skewed_workload_50_steps():
    """Both 4096x1024 / 1024x4096 matrices under Muon for all 50 steps with
    the rank-8 skewed gradient; steps 1, 2, 25 and 50 are checked from the
    state the GPU started them with."""
    w = S.muon_8m_skewed()
    Ws = [dev(S.init_value(sp, i)) for i, sp in enumerate(w.tensors)]
    ms = [torch.zeros_like(x) for x in Ws]
    gs = [torch.zeros_like(x) for x in Ws]
    bs = [torch.zeros(sp.shape, dtype=torch.bfloat16, device="cuda") for sp in w.tensors]
    params = [mp.Param(W, g, m, None, b) for W, g, m, b in zip(Ws, gs, ms, bs)]
    ws = mp.alloc_workspace(mp.workspace_size(params))
    hm = mp.muon_hp(lr=w.muon.lr, momentum=w.muon.momentum, nesterov=True, ns_steps=5)
    for t in range(1, w.steps + 1):
        gh = [S.grad_value(sp, i, t) for i, sp in enumerate(w.tensors)]
        for gd, g in zip(gs, gh):
            gd.copy_(dev(g))
        checked = t in (1, 2, 25, w.steps)
        if checked:
            W0 = [host(x).copy() for x in Ws]
            m0 = [host(x).copy() for x in ms]
        mp.mixed_step(params, hm, None, ws)
        if checked:
            assert mp.device_status(ws) == mp.OPT_OK
            for i, sp in enumerate(w.tensors):
                Wn, mn, _ = OM.muon_step(W0[i], gh[i], m0[i], lr=w.muon.lr, momentum=w.muon.momentum)
                upd = W0[i] - host(Ws[i]).astype(np.float64)
                assert rel(upd, W0[i] - Wn) < NS_TOL, (t, i)
                assert np.allclose(host(ms[i]), mn, rtol=1e-5, atol=1e-9)
                sv = np.linalg.svd(upd / (w.muon.lr * OM.update_scale(*sp.shape)), compute_uv=False)
                assert 0.6 <= sv.min() and sv.max() <= 1.3, (t, i, sv.min(), sv.max())
                assert np.array_equal(bf16_host(bs[i]), OA.bf16_rne(host(Ws[i])))


def test_group_splitting_with_small_workspace():
    """Several same-shape matrices in both orientations: with the full
    workspace they share batched launches; with the minimum workspace they
    run one at a time.  Both give the oracle's result."""
    rng = np.random.default_rng(21)
    shapes = [(192, 320), (320, 192), (192, 320), (320, 192), (192, 320)]
    Ws0 = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    gs = [(rng.standard_normal(s) * 1e-2).astype(np.float32) for s in shapes]
    hm = mp.muon_hp()
    results = []
    for small in (False, True):
        Ws = [dev(W) for W in Ws0]
        ms = [torch.zeros_like(x) for x in Ws]
        params = [mp.Param(W, dev(g), m, None, None) for W, g, m in zip(Ws, gs, ms)]
        need = mp.workspace_size(params)
        one = mp.workspace_size(params[:1])
        ws = mp.alloc_workspace(one if small else need)
        assert one < need
        mp.mixed_step(params, hm, None, ws)
        assert mp.device_status(ws) == mp.OPT_OK
        results.append([host(W) for W in Ws])
        for i in range(len(shapes)):
            Wn, _, _ = OM.muon_step(Ws0[i], gs[i], np.zeros(shapes[i]), lr=0.02, momentum=0.95)
            assert rel(Ws0[i] - results[-1][i].astype(np.float64), Ws0[i] - Wn) < NS_TOL
    for a, b in zip(*results):       # grouping does not change the arithmetic
        assert np.array_equal(a, b)


def test_mixed_routing():
    """2-D non-embedding -> Muon; 1-D and flagged embedding/output -> AdamW."""
    rng = np.random.default_rng(8)
    W = (rng.standard_normal((64, 96)) * 0.02).astype(np.float32)
    E = (rng.standard_normal((50, 64)) * 0.02).astype(np.float32)
    g_w = (rng.standard_normal(W.shape) * 1e-2).astype(np.float32)
    g_e = (rng.standard_normal(E.shape) * 1e-2).astype(np.float32)
    dW, dE = dev(W), dev(E)
    mW, mE, vE = torch.zeros_like(dW), torch.zeros_like(dE), torch.zeros_like(dE)
    params = [mp.Param(dW, dev(g_w), mW, None, None),
              mp.Param(dE, dev(g_e), mE, vE, None, embedding_or_output=True)]
    ws = mp.alloc_workspace(mp.workspace_size(params))
    ah = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    mp.mixed_step(params, mp.muon_hp(), mp.adamw_hp(step=1, **ah), ws)
    Ep, Em, Ev = E.copy(), np.zeros_like(E), np.zeros_like(E)
    OA.adamw_step_fp32(Ep, g_e, Em, Ev, t=1, **ah)
    assert np.array_equal(host(dE).view(np.uint32), Ep.view(np.uint32))
    Wn, _, _ = OM.muon_step(W, g_w, np.zeros_like(W), lr=0.02, momentum=0.95)
    assert rel(W - host(dW).astype(np.float64), W - Wn) < NS_TOL


def test_repeatable():
    """Two runs from the same state give identical bits (fixed reduction
    order, no atomics on the data path)."""
    rng = np.random.default_rng(2)
    W = (rng.standard_normal((384, 640)) * 0.02).astype(np.float32)
    g = (rng.standard_normal(W.shape) * 1e-2).astype(np.float32)
    outs = []
    for _ in range(2):
        dW, m = dev(W), torch.zeros(W.shape, device="cuda")
        p = mp.Param(dW, dev(g), m, None, None)
        mp.muon_step(p, mp.muon_hp(), mp.alloc_workspace(mp.workspace_size([p], "muon")))
        outs.append(host(dW))
    assert np.array_equal(outs[0], outs[1])
