"""Global grad-norm clipping fused into the step (opt_mixed_step_clipped),
against the oracle of "02 · Optimizer：算法与 infra" §11.1 / §11.4.

Bars: the total norm within 1e-6 relative of the fp64 oracle (fp32 partial
sums per 16K-element chunk); the factor applied equal to the oracle's formula
evaluated on the GPU's norm; AdamW bit-exact against the fp32 oracle fed the
gradient times the GPU's factor; Muon within the Newton-Schulz tolerance."""

import numpy as np
import pytest

from gpu_helpers import bf16_host, dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
from oracle import clip as OC
from oracle import muon as OM

pytestmark = pytest.mark.gpu

AH = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _problem(rng, n_vec=5, vec_sizes=(1, 17, 16384, 40001, 3), muon_shapes=((96, 160), (160, 96)), offset=1):
    """AdamW vectors (one of them an unaligned view) and Muon matrices."""
    vecs, mats = [], []
    for i, n in enumerate(vec_sizes[:n_vec]):
        base = rng.standard_normal(n + offset).astype(np.float32)
        g = (rng.standard_normal(n + offset) * 1e-2).astype(np.float32)
        o = offset if i == 2 else 0
        vecs.append(dict(p=base[o:o + n].copy(), g=g[o:o + n].copy(), gbuf=g, off=o,
                         m=np.zeros(n, np.float32), v=np.zeros(n, np.float32)))
    for shp in muon_shapes:
        mats.append(dict(W=(rng.standard_normal(shp) * 0.02).astype(np.float32),
                         g=(rng.standard_normal(shp) * 1e-2).astype(np.float32),
                         m=np.zeros(shp, np.float32)))
    return vecs, mats


def _device(vecs, mats):
    params, dvec, dmat = [], [], []
    for d in vecs:
        gfull = dev(d["gbuf"])
        t = dict(p=dev(d["p"]), g=gfull[d["off"]:d["off"] + d["p"].size], m=dev(d["m"]), v=dev(d["v"]),
                 b=torch.zeros(d["p"].size, dtype=torch.bfloat16, device="cuda"), keep=gfull)
        dvec.append(t)
        params.append(mp.Param(t["p"], t["g"], t["m"], t["v"], t["b"]))
    for d in mats:
        t = dict(W=dev(d["W"]), g=dev(d["g"]), m=dev(d["m"]))
        dmat.append(t)
        params.append(mp.Param(t["W"], t["g"], t["m"], None, None))
    return params, dvec, dmat


@pytest.mark.parametrize("max_norm", [0.05, 1e6])
def test_clipped_step_against_oracle(max_norm):
    rng = np.random.default_rng(4)
    vecs, mats = _problem(rng)
    params, dvec, dmat = _device(vecs, mats)
    ws = mp.alloc_workspace(mp.workspace_size(params, clip=True))
    norm = torch.zeros(1, device="cuda")
    scale = torch.zeros(1, device="cuda")
    mp.mixed_step_clipped(params, mp.muon_hp(), mp.adamw_hp(step=1, **AH), max_norm, ws, norm, scale)
    assert mp.device_status(ws) == mp.OPT_OK
    grads = [d["g"] for d in vecs] + [d["g"] for d in mats]
    want_norm = OC.total_norm(grads)
    got_norm = float(host(norm)[0])
    assert abs(got_norm - want_norm) <= 1e-6 * want_norm
    got_scale = np.float32(host(scale)[0])
    want_scale = OC.clip_scale(grads, max_norm)
    if max_norm > want_norm:
        assert got_scale == 1.0
    else:
        # the factor is the formula on the GPU's own norm, rounded once to fp32
        assert got_scale == np.float32(max_norm / (np.float64(got_norm) + 1e-6)) or \
            abs(got_scale - want_scale) <= 2e-6 * want_scale
    # AdamW: bit-exact against the fp32 oracle fed g * (the GPU's factor)
    for d, t in zip(vecs, dvec):
        g = (d["g"] * got_scale).astype(np.float32)
        OA.adamw_step_fp32(d["p"], g, d["m"], d["v"], t=1, **AH)
        assert np.array_equal(host(t["p"]).view(np.uint32), d["p"].view(np.uint32))
        assert np.array_equal(host(t["m"]).view(np.uint32), d["m"].view(np.uint32))
        assert np.array_equal(bf16_host(t["b"]), OA.bf16_rne(d["p"]))
    # Muon: the clipped gradient enters the momentum
    for d, t in zip(mats, dmat):
        gc = d["g"].astype(np.float64) * float(got_scale)
        Wn, mn, _ = OM.muon_step(d["W"], gc, d["m"], lr=0.02, momentum=0.95)
        upd = d["W"].astype(np.float64) - host(t["W"]).astype(np.float64)
        assert np.linalg.norm(upd - (d["W"] - Wn)) / np.linalg.norm(d["W"] - Wn) < 2e-2
        assert np.allclose(host(t["m"]), mn, rtol=1e-5, atol=1e-10)


def test_clipped_step_with_iterate_fixup():
    """Clipping active and a Muon gradient whose iterate takes the fix-up (one
    element 1e4 times the rest, where the scale sample does not look): the
    clipping factor enters the sample, the one-pass prologue and the fix-up
    alike, so the update is the oracle's for g * factor."""
    rng = np.random.default_rng(8)
    vecs, mats = _problem(rng, n_vec=2, muon_shapes=((256, 640), (640, 256)))
    for d in mats:
        d["g"].reshape(-1)[7] = 1e2
    params, dvec, dmat = _device(vecs, mats)
    ws = mp.alloc_workspace(mp.workspace_size(params, clip=True))
    scale = torch.zeros(1, device="cuda")
    mp.mixed_step_clipped(params, mp.muon_hp(), mp.adamw_hp(step=1, **AH), 1.0, ws, None, scale)
    assert mp.device_status(ws) == mp.OPT_OK
    got_scale = float(host(scale)[0])
    assert got_scale < 0.01
    for d, t in zip(mats, dmat):
        gc = d["g"].astype(np.float64) * got_scale
        Wn, mn, _ = OM.muon_step(d["W"], gc, d["m"], lr=0.02, momentum=0.95)
        upd = d["W"].astype(np.float64) - host(t["W"]).astype(np.float64)
        assert np.linalg.norm(upd - (d["W"] - Wn)) / np.linalg.norm(d["W"] - Wn) < 2e-2
        assert np.allclose(host(t["m"]), mn, rtol=1e-5, atol=1e-10)


def test_disabled_clip_equals_unclipped_step():
    rng = np.random.default_rng(5)
    outs = []
    for clipped in (False, True):
        vecs, mats = _problem(np.random.default_rng(5))
        params, dvec, dmat = _device(vecs, mats)
        ws = mp.alloc_workspace(mp.workspace_size(params, clip=clipped))
        if clipped:
            mp.mixed_step_clipped(params, mp.muon_hp(), mp.adamw_hp(step=2, **AH), 0.0, ws)
        else:
            mp.mixed_step(params, mp.muon_hp(), mp.adamw_hp(step=2, **AH), ws)
        outs.append([host(t["p"]) for t in dvec] + [host(t["W"]) for t in dmat])
    for a, b in zip(*outs):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_norm_over_many_tensors():
    """More tensors than one norm launch takes (1200): the partial sums of
    several launches meet in one reduction."""
    rng = np.random.default_rng(6)
    sizes = rng.integers(1, 5000, 2500)
    gs = [(rng.standard_normal(int(n)) * 1e-3).astype(np.float32) for n in sizes]
    params = []
    keep = []
    for g in gs:
        gd = dev(g)
        p = torch.zeros_like(gd)
        m = torch.zeros_like(gd)
        v = torch.zeros_like(gd)
        keep += [gd, p, m, v]
        params.append(mp.Param(p, gd, m, v, None))
    ws = mp.alloc_workspace(mp.workspace_size(params, clip=True))
    norm = torch.zeros(1, device="cuda")
    mp.mixed_step_clipped(params, None, mp.adamw_hp(step=1, **AH), 1e-3, ws, norm)
    want = OC.total_norm(gs)
    assert abs(float(host(norm)[0]) - want) <= 1e-6 * want


def test_clip_workspace_required():
    rng = np.random.default_rng(7)
    vecs, mats = _problem(rng, muon_shapes=())
    params, _, _ = _device(vecs, mats)
    assert mp.workspace_size(params) == 0
    with pytest.raises(mp.MpoptError):
        mp.mixed_step_clipped(params, None, mp.adamw_hp(step=1, **AH), 0.5, None)
