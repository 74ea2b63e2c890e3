"""Muon variants on the GPU against the fp64 oracle ("02 · Optimizer：算法与
infra" §14.6 scale modes, §5.5/§14.4 QKV split, §5.2 coefficient schedules,
§1 plain momentum SGD).  Bars as in test_muon_gpu: the update within 2e-2
relative Frobenius error; plain momentum SGD has no Newton-Schulz, so it is
fp32 elementwise arithmetic: within 1e-6 relative."""

import numpy as np
import pytest

from gpu_helpers import dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import muon as OM

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def run(W, g, hp, split=None, m=None):
    Wd, gd = dev(W), dev(g)
    md = dev(m) if m is not None else torch.zeros_like(Wd)
    p = mp.Param(Wd, gd, md, None, None)
    params = p.split_rows(split) if split else [p]
    ws = mp.alloc_workspace(mp.workspace_size(params))
    mp.mixed_step(params, hp, None, ws)
    assert mp.device_status(ws) == mp.OPT_OK
    return host(Wd).astype(np.float64), host(md)


@pytest.mark.parametrize("mode", ["spectral", "shape_scaling", "unit_rms_norm"])
@pytest.mark.parametrize("shape", [(300, 200), (200, 300)])
def test_scale_modes(mode, shape):
    rng = np.random.default_rng(hash((mode, shape)) % 2 ** 32)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    got, _ = run(W, g, mp.muon_hp(scale_mode=mode))
    Wn, _, _ = OM.muon_step(W, g, np.zeros(shape), lr=0.02, momentum=0.95, mode=mode)
    assert rel(W - got, W - Wn) < NS_TOL


def test_qkv_split_row_blocks():
    """A [q + k + v, h] parameter passed as three row-block views: each block
    is orthogonalised on its own, and the update scale is the whole
    parameter's (160 x 64 here)."""
    rng = np.random.default_rng(40)
    split = [96, 32, 32]
    W = (rng.standard_normal((160, 64)) * 0.02).astype(np.float32)
    g = (rng.standard_normal((160, 64)) * 1e-2).astype(np.float32)
    got, _ = run(W, g, mp.muon_hp(), split=split)
    Wn, _, _ = OM.muon_step(W, g, np.zeros_like(W), lr=0.02, momentum=0.95, split_rows=split)
    assert rel(W - got, W - Wn) < NS_TOL
    whole, _, _ = OM.muon_step(W, g, np.zeros_like(W), lr=0.02, momentum=0.95)
    assert rel(W - got, W - whole) > 0.05            # really split, not whole-matrix


def test_coefficient_schedule():
    rng = np.random.default_rng(41)
    sched = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]
    W = (rng.standard_normal((256, 384)) * 0.02).astype(np.float32)
    g = (rng.standard_normal((256, 384)) * 1e-2).astype(np.float32)
    got, _ = run(W, g, mp.muon_hp(ns_steps=4, schedule=sched))
    Wn, _, _ = OM.muon_step(W, g, np.zeros_like(W), lr=0.02, momentum=0.95, ns_steps=4, coeffs=sched)
    assert rel(W - got, W - Wn) < NS_TOL


def test_plain_momentum_sgd():
    rng = np.random.default_rng(42)
    W = (rng.standard_normal((70, 90)) * 0.02).astype(np.float32)
    g = (rng.standard_normal((70, 90)) * 1e-2).astype(np.float32)
    m = (rng.standard_normal((70, 90)) * 1e-2).astype(np.float32)
    got, mnew = run(W, g, mp.muon_hp(lr=0.1, scale_coeff=1.0, orthogonalize=False, weight_decay=0.01), m=m)
    Wn, mn, _ = OM.muon_step(W, g, m, lr=0.1, momentum=0.95, weight_decay=0.01, orthogonalize=False,
                             scale_coeff=1.0)
    assert rel(got, Wn) < 1e-6
    assert np.allclose(mnew, mn, rtol=1e-5, atol=1e-10)
