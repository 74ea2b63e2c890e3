"""Seeded random Muon and mixed steps against the oracle: shapes from 1 to 700
on each side (ragged against the 256-element padding, tall and wide, square,
1-wide), every evaluation order of the iterations, 0 to 8 iterations,
Nesterov on and off, weight decay, several matrices of one shape class in one
call (batched, both orientations), and AdamW tensors beside them.  The bar is
the one of every Muon and AdamW test: the Muon update within 2e-2 relative
Frobenius error of the fp64 oracle, momentum within 1e-5 per element, AdamW
bit-exact against the fp32 oracle, bf16 copies bit-exact against the GPU's
own masters."""

import numpy as np
import pytest

from gpu_helpers import bf16_host, dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
from oracle import muon as OM

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2
ORDERS = ("auto", "per_iteration", "grouped")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rel(a, b):
    n = np.linalg.norm(b)
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / n) if n > 0 else float(np.linalg.norm(a))


def random_case(rng):
    def side():
        return int(rng.choice([1, 2, 7, 64, 96, 127, 256, 257, 300, 511, 512, 700]))
    R, C = side(), side()
    if rng.random() < 0.2:
        C = R                                           # square
    return dict(shape=(R, C), copies=int(rng.integers(1, 4)), order=str(rng.choice(ORDERS)),
                ns_steps=int(rng.choice([0, 1, 2, 3, 4, 5, 5, 5, 7, 8])), nesterov=bool(rng.random() < 0.8),
                wd=float(rng.choice([0.0, 0.1])), adamw=int(rng.integers(0, 3)))


@pytest.mark.parametrize("seed", range(24))
def test_random_mixed_step(seed):
    rng = np.random.default_rng(7000 + seed)
    c = random_case(rng)
    R, C = c["shape"]
    lr, mu = 0.02, 0.95
    # matrices of one class in both orientations; AdamW vectors beside them
    shapes = [(R, C) if k % 2 == 0 else (C, R) for k in range(c["copies"])]
    Ws = [(rng.standard_normal(s) * 0.02).astype(np.float32) for s in shapes]
    ms = [(rng.standard_normal(s) * 1e-2).astype(np.float32) for s in shapes]
    gs = [(rng.standard_normal(s) * 1e-2).astype(np.float32) for s in shapes]
    n_vec = [int(rng.integers(1, 5000)) for _ in range(c["adamw"])]
    vp = [rng.standard_normal(n).astype(np.float32) for n in n_vec]
    vg = [(rng.standard_normal(n) * 1e-3).astype(np.float32) for n in n_vec]
    params = []
    for W, m, g, s in zip(Ws, ms, gs, shapes):
        params.append(mp.Param(dev(W), dev(g), dev(m), None, torch.zeros(s, dtype=torch.bfloat16, device="cuda")))
    for p0, g0 in zip(vp, vg):
        params.append(mp.Param(dev(p0), dev(g0), torch.zeros(p0.shape, device="cuda"),
                               torch.zeros(p0.shape, device="cuda"),
                               torch.zeros(p0.shape, dtype=torch.bfloat16, device="cuda")))
    hm = mp.muon_hp(lr=lr, momentum=mu, weight_decay=c["wd"], nesterov=c["nesterov"], ns_steps=c["ns_steps"],
                    ns_order=c["order"])
    ah = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01)
    ws = mp.alloc_workspace(mp.workspace_size(params, ns_order=c["order"]))
    mp.mixed_step(params, hm, mp.adamw_hp(step=1, **ah), ws)
    torch.cuda.synchronize()
    assert mp.device_status(ws) == mp.OPT_OK
    for k, (W, m, g) in enumerate(zip(Ws, ms, gs)):
        Wn, mn, _ = OM.muon_step(W, g, m, lr=lr, momentum=mu, weight_decay=c["wd"], nesterov=c["nesterov"],
                                 ns_steps=c["ns_steps"])
        W1 = host(params[k].main_param)
        decay = 1 - lr * c["wd"]
        assert rel(W.astype(np.float64) * decay - W1, W.astype(np.float64) * decay - Wn) < NS_TOL, (c, k)
        assert np.allclose(host(params[k].exp_avg), mn, rtol=1e-5, atol=1e-9), (c, k)
        assert np.array_equal(bf16_host(params[k].model), OA.bf16_rne(W1)), (c, k)
    for j, (p0, g0) in enumerate(zip(vp, vg)):
        prm = params[len(Ws) + j]
        p, m, v = p0.copy(), np.zeros_like(p0), np.zeros_like(p0)
        OA.adamw_step_fp32(p, g0, m, v, t=1, **ah)
        assert np.array_equal(host(prm.main_param).view(np.uint32), p.view(np.uint32)), (c, j)
        assert np.array_equal(bf16_host(prm.model), OA.bf16_rne(p))
