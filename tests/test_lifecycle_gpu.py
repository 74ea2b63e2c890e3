"""Master-weight lifecycle ("支持FP32优化器" §2.2, §2.3, §9; "02 · Optimizer：
算法与 infra" §9.2): a checkpoint that keeps the fp32 masters and the optimizer
state resumes bit for bit; rebuilding the masters from the bf16 model
(reload_model_params, the plain-checkpoint branch) is exact as a conversion
but loses the masters' fp32 tail; fp32-native parameters are their own
master and get no writeback."""

import numpy as np
import pytest

from gpu_helpers import bf16_host, dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA

pytestmark = pytest.mark.gpu

AH = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SHAPES = [(192, 320), (320, 192), (1000,), (64,)]    # two Muon matrices, two AdamW vectors


class Model:
    """Master weights, state and bf16 copies of a small Muon + AdamW model."""

    def __init__(self, seed):
        rng = np.random.default_rng(seed)
        self.t = []
        for shp in SHAPES:
            p = dev((rng.standard_normal(shp) * 0.02).astype(np.float32))
            d = dict(p=p, g=torch.zeros_like(p), m=torch.zeros_like(p),
                     v=torch.zeros_like(p) if len(shp) == 1 else None, b=p.to(torch.bfloat16))
            self.t.append(d)
        self.params = [mp.Param(d["p"], d["g"], d["m"], d["v"], d["b"]) for d in self.t]
        self.ws = mp.alloc_workspace(mp.workspace_size(self.params))

    def step(self, t, grads):
        for d, g in zip(self.t, grads):
            d["g"].copy_(g)
        mp.mixed_step(self.params, mp.muon_hp(), mp.adamw_hp(step=t, **AH), self.ws)

    def state(self):
        return [{k: (v.clone() if v is not None else None) for k, v in d.items() if k != "g"} for d in self.t]

    def load(self, st):
        for d, s in zip(self.t, st):
            for k, v in s.items():
                if v is not None:
                    d[k].copy_(v)


def grads_for(step):
    rng = np.random.default_rng(100 + step)
    return [dev((rng.standard_normal(s) * 1e-2).astype(np.float32)) for s in SHAPES]


def test_resume_from_checkpoint_is_bit_exact():
    """§2.2: train, save masters + moments + momentum + step, restore into a
    fresh set of buffers, continue with the same next gradients: identical to
    continuous training, bit for bit."""
    cont = Model(0)
    for t in (1, 2, 3):
        cont.step(t, grads_for(t))
    saved = Model(0)
    saved.step(1, grads_for(1))
    ckpt = saved.state()
    resumed = Model(77)                # different initial values, overwritten by the checkpoint
    resumed.load(ckpt)
    for t in (2, 3):
        resumed.step(t, grads_for(t))
    torch.cuda.synchronize()
    for a, b in zip(cont.t, resumed.t):
        for k in ("p", "m", "v", "b"):
            if a[k] is not None:
                assert torch.equal(a[k].view(torch.int16) if a[k].dtype == torch.bfloat16 else a[k].view(torch.int32),
                                   b[k].view(torch.int16) if b[k].dtype == torch.bfloat16 else b[k].view(torch.int32))


def test_reload_model_params_exact_and_loses_fp32_tail():
    """§9.3 branch two: main_param rebuilt from the bf16 model.  The
    conversion is exact, so masters equal the model copy widened to fp32 --
    which differs from the trained fp32 masters (their tail is lost)."""
    m = Model(1)
    m.step(1, grads_for(1))
    trained = [host(d["p"]).copy() for d in m.t]
    mp.reload_model_params(m.params)
    torch.cuda.synchronize()
    lost = 0
    for d, tr in zip(m.t, trained):
        got = host(d["p"])
        assert np.array_equal(got.view(np.uint32), OA.bf16_to_f32(bf16_host(d["b"])).view(np.uint32))
        lost += int(np.sum(got.view(np.uint32) != tr.view(np.uint32)))
    assert lost > 0


def test_fp32_native_parameters_alias_their_master():
    """§2.3: with an fp32 model the parameter is its own main_param (no bf16
    copy is passed): the step updates it in place, and reload_model_params
    leaves it alone."""
    rng = np.random.default_rng(2)
    p = dev(rng.standard_normal(5000).astype(np.float32))
    before = host(p).copy()
    g = dev((rng.standard_normal(5000) * 1e-3).astype(np.float32))
    m, v = torch.zeros_like(p), torch.zeros_like(p)
    prm = mp.Param(p, g, m, v, None)
    mp.adamw_step([prm], mp.adamw_hp(step=1, **AH))
    mp.reload_model_params([prm])
    torch.cuda.synchronize()
    want = before.copy()
    OA.adamw_step_fp32(want, host(g), np.zeros(5000, np.float32), np.zeros(5000, np.float32), t=1, **AH)
    assert np.array_equal(host(p).view(np.uint32), want.view(np.uint32))
