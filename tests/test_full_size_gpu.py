"""Parity at full size, in the launch configuration bench.py times, on
sampled outputs the oracle can compute one by one.

* llama16_mixed (4.54e9 parameters, one opt_mixed_step over all 147 tensors):
  two steps; AdamW checked bit-exact on sampled elements of the embedding, the
  LM head and norm vectors; Muon checked against the fp64 oracle on one matrix
  of each shape class (4096 x 4096, 1024 x 4096, 14336 x 4096 -- transposed --
  and 4096 x 14336): the update within 2e-2 relative Frobenius error, the
  direction's singular values in [0.6, 1.3] on the rectangular classes and,
  on the square class, within 0.05 of the oracle's sorted singular values
  with none above 1.3.
* adamw_sweep_10k (10,000 tensors, ~1.0e10 parameters, log-uniform sizes in
  [1, 2^24)): all 20 steps; bit-exact on sampled elements of every size
  decade.

Inputs are drawn on the GPU with the seeded generators of synthetic/; the
sampled inputs are copied back before each step, so every expected value comes
from the oracle.  Gradients and bf16 model copies are views of flat buffers, as
in the bench."""

import math

import numpy as np
import pytest

from gpu_helpers import assert_square_spectrum, bf16_host, host, require_gpu, singular_values, torch
import bench
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
from oracle import muon as OM
import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.fixture(autouse=True)
def _release_memory():
    yield
    import gc
    gc.collect()
    torch.cuda.empty_cache()


def free_gb():
    free, _ = torch.cuda.mem_get_info()
    return free / 1e9


def build(w, muon_route):
    """The workload in the layout bench.py times: every main_grad a view of one
    flat fp32 buffer and every bf16 model copy a view of one flat bf16 buffer."""
    shapes = [spec.shape for spec in w.tensors]
    offs, n_flat = bench.flat_layout(spec.numel for spec in w.tensors)
    grads = bench.flat_views(torch.empty(n_flat, dtype=torch.float32, device="cuda"), offs, shapes)
    models = bench.flat_views(torch.empty(n_flat, dtype=torch.bfloat16, device="cuda"), offs, shapes)
    params, specs = [], []
    for i, spec in enumerate(w.tensors):
        p = torch.empty(spec.shape, dtype=torch.float32, device="cuda")
        S.torch_init_(p, spec, i)
        m = torch.zeros_like(p)
        v = None if muon_route(spec) else torch.zeros_like(p)
        models[i].copy_(p)
        params.append(mp.Param(p, grads[i], m, v, models[i], embedding_or_output=spec.embedding_or_output,
                               kind="adamw" if w.force_adamw else None))
        specs.append(spec)
    return params, specs


def take(t, idx):
    return host(t.reshape(-1)[idx])


def test_llama16_mixed_full_size_sampled():
    w = S.llama16_mixed()
    if free_gb() < 110:
        pytest.skip("needs ~105 GB of free device memory")
    route = lambda sp: len(sp.shape) == 2 and not sp.embedding_or_output
    params, specs = build(w, route)
    ws = mp.alloc_workspace(mp.workspace_size(params))
    hm = mp.muon_hp(lr=w.muon.lr, momentum=w.muon.momentum, weight_decay=w.muon.weight_decay)
    ah = dict(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
              weight_decay=w.adamw.weight_decay)
    rng = np.random.default_rng(0)
    adamw_ids = [i for i, sp in enumerate(specs) if not route(sp)]
    samples = {i: rng.choice(specs[i].numel, size=min(specs[i].numel, 20000), replace=False) for i in adamw_ids}
    muon_check = {}
    for i, sp in enumerate(specs):
        if route(sp) and sp.shape not in muon_check:
            muon_check[sp.shape] = i
    for t in (1, 2):
        for i, (prm, sp) in enumerate(zip(params, specs)):
            S.torch_grad_(prm.main_grad, sp, i, t)
        before = {i: [take(getattr(params[i], k), samples[i]) for k in ("main_param", "main_grad", "exp_avg",
                                                                          "exp_avg_sq")] for i in adamw_ids}
        mbefore = {i: (host(params[i].main_param), host(params[i].main_grad), host(params[i].exp_avg))
                   for i in muon_check.values()} if t == 2 else {}
        mp.mixed_step(params, hm, mp.adamw_hp(step=t, **ah), ws)
        assert mp.device_status(ws) == mp.OPT_OK
        torch.cuda.synchronize()
        for i in adamw_ids:
            p, g, m, v = before[i]
            OA.adamw_step_fp32(p, g, m, v, t=t, **ah)
            idx = samples[i]
            assert np.array_equal(take(params[i].main_param, idx).view(np.uint32), p.view(np.uint32)), specs[i].name
            assert np.array_equal(take(params[i].exp_avg_sq, idx).view(np.uint32), v.view(np.uint32))
            assert np.array_equal(bf16_host(params[i].model.reshape(-1)[idx]), OA.bf16_rne(p))
        for shape, i in muon_check.items():
            if t != 2:
                continue
            W0, g0, m0 = mbefore[i]
            Wn, mn, _ = OM.muon_step(W0, g0, m0, lr=w.muon.lr, momentum=w.muon.momentum)
            W1 = host(params[i].main_param).astype(np.float64)
            rel = np.linalg.norm((W0 - W1) - (W0 - Wn)) / np.linalg.norm(W0 - Wn)
            assert rel < 2e-2, (shape, rel)
            # the update's direction O: singular values in [0.6, 1.3] on the
            # rectangular classes; on the square q/o class the spectrum of the
            # fp64 oracle's O (sorted values within 0.05, none above 1.3)
            s = w.muon.lr * OM.update_scale(*shape)
            O_gpu, O_want = (W0 - W1) / s, (W0 - Wn) / s
            if shape[0] == shape[1]:
                assert_square_spectrum(O_gpu, O_want, f"{shape}")
            else:
                sv = singular_values(O_gpu)
                assert 0.6 <= sv.min() and sv.max() <= 1.3, (shape, sv.min(), sv.max())
            assert np.allclose(host(params[i].exp_avg), mn, rtol=1e-5, atol=1e-10)
            b = bf16_host(params[i].model)
            assert np.array_equal(b, OA.bf16_rne(host(params[i].main_param))), shape


def test_adamw_sweep_10k_full_size_sampled():
    w = S.adamw_sweep_10k()
    need = w.numel * 18 / 1e9 + 5
    if free_gb() < need:
        pytest.skip(f"needs ~{need:.0f} GB of free device memory")
    params, specs = build(w, lambda sp: False)
    ah = dict(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
              weight_decay=w.adamw.weight_decay)
    rng = np.random.default_rng(1)
    # per size decade: up to 40 tensors, up to 2000 elements each
    decade = [int(math.log10(sp.numel)) for sp in specs]
    chosen = []
    for d in sorted(set(decade)):
        ids = [i for i, x in enumerate(decade) if x == d]
        chosen += list(rng.choice(ids, size=min(len(ids), 40), replace=False))
    samples = {i: rng.choice(specs[i].numel, size=min(specs[i].numel, 2000), replace=False) for i in chosen}
    state = {i: [take(params[i].main_param, samples[i]), None, np.zeros(len(samples[i]), np.float32),
                 np.zeros(len(samples[i]), np.float32)] for i in chosen}
    for t in range(1, w.steps + 1):
        for i, (prm, sp) in enumerate(zip(params, specs)):
            S.torch_grad_(prm.main_grad, sp, i, t)
        for i in chosen:
            state[i][1] = take(params[i].main_grad, samples[i])
        mp.adamw_step(params, mp.adamw_hp(step=t, **ah))
        for i in chosen:
            p, g, m, v = state[i]
            OA.adamw_step_fp32(p, g, m, v, t=t, **ah)
    torch.cuda.synchronize()
    for i in chosen:
        p, _, m, v = state[i]
        idx = samples[i]
        assert np.array_equal(take(params[i].main_param, idx).view(np.uint32), p.view(np.uint32)), specs[i].numel
        assert np.array_equal(take(params[i].exp_avg, idx).view(np.uint32), m.view(np.uint32))
        assert np.array_equal(take(params[i].exp_avg_sq, idx).view(np.uint32), v.view(np.uint32))
        assert np.array_equal(bf16_host(params[i].model.reshape(-1)[idx]), OA.bf16_rne(p))
