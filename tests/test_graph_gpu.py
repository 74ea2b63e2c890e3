"""The step enqueues device work only: no host synchronisation and no
allocation.  So it can be captured into a CUDA graph, and replays of the
graph give the same bits as the same number of eager steps.

The hyper-parameters (and AdamW's step counter) are baked into a captured
graph, so the comparison uses the same step number on both sides."""

import numpy as np
import pytest

from gpu_helpers import bf16_host, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def make_params():
    """Two Muon matrices (one tall, one wide, different shape classes), one
    embedding under AdamW and one vector, with seeded values and gradients."""
    shapes = [((384, 640), False), ((768, 256), False), ((1000, 64), True), ((300,), False)]
    params = []
    for i, (shape, emb) in enumerate(shapes):
        spec = S.TensorSpec(f"t{i}", shape, "normal", init_std=0.02, embedding_or_output=emb)
        p = torch.empty(shape, dtype=torch.float32, device="cuda")
        S.torch_init_(p, spec, i)
        g = torch.empty_like(p)
        S.torch_grad_(g, spec, i, 1)
        muon = len(shape) == 2 and not emb
        params.append(mp.Param(p, g, torch.zeros_like(p), None if muon else torch.zeros_like(p),
                               p.to(torch.bfloat16), embedding_or_output=emb))
    return params


def snapshot(params):
    out = []
    for p in params:
        out += [host(p.main_param), host(p.exp_avg), bf16_host(p.model)]
        if p.exp_avg_sq is not None:
            out.append(host(p.exp_avg_sq))
    return out


@pytest.mark.parametrize("clip,order", [(0.0, "auto"), (0.5, "auto"), (0.0, "grouped")])
def test_captured_step_replays_bit_exact(clip, order):
    """Eager steps and the replays of a captured step give the same bits, with
    the iterations evaluated one by one and in groups (whose launches rotate
    four square buffers)."""
    hm = mp.muon_hp(lr=0.02, momentum=0.95, ns_order=order)
    ha = mp.adamw_hp(lr=1e-3, weight_decay=0.1, step=1)

    def step(params, ws):
        if clip > 0:
            mp.mixed_step_clipped(params, hm, ha, clip, ws)
        else:
            mp.mixed_step(params, hm, ha, ws)

    eager, captured = make_params(), make_params()
    nbytes = mp.workspace_size(eager, clip=clip > 0, ns_order=order)
    ws_e = mp.alloc_workspace(nbytes)
    ws_c = mp.alloc_workspace(nbytes)
    reps = 3
    for _ in range(reps):
        step(eager, ws_e)
    torch.cuda.synchronize()

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step(captured, ws_c)          # first call outside capture: one-time setup
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step(captured, ws_c)
    for _ in range(reps - 1):
        graph.replay()
    torch.cuda.synchronize()
    assert mp.device_status(ws_c) == mp.OPT_OK
    for a, b in zip(snapshot(eager), snapshot(captured)):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
