"""The sharded step's GPU work on one GPU: the ranks of a world of 2 or 3 run
one after another (no rank waits on another), each stepping its own pieces
through opt_mixed_step: AdamW ranges as 1-D views at arbitrary element
offsets into its flat state and into the shared main_grad and bf16 model,
and its whole Muon matrices.  Every piece is written by exactly one rank, so
after all ranks the shared bf16 model is what the exchange would deliver.
It must equal the unsharded step bit for bit (AdamW is elementwise; Muon's
arithmetic does not depend on how matrices are grouped), and so must each
rank's master and state pieces.  The exchange itself (torch.distributed
broadcasts) is covered on CPU ranks in test_sharded_host.py."""

import numpy as np
import pytest

from gpu_helpers import bf16_host, dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from mixed_precision_optimizer_gb300 import sharded as sh
from oracle import adamw as OA

pytestmark = pytest.mark.gpu

# ragged AdamW sizes (cuts fall mid-tensor at unaligned offsets), wide, tall
# and square Muon matrices, and an embedding that AdamW takes
SHAPES = [((1000,), False), ((96, 160), False), ((300, 64), True), ((160, 96), False), ((37,), False),
          ((256, 256), False), ((4099,), False), ((128, 200), False), ((200, 128), False), ((1,), False)]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def full_params(seed):
    rng = np.random.default_rng(seed)
    out = []
    for shape, emb in SHAPES:
        W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
        g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
        m = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
        v = (np.abs(rng.standard_normal(shape)) * 1e-5).astype(np.float32)
        model = torch.zeros(shape, dtype=torch.bfloat16, device="cuda")
        out.append(mp.Param(dev(W), dev(g), dev(m), dev(v), model, emb))
    return out


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_ranks_match_unsharded_step(world):
    hm = mp.muon_hp(lr=0.02, momentum=0.95, weight_decay=0.01)
    ha = mp.adamw_hp(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1, step=4)
    ref = full_params(7)
    full = full_params(7)
    plan = sh.shard_plan(full, world, align=8)
    assert len({plan.owner[i] for i in range(len(SHAPES)) if plan.is_muon(i)}) > 1
    states = []
    for r in range(world):
        st = sh.RankState.empty(plan, r, "cuda")
        st.load(plan, full)
        states.append(st)
    shared = [mp.Param(None, p.main_grad, None, None, p.model, p.embedding_or_output) for p in full]
    for r in range(world):
        pieces = sh.rank_params(shared, plan, states[r])
        ws = mp.alloc_workspace(mp.workspace_size(pieces))
        mp.mixed_step(pieces, hm, ha, ws)
        assert mp.device_status(ws) == mp.OPT_OK
    ws = mp.alloc_workspace(mp.workspace_size(ref))
    mp.mixed_step(ref, hm, ha, ws)
    torch.cuda.synchronize()
    for i, (p, q) in enumerate(zip(shared, ref)):
        assert np.array_equal(bf16_host(p.model), bf16_host(q.model)), i
        assert np.array_equal(bf16_host(q.model), OA.bf16_rne(host(q.main_param)))
    for r, st in enumerate(states):
        base = plan.rank_bounds[r]
        for i, q in enumerate(ref):
            if plan.is_muon(i):
                if plan.owner[i] == r:
                    W, m = st.muon[i]
                    assert np.array_equal(host(W), host(q.main_param)) and np.array_equal(host(m), host(q.exp_avg))
                continue
            rng = plan.adamw_range(i, r)
            if rng is None:
                continue
            lo, hi = rng
            off = plan.flat_begin[i] + lo - base
            for mine, want in ((st.adamw_master, q.main_param), (st.adamw_m, q.exp_avg), (st.adamw_v, q.exp_avg_sq)):
                a = host(mine[off:off + hi - lo]).view(np.uint32)
                b = host(want.reshape(-1)[lo:hi]).view(np.uint32)
                assert np.array_equal(a, b), (r, i)
