"""The data-parallel sharded step on the CPU: the plan (opt_shard_plan, host
only) and a world-size-2 gloo run whose per-rank compute is the oracle.

What the sharding must guarantee ("02 · Optimizer：算法与 infra" §12.1-§12.2,
§14.3; "优化器：AdamW、Muon 与分布式优化器", distributed Muon, scheme ③):
every AdamW element and every Muon matrix is stepped by exactly one rank,
Muon matrices stay whole, and after the exchange every rank holds the bf16
model of the unsharded step.  With the oracle as each rank's compute the
sharded result must equal the unsharded oracle bit for bit (AdamW is
elementwise; each Muon matrix runs the same oracle call on its owner)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as tmp

import mixed_precision_optimizer_gb300 as mp
from mixed_precision_optimizer_gb300 import sharded as sh
from oracle import adamw as OA
from oracle import muon as OM

LLAMA_LAYER = [((4096, 4096), None, False), ((1024, 4096), None, False), ((1024, 4096), None, False),
               ((4096, 4096), None, False), ((14336, 4096), None, False), ((14336, 4096), None, False),
               ((4096, 14336), None, False)]


def llama16_specs():
    specs = [((128256, 4096), None, True)]
    for _ in range(16):
        specs.append(((4096,), None, False))
        specs += LLAMA_LAYER
        specs.append(((4096,), None, False))
    specs += [((4096,), None, False), ((128256, 4096), None, True)]
    return specs


def ns_work(shape):
    a, b = sorted(shape)
    return 2.0 * (2.0 * a * a * b + a ** 3)


@pytest.mark.parametrize("world", [1, 2, 3, 8])
def test_plan_partitions_every_element_and_matrix_once(world):
    specs = llama16_specs()
    p = sh.shard_plan(specs, world)
    adamw = [i for i, (s, _, e) in enumerate(specs) if not (len(s) == 2 and not e)]
    muon = [i for i in range(len(specs)) if i not in adamw]
    N = 0
    for i in adamw:
        N = -(-N // sh.ALIGN_ELEMS) * sh.ALIGN_ELEMS + int(np.prod(specs[i][0]))
    b = p.rank_bounds
    assert b[0] == 0 and b[-1] == N and all(x <= y for x, y in zip(b, b[1:]))
    assert all(x % sh.ALIGN_ELEMS == 0 for x in b[1:-1])
    lens = [p.adamw_len(r) for r in range(world)]
    assert max(lens) - min(lens) <= sh.ALIGN_ELEMS + 1
    # every AdamW element owned by exactly one rank, in list order
    off = 0
    for i in adamw:
        off = -(-off // sh.ALIGN_ELEMS) * sh.ALIGN_ELEMS        # each tensor starts aligned
        assert p.flat_begin[i] == off and p.owner[i] == -1
        n = int(np.prod(specs[i][0]))
        covered = sorted(p.adamw_range(i, r) for r in range(world) if p.adamw_range(i, r))
        assert covered[0][0] == 0 and covered[-1][1] == n
        assert all(x[1] == y[0] for x, y in zip(covered, covered[1:]))
        assert all(lo % sh.ALIGN_ELEMS == 0 for lo, _ in covered)   # cuts aligned within the tensor
        off += n
    # Muon: whole matrices, one owner each, LPT balance on Newton-Schulz work
    assert all(0 <= p.owner[i] < world and p.flat_begin[i] == -1 for i in muon)
    loads = [sum(ns_work(specs[i][0]) for i in muon if p.owner[i] == r) for r in range(world)]
    assert np.allclose(loads, p.muon_work)
    biggest = max(ns_work(specs[i][0]) for i in muon)
    assert max(loads) <= sum(loads) / world + biggest          # the LPT bound
    assert p.shapes == [s for s, _, _ in specs]


def test_plan_lpt_order_and_ties():
    """Largest first onto the least-loaded rank, lowest rank on ties, equal
    sizes in list order."""
    specs = [((64, 64), "muon", False), ((256, 512), "muon", False), ((64, 64), "muon", False),
             ((128, 128), "muon", False), ((64, 64), "muon", False)]
    p = sh.shard_plan(specs, 2)
    # 256x512 -> r0; 128x128 -> r1; 64x64 (#0) -> r1; #2 -> r1; #4 -> r1 (r1 still lighter)
    w = [ns_work(s) for s, _, _ in specs]
    assert p.owner[1] == 0 and p.owner[3] == 1
    loads = [w[1], w[3]]
    for i in (0, 2, 4):
        r = 0 if loads[0] <= loads[1] else 1
        assert p.owner[i] == r
        loads[r] += w[i]


def test_plan_rejects_bad_arguments():
    with pytest.raises(mp.MpoptError):
        sh.shard_plan([((4, 4), None, False)], 0)
    with pytest.raises(mp.MpoptError):
        sh.shard_plan([((4, 4), None, False)], 2, align=0)
    with pytest.raises(mp.MpoptError):
        sh.shard_plan([((2, 3, 4), "muon", False)], 2)     # Muon needs 2-D


# ------------------------------------------------------------ gloo run --

AH = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
MH = dict(lr=0.02, momentum=0.95)
SPECS = [((300,), None, False), ((96, 160), None, False), ((50, 64), None, True), ((160, 96), None, False),
         ((1000,), None, False), ((64, 64), None, False), ((7,), None, False), ((128, 200), None, False)]


def make_full(seed=0):
    """Seeded full-size CPU tensors of the small mixed workload (Param per tensor)."""
    rng = np.random.default_rng(seed)
    out = []
    for shape, kind, emb in SPECS:
        W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
        g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
        m = (rng.standard_normal(shape) * 1e-3).astype(np.float32)
        v = (np.abs(rng.standard_normal(shape)) * 1e-5).astype(np.float32)
        T = lambda a: torch.from_numpy(a.copy())
        model = torch.from_numpy(OA.bf16_rne(W).view(np.int16)).view(torch.bfloat16).reshape(shape)
        out.append(mp.Param(T(W), T(g), T(m), T(v), model.clone(), emb, kind))
    return out


def oracle_step(pieces, hp_muon, hp_adamw, workspace):
    """The oracle as a rank's compute, in place on CPU tensors: AdamW in fp32
    (literal order), Muon in fp64 (stored back as fp32), bf16 copies rounded
    to nearest even."""
    for p in pieces:
        routed_muon = p.kind == "muon" or (p.kind is None and p.main_param.dim() == 2 and not p.embedding_or_output)
        if routed_muon:
            W, m = p.main_param.numpy(), p.exp_avg.numpy()
            Wn, mn, _ = OM.muon_step(W, p.main_grad.numpy(), m, **MH)
            W[...] = Wn.astype(np.float32)
            m[...] = mn.astype(np.float32)
        else:
            W = p.main_param.numpy().reshape(-1)
            OA.adamw_step_fp32(W, p.main_grad.numpy().reshape(-1).copy(), p.exp_avg.numpy().reshape(-1),
                               p.exp_avg_sq.numpy().reshape(-1), t=3, **AH)
        p.model.view(torch.int16).numpy()[...] = OA.bf16_rne(p.main_param.numpy()).view(np.int16)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, q):
    try:
        _rank_body(rank, world, port, q)
    except BaseException as e:          # report at once instead of leaving the queue empty
        q.put((rank, repr(e), None, None, None))
        raise


def _rank_body(rank, world, port, q):
    import datetime
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=60))
    full = make_full()
    plan = sh.shard_plan(full, world)
    state = sh.RankState.empty(plan, rank, "cpu")
    state.load(plan, full)
    # the rank keeps only the replicated main_grad and bf16 model of every tensor
    params = [mp.Param(None, p.main_grad, None, None, p.model, p.embedding_or_output, p.kind) for p in full]
    sh.sharded_step(params, plan, state, None, None, None, local_step=oracle_step)
    bits = [p.model.view(torch.int16).numpy().copy() for p in params]
    q.put((rank, bits, state.adamw_master.numpy().copy(),
           {i: (W.numpy().copy(), m.numpy().copy()) for i, (W, m) in state.muon.items()}, plan.rank_bounds))
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_step_gloo_matches_unsharded_oracle(world):
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        r, bits, master, muon, bounds = q.get(timeout=300)
        assert not isinstance(bits, str), f"rank {r}: {bits}"
        got[r] = (bits, master, muon, bounds)
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    # the unsharded step, same oracle
    ref = make_full()
    oracle_step(ref, None, None, None)
    want_bits = [p.model.view(torch.int16).numpy() for p in ref]
    plan = sh.shard_plan(ref, world)
    for r in range(world):
        bits, master, muon, bounds = got[r]
        for i, (b, wb) in enumerate(zip(bits, want_bits)):     # every rank: the full bf16 model
            assert np.array_equal(b, wb), (r, i)
        for i, (W, m) in muon.items():                        # owned Muon masters and momenta
            assert plan.owner[i] == r
            assert np.array_equal(W, ref[i].main_param.numpy()) and np.array_equal(m, ref[i].exp_avg.numpy())
        for i in range(len(SPECS)):                           # owned AdamW master pieces
            rng = plan.adamw_range(i, r)
            if rng:
                off = plan.flat_begin[i] + rng[0] - bounds[r]
                want = ref[i].main_param.numpy().reshape(-1)[rng[0]:rng[1]]
                assert np.array_equal(master[off:off + rng[1] - rng[0]].view(np.uint32), want.view(np.uint32))
    # both Muon and AdamW work was split across the ranks
    n_muon = sum(plan.is_muon(i) for i in range(len(SPECS)))
    assert len({plan.owner[i] for i in range(len(SPECS)) if plan.is_muon(i)}) == min(world, n_muon)
    assert all(plan.adamw_len(r) > 0 for r in range(world))
