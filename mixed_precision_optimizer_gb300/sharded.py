"""Data-parallel sharded optimizer step: ZeRO-1 for AdamW, one owner per Muon
matrix ("02 · Optimizer：算法与 infra" §12.1-§12.2, §14.3; "优化器：AdamW、Muon 与
分布式优化器", distributed Muon, scheme ③).

Every rank holds the full bf16 model copy and the full reduced gradient
(main_grad), but fp32 master weights and optimizer state only for what it
owns:

  * AdamW elements: the AdamW tensors, end to end in list order, form one
    index space that opt_shard_plan cuts into ``world`` near-equal contiguous
    ranges (the cuts ignore tensor boundaries).  A rank's master, m and v are
    three flat buffers of its range's length.
  * Muon matrices stay whole (Newton-Schulz needs the whole matrix); each has
    one owner, assigned by LPT on its Newton-Schulz work.

One step on rank r is: the library's opt_mixed_step over rank r's pieces (views
into its state, its slices of main_grad and of the bf16 model), then every
rank receives the bf16 values of the pieces it does not own, broadcast by
their owners (torch.distributed: NCCL on GPUs, gloo on CPUs).  The owners' bf16
pieces come out of the same kernels as in the unsharded step, so a sharded
step gives the unsharded step's results bit for bit.

Only plumbing lives here: the plan is computed by the C library, the
arithmetic by its kernels, and the exchange by the collective library.
"""

from __future__ import annotations

import ctypes
import dataclasses
from typing import Callable, Dict, List, Optional, Sequence, Tuple

from . import (KIND_ADAMW, KIND_AUTO, KIND_MUON, FLAG_EMBEDDING_OR_OUTPUT, OptShardEntry, OptTensor, Param,
               _check, lib, mixed_step)

ALIGN_ELEMS = 64   # inner cuts of the AdamW index space: 256-byte fp32 / 128-byte bf16 boundaries


@dataclasses.dataclass
class ShardPlan:
    """Who steps what (opt_shard_plan).  ``owner[i]`` is the rank that owns
    Muon tensor i (-1 for AdamW tensors and empty ones); ``flat_begin[i]`` is
    AdamW tensor i's first index in the AdamW index space (-1 for Muon);
    rank r owns AdamW indices [rank_bounds[r], rank_bounds[r + 1])."""
    world: int
    rank_bounds: List[int]
    owner: List[int]
    flat_begin: List[int]
    numel: List[int]
    shapes: List[tuple]
    muon_work: List[float]

    def is_muon(self, i: int) -> bool:
        return self.owner[i] >= 0

    def adamw_range(self, i: int, r: int) -> Optional[Tuple[int, int]]:
        """Rank r's elements [lo, hi) of AdamW tensor i, or None."""
        fb = self.flat_begin[i]
        if fb < 0:
            return None
        lo = max(self.rank_bounds[r], fb)
        hi = min(self.rank_bounds[r + 1], fb + self.numel[i])
        return (lo - fb, hi - fb) if hi > lo else None

    def adamw_len(self, r: int) -> int:
        return self.rank_bounds[r + 1] - self.rank_bounds[r]

    def owned_muon(self, r: int) -> List[int]:
        return [i for i, o in enumerate(self.owner) if o == r]


def _spec(p) -> Tuple[tuple, Optional[str], bool]:
    """(shape, kind, embedding_or_output) of a Param or of such a tuple."""
    if isinstance(p, Param):
        t = p.main_grad if p.main_grad is not None else p.model
        return tuple(t.shape), p.kind, bool(p.embedding_or_output)
    shape, kind, emb = p
    return tuple(shape), kind, bool(emb)


def shard_plan(params: Sequence, world: int, align: int = ALIGN_ELEMS, routing: str = "auto") -> ShardPlan:
    """The sharding plan of a parameter list over ``world`` ranks.  Only
    shapes, kinds and the embedding/output flag are read, so ``params`` may be
    Params whose master and state are absent (a sharded rank) or tuples
    (shape, kind, embedding_or_output)."""
    specs = [_spec(p) for p in params]
    n = len(specs)
    arr = (OptTensor * max(1, n))()
    for i, (shape, kind, emb) in enumerate(specs):
        ct = OptTensor()
        ndim = len(shape)
        rows, cols = (shape if ndim == 2 else (1, int(_prod(shape))))
        ct.rows, ct.cols, ct.ndim = int(rows), int(cols), ndim
        ct.kind = {None: KIND_AUTO, "adamw": KIND_ADAMW, "muon": KIND_MUON}[kind]
        ct.flags = FLAG_EMBEDDING_OR_OUTPUT if emb else 0
        arr[i] = ct
    entries = (OptShardEntry * max(1, n))()
    bounds = (ctypes.c_int64 * (world + 1))()
    work = (ctypes.c_double * world)()
    r = {"auto": KIND_AUTO, "adamw": KIND_ADAMW, "muon": KIND_MUON}[routing]
    _check(lib().opt_shard_plan(arr, n, r, int(world), int(align), entries, bounds, work), "opt_shard_plan")
    return ShardPlan(world=int(world), rank_bounds=[int(b) for b in bounds],
                     owner=[int(entries[i].owner) for i in range(n)],
                     flat_begin=[int(entries[i].flat_begin) for i in range(n)],
                     numel=[int(_prod(s)) for s, _, _ in specs], shapes=[s for s, _, _ in specs],
                     muon_work=[float(work[k]) for k in range(world)])


def _prod(shape) -> int:
    out = 1
    for x in shape:
        out *= int(x)
    return out


@dataclasses.dataclass
class RankState:
    """The fp32 master weights and optimizer state one rank owns: three flat
    buffers over its AdamW range (master, m, v) and (master, momentum) of
    every Muon matrix it owns."""
    rank: int
    adamw_master: object
    adamw_m: object
    adamw_v: object
    muon: Dict[int, Tuple[object, object]]

    @staticmethod
    def empty(plan: ShardPlan, rank: int, device) -> "RankState":
        import torch
        n = plan.adamw_len(rank)
        z = lambda *shape: torch.zeros(shape, dtype=torch.float32, device=device)
        return RankState(rank, z(n), z(n), z(n), {i: (z(*plan.shapes[i]), z(*plan.shapes[i]))
                                                  for i in plan.owned_muon(rank)})

    def load(self, plan: ShardPlan, full: Sequence[Param]):
        """Copies the owned pieces of full-size master/state tensors (the
        unsharded optimizer's) into this rank's buffers."""
        base = plan.rank_bounds[self.rank]
        for i, p in enumerate(full):
            if plan.is_muon(i):
                if plan.owner[i] == self.rank:
                    W, m = self.muon[i]
                    W.copy_(p.main_param)
                    m.copy_(p.exp_avg)
                continue
            rng = plan.adamw_range(i, self.rank)
            if rng is None:
                continue
            lo, hi = rng
            off = plan.flat_begin[i] + lo - base
            for dst, src in ((self.adamw_master, p.main_param), (self.adamw_m, p.exp_avg),
                             (self.adamw_v, p.exp_avg_sq)):
                dst[off:off + hi - lo].copy_(src.reshape(-1)[lo:hi])


def rank_params(params: Sequence[Param], plan: ShardPlan, state: RankState) -> List[Param]:
    """The Params rank ``state.rank`` steps: a 1-D AdamW Param per owned piece
    of an AdamW tensor (views into the rank's flat state and into the
    tensor's main_grad and bf16 model), and every owned Muon matrix whole.
    ``params`` hold the replicated main_grad and bf16 model copy of every
    tensor; their main_param and state are not read."""
    r = state.rank
    base = plan.rank_bounds[r]
    out = []
    for i, p in enumerate(params):
        if p.model is None:
            raise ValueError("a sharded step needs the bf16 model copy of every parameter")
        if plan.is_muon(i):
            if plan.owner[i] == r:
                W, m = state.muon[i]
                out.append(Param(W, p.main_grad, m, None, p.model, p.embedding_or_output, "muon", p.scale_shape))
            continue
        rng = plan.adamw_range(i, r)
        if rng is None:
            continue
        lo, hi = rng
        off = plan.flat_begin[i] + lo - base
        sl = slice(off, off + hi - lo)
        out.append(Param(state.adamw_master[sl], p.main_grad.reshape(-1)[lo:hi], state.adamw_m[sl],
                         state.adamw_v[sl], p.model.reshape(-1)[lo:hi], p.embedding_or_output, "adamw"))
    return out


def exchange(params: Sequence[Param], plan: ShardPlan, group=None, src_ranks: Optional[Sequence[int]] = None):
    """Every rank receives the bf16 model values of the pieces it does not own:
    one broadcast per owned piece, from its owner, in list order (the same
    sequence of collectives on every rank).  bf16 travels as its bytes (a
    type every backend broadcasts).  ``src_ranks[r]`` maps plan rank r to its
    global rank (default: the same)."""
    import torch
    import torch.distributed as dist
    if plan.world == 1:
        return
    g = lambda r: src_ranks[r] if src_ranks is not None else r
    works = []
    for i, p in enumerate(params):
        if plan.numel[i] == 0:
            continue
        if not p.model.is_contiguous():
            raise ValueError("the bf16 model copies must be contiguous (a broadcast into a reshaped copy is lost)")
        raw = p.model.reshape(-1).view(torch.uint8)      # 2 bytes per element
        if plan.is_muon(i):
            works.append(dist.broadcast(raw, src=g(plan.owner[i]), group=group, async_op=True))
            continue
        for r in range(plan.world):
            rng = plan.adamw_range(i, r)
            if rng is not None:
                works.append(dist.broadcast(raw[2 * rng[0]:2 * rng[1]], src=g(r), group=group, async_op=True))
    for w in works:
        w.wait()


def sharded_step(params: Sequence[Param], plan: ShardPlan, state: RankState, hp_muon, hp_adamw, workspace,
                 local_step: Optional[Callable] = None, group=None, prepared=None):
    """One data-parallel step on this rank: the library's mixed step over the
    rank's pieces, then the bf16 exchange.  ``local_step(pieces, hp_muon,
    hp_adamw, workspace)`` defaults to mixed_step; ``prepared`` may hold the
    rank's pieces marshalled once (mixed_step accepts a Prepared list)."""
    pieces = prepared if prepared is not None else rank_params(params, plan, state)
    (local_step or mixed_step)(pieces, hp_muon, hp_adamw, workspace)
    exchange(params, plan, group)
