"""Seeded synthetic workloads for the optimizer step.

This module only describes parameter sets and draws random numbers; it holds
none of the optimizer's arithmetic.  Both the CUDA path (tests, bench) and the
oracle take their inputs from here.

Five workloads, shaped like the pages' examples (a 4096x1024 / 1024x4096
pair as in the memory-ledger script of "优化器：AdamW、Muon 与分布式优化器",
and a Llama-like 16-layer model):

  tiny_mixed       one 256x512 Muon matrix + one 512-vector for AdamW, 10 steps
  adamw_8m         4096x1024 + 1024x4096 AdamW, 100 steps
  muon_8m_skewed   the same two shapes under Muon, gradient = noise + rank-8
                   component of 10x the noise RMS, 50 steps
  adamw_sweep_10k  10,000 AdamW tensors, sizes log-uniform in [1, 2^24), 20 steps
  llama16_mixed    16 layers x {q,o 4096^2; k,v 1024x4096; gate,up 14336x4096;
                   down 4096x14336} under Muon; embedding + LM head
                   (128256x4096) + 33 RMSNorm vectors of 4096 under AdamW; 10 steps

Distributions: N(0, s) means mean 0, standard deviation s.  Seeds: tensor i
of a workload draws its initial value from (seed 0, i) and its step-t
gradient from (seed 1000 + t, i).
"""

from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

INIT_SEED = 0
GRAD_SEED_BASE = 1000


@dataclasses.dataclass(frozen=True)
class TensorSpec:
    name: str
    shape: tuple
    init: str                  # "normal" or "ones"
    init_std: float = 0.0
    grad_std: float = 1e-3
    lowrank: int = 0           # rank of the added gradient component (0: none)
    lowrank_rms: float = 0.0   # entry RMS of that component
    embedding_or_output: bool = False

    @property
    def numel(self):
        return int(np.prod(self.shape))


@dataclasses.dataclass(frozen=True)
class AdamWHP:
    lr: float = 1e-3
    beta1: float = 0.9
    beta2: float = 0.999
    eps: float = 1e-8
    weight_decay: float = 0.01


@dataclasses.dataclass(frozen=True)
class MuonHP:
    lr: float = 0.02
    momentum: float = 0.95
    weight_decay: float = 0.0
    nesterov: bool = True
    ns_steps: int = 5


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    tensors: tuple
    steps: int
    adamw: Optional[AdamWHP]
    muon: Optional[MuonHP]
    force_adamw: bool = False  # every tensor goes to AdamW (AdamW-only workloads)

    @property
    def numel(self):
        return sum(t.numel for t in self.tensors)


def _sweep_sizes(n=10_000, seed=INIT_SEED, max_log2=24):
    rng = np.random.default_rng([seed, 424242])
    u = rng.random(n)
    return np.floor(np.exp(u * math.log(2.0 ** max_log2))).astype(np.int64)


def tiny_mixed():
    return Workload(
        "tiny_mixed",
        (TensorSpec("hidden", (256, 512), "normal", 0.02, grad_std=1e-2),
         TensorSpec("vector", (512,), "ones", grad_std=1e-2)),
        steps=10, adamw=AdamWHP(weight_decay=0.01), muon=MuonHP())


def adamw_8m():
    return Workload(
        "adamw_8m",
        (TensorSpec("w1", (4096, 1024), "normal", 1.0), TensorSpec("w2", (1024, 4096), "normal", 1.0)),
        steps=100, adamw=AdamWHP(weight_decay=0.1), muon=None, force_adamw=True)


def muon_8m_skewed():
    kw = dict(init="normal", init_std=0.02, grad_std=1e-3, lowrank=8, lowrank_rms=1e-2)
    return Workload(
        "muon_8m_skewed",
        (TensorSpec("w1", (4096, 1024), **kw), TensorSpec("w2", (1024, 4096), **kw)),
        steps=50, adamw=None, muon=MuonHP())


def adamw_sweep_10k(n=10_000):
    sizes = _sweep_sizes(n)
    return Workload(
        "adamw_sweep_10k",
        tuple(TensorSpec(f"t{i}", (int(s),), "normal", 1.0) for i, s in enumerate(sizes)),
        steps=20, adamw=AdamWHP(weight_decay=0.01), muon=None, force_adamw=True)


LLAMA_LAYER = (("q", (4096, 4096)), ("k", (1024, 4096)), ("v", (1024, 4096)), ("o", (4096, 4096)),
               ("gate", (14336, 4096)), ("up", (14336, 4096)), ("down", (4096, 14336)))


def llama16_mixed(layers=16, vocab=128256, hidden=4096):
    ts: List[TensorSpec] = [TensorSpec("embed", (vocab, hidden), "normal", 0.02, embedding_or_output=True)]
    for l in range(layers):
        ts.append(TensorSpec(f"l{l}.attn_norm", (hidden,), "ones"))
        for nm, shp in LLAMA_LAYER:
            ts.append(TensorSpec(f"l{l}.{nm}", shp, "normal", 0.02))
        ts.append(TensorSpec(f"l{l}.mlp_norm", (hidden,), "ones"))
    ts.append(TensorSpec("final_norm", (hidden,), "ones"))
    ts.append(TensorSpec("lm_head", (vocab, hidden), "normal", 0.02, embedding_or_output=True))
    return Workload("llama16_mixed", tuple(ts), steps=10,
                    adamw=AdamWHP(weight_decay=0.1), muon=MuonHP(weight_decay=0.0))


def llama_mlp_1layer():
    """gate, up and down of one layer of the 16-layer set: the dominant
    Newton-Schulz shape class (4096 x 14336) at a few GB, the small case for
    kernel profiling."""
    ts = tuple(TensorSpec(nm, shp, "normal", 0.02) for nm, shp in LLAMA_LAYER if nm in ("gate", "up", "down"))
    return Workload("llama_mlp_1layer", ts, steps=10, adamw=None, muon=MuonHP(weight_decay=0.0))


def attn_qo8():
    """Eight 4096 x 4096 matrices (the q/o shape class of the 16-layer set) under
    Muon: 256 MB of fp16 iterate, larger than L2, a few GB in all; the small
    case for profiling that class."""
    ts = tuple(TensorSpec(f"qo{i}", (4096, 4096), "normal", 0.02) for i in range(8))
    return Workload("attn_qo8", ts, steps=10, adamw=None, muon=MuonHP(weight_decay=0.0))


def attn_kv32():
    """The 32 k/v matrices (1024 x 4096) of the 16-layer set under Muon: that
    shape class's group exactly as the full step batches it."""
    ts = tuple(TensorSpec(f"kv{i}", (1024, 4096), "normal", 0.02) for i in range(32))
    return Workload("attn_kv32", ts, steps=10, adamw=None, muon=MuonHP(weight_decay=0.0))


WORKLOADS = {
    "tiny_mixed": tiny_mixed,
    "adamw_8m": adamw_8m,
    "muon_8m_skewed": muon_8m_skewed,
    "adamw_sweep_10k": adamw_sweep_10k,
    "llama16_mixed": llama16_mixed,
    "llama_mlp_1layer": llama_mlp_1layer,
    "attn_qo8": attn_qo8,
    "attn_kv32": attn_kv32,
}


def scaled_copy(w: Workload, name: str, shapes) -> Workload:
    """The same distributions and hyper-parameters on other shapes (used for
    small parity cases with ragged sizes)."""
    base = w.tensors[0]
    ts = tuple(dataclasses.replace(base, name=f"s{i}", shape=tuple(s)) for i, s in enumerate(shapes))
    return dataclasses.replace(w, name=name, tensors=ts)


# --------------------------------------------------------------------------
# host (numpy) generators: exact bytes both sides can see
# --------------------------------------------------------------------------

def init_value(spec: TensorSpec, index: int, seed: int = INIT_SEED) -> np.ndarray:
    if spec.init == "ones":
        return np.ones(spec.shape, np.float32)
    rng = np.random.default_rng([seed, index])
    return (rng.standard_normal(spec.shape, dtype=np.float32) * np.float32(spec.init_std)).astype(np.float32)


def grad_value(spec: TensorSpec, index: int, step: int) -> np.ndarray:
    rng = np.random.default_rng([GRAD_SEED_BASE + int(step), index])
    g = rng.standard_normal(spec.shape, dtype=np.float32) * np.float32(spec.grad_std)
    if spec.lowrank:
        R, C = spec.shape
        Pm = rng.standard_normal((R, spec.lowrank), dtype=np.float32)
        Qm = rng.standard_normal((C, spec.lowrank), dtype=np.float32)
        g = g + (Pm @ Qm.T) * np.float32(spec.lowrank_rms / math.sqrt(spec.lowrank))
    return g.astype(np.float32)


# --------------------------------------------------------------------------
# device (torch) generators: same distributions, drawn on the GPU for
# workloads too large to draw on the host.  Seeded, but a different stream of
# numbers from the numpy generators; whoever checks such a run copies the
# sampled inputs back before the step.
# --------------------------------------------------------------------------

def torch_init_(t, spec: TensorSpec, index: int, seed: int = INIT_SEED):
    import torch
    if spec.init == "ones":
        t.fill_(1.0)
        return t
    g = torch.Generator(device=t.device)
    g.manual_seed(seed * 1_000_003 + index)
    t.normal_(0.0, spec.init_std, generator=g)
    return t


def torch_grad_(t, spec: TensorSpec, index: int, step: int):
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed((GRAD_SEED_BASE + int(step)) * 1_000_003 + index)
    t.normal_(0.0, spec.grad_std, generator=g)
    if spec.lowrank:
        R, C = spec.shape
        Pm = torch.randn(R, spec.lowrank, generator=g, device=t.device)
        Qm = torch.randn(C, spec.lowrank, generator=g, device=t.device)
        t.view(R, C).add_(Pm @ Qm.T, alpha=spec.lowrank_rms / math.sqrt(spec.lowrank))
    return t
