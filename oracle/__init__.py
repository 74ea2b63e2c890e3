"""CPU oracle for the mixed-precision optimizer step.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code, tables or constants with the CUDA
library in ``mixed_precision_optimizer_gb300/``; the two meet only through the
seeded inputs built by ``synthetic/``.

The oracle is plain numpy: slow, literal, and written to be checked against
the pages by eye.

* ``adamw``  -- Adam / AdamW (decoupled decay) and Adam + L2, in fp32 (the
  precision the pages fix for master weights and moments) and in fp64, plus
  the step scalars (bias corrections) and round-to-nearest-even bf16.
  Sources: "02 · Optimizer：算法与 infra" §2 (Adam), §3 (AdamW), §9.1/§9.2
  (fp32 master, writeback); "优化器：AdamW、Muon 与分布式优化器", section
  "AdamW：解耦的权重衰减" (the decay experiment).
* ``muon``   -- lerp momentum, Nesterov lerp, Newton-Schulz quintic, the
  0.2*sqrt(max(A, B)) scaled update with decoupled decay, all in fp64; an
  SVD polar factor U V^T for sanity checks only.
  Sources: "02 · Optimizer：算法与 infra" §1, §5.1, §5.2, §5.4, §14.1;
  "优化器：AdamW、Muon 与分布式优化器", section "Muon：把更新“正交化”".

* ``clip``   -- global gradient-norm clipping, fp64.
  Source: "02 · Optimizer：算法与 infra" §11.1 (definition) and §11.4 (one
  global norm shared by the Muon and AdamW groups).

Every function is pinned by a CPU test in ``tests/test_oracle_pins.py``
against values the pages print, closed forms, or library routines.  No
function here is "parity unpinned".
"""

from . import adamw, clip, muon  # noqa: F401
