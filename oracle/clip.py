"""Global gradient-norm clipping oracle (test infrastructure only; see
``oracle/__init__``).

Definition ("02 · Optimizer：算法与 infra" §11.1, with §11.4 for the chained
Muon + AdamW case: one global norm over the gradients of both groups)::

    total_norm = sqrt( sum_p ||g_p||^2 )
    clip_coeff = max_norm / (total_norm + 1e-6)
    if clip_coeff < 1:  g_p <- clip_coeff * g_p      (every p, the same factor)

and clipping is skipped entirely when max_norm <= 0 (§11.1: clip_grad <= 0).
Everything here is fp64.
"""

from __future__ import annotations

import numpy as np


def total_norm(grads) -> float:
    """sqrt of the sum of squares of every gradient, in fp64."""
    return float(np.sqrt(sum(float(np.sum(np.asarray(g, dtype=np.float64) ** 2)) for g in grads)))


def clip_scale(grads, max_norm: float) -> float:
    """The factor every gradient is multiplied by: clip_coeff when it is
    below 1, else 1; 1 when clipping is off (max_norm <= 0)."""
    if max_norm <= 0:
        return 1.0
    coeff = max_norm / (total_norm(grads) + 1e-6)
    return coeff if coeff < 1.0 else 1.0


def clip(grads, max_norm: float):
    """Clipped copies of the gradients (fp64)."""
    s = clip_scale(grads, max_norm)
    return [np.asarray(g, dtype=np.float64) * s for g in grads]
