"""Muon oracle in fp64 (test infrastructure only; see ``oracle/__init__``).

Definitions followed
--------------------
Momentum as an EMA written with lerp(a, b, w) = a + w (b - a)
("02 · Optimizer：算法与 infra" §1)::

    m_t     = lerp(m_{t-1}, g_t, 1 - mu)
    gtilde  = lerp(g_t, m_t, mu)            (Nesterov; plain momentum: m_t)

Newton-Schulz quintic (same page §5.2; "优化器：AdamW、Muon 与分布式优化器",
``newton_schulz`` in the Muon section)::

    X = G / (||G||_F + eps)                 eps = 1e-7
    if rows > cols: X = X^T                 (work on the wide orientation)
    repeat steps:  A = X X^T ;  B = b A + c A A ;  X = a X + B X
    result = X^T if transposed else X       (a, b, c) = (3.4445, -4.7750, 2.0315)

Update with decoupled decay and the RMS-matching scale (§5.4 Moonlight Eq. 3
and Eq. 4; §14.1 decay before the update)::

    W_t = W_{t-1} * (1 - lr * lambda) - lr * 0.2 * sqrt(max(A, B)) * O_t

Variants (same page, §14.6 and §14.4, §5.5, §1):

* scale modes on the Newton-Schulz output, with fan_out = rows (m) and
  fan_in = cols (n) of the parameter: ``spectral`` sqrt(max(m, n)) (the
  default, Eq. 4's shape factor), ``shape_scaling`` sqrt(max(1, m / n)),
  ``unit_rms_norm`` sqrt(m / n), each times a free factor (0.2 above);
* QKV split: a [q + k + v, h] parameter is orthogonalised block by block
  (rows q, k, v separately) and the blocks are put back together; the scale
  factor uses the whole parameter's shape;
* a per-iteration coefficient schedule (a list of (a, b, c), one per step);
* plain momentum SGD (no orthogonalisation): W -= lr * gtilde (§1).

The iteration is the oracle; ``polar_svd`` (U V^T from an SVD, §5.1) is only
a sanity reference, since five quintic steps do not converge to it.

Readings where the pages are silent
-----------------------------------
* The Frobenius norm and every product are fp64 here; the momentum buffer is
  returned in fp64 and the caller rounds to fp32 where it compares against
  fp32 state.
* Transpose only when rows > cols strictly; square matrices are not
  transposed.
* The 0.2*sqrt(max(A, B)) scale multiplies the Newton-Schulz output, and the
  decay factor multiplies W_{t-1} (not W after the update).
"""

from __future__ import annotations

import math

import numpy as np

NS_COEFFS = (3.4445, -4.7750, 2.0315)
NS_EPS = 1e-7


def lerp(a, b, w):
    """lerp(a, b, w) = a + w (b - a), §1 of "02 · Optimizer：算法与 infra"."""
    return a + w * (b - a)


def momentum_update(m, g, mu, nesterov=True):
    """Returns (m_t, gtilde) in fp64.  m_t = lerp(m, g, 1-mu); gtilde =
    lerp(g, m_t, mu) with Nesterov, else m_t."""
    m = np.asarray(m, dtype=np.float64)
    g = np.asarray(g, dtype=np.float64)
    m_new = lerp(m, g, 1.0 - mu)
    gt = lerp(g, m_new, mu) if nesterov else m_new
    return m_new, gt


def _schedule(coeffs, steps):
    """One (a, b, c) per iteration: a single triple repeats; a list gives the
    coefficients of each iteration in order."""
    if len(coeffs) == 3 and np.isscalar(coeffs[0]):
        return [tuple(coeffs)] * int(steps)
    assert len(coeffs) == int(steps)
    return [tuple(c) for c in coeffs]


def newton_schulz(G, steps=5, coeffs=NS_COEFFS, eps=NS_EPS):
    """Quintic Newton-Schulz iteration in fp64, literally as printed."""
    G = np.asarray(G, dtype=np.float64)
    assert G.ndim == 2
    X = G / (np.linalg.norm(G) + eps)          # ||.||_F for a 2-D array
    transposed = G.shape[0] > G.shape[1]
    if transposed:
        X = X.T
    for a, b, c in _schedule(coeffs, steps):
        A = X @ X.T
        B = b * A + c * (A @ A)
        X = a * X + B @ X
    return X.T if transposed else X


SCALE_MODES = ("spectral", "shape_scaling", "unit_rms_norm")


def update_scale(rows, cols, scale_coeff=0.2, mode="spectral"):
    """The factor on the Newton-Schulz output, fan_out = rows, fan_in = cols:
    spectral 0.2 * sqrt(max(m, n)) (§5.4 Eq. 4: max of the two dimensions, not
    fan_in), shape_scaling sqrt(max(1, m / n)), unit_rms_norm sqrt(m / n)
    (§14.6), times the free factor scale_coeff."""
    m, n = float(rows), float(cols)
    if mode == "spectral":
        f = math.sqrt(max(m, n))
    elif mode == "shape_scaling":
        f = math.sqrt(max(1.0, m / n))
    elif mode == "unit_rms_norm":
        f = math.sqrt(m / n)
    else:
        raise ValueError(mode)
    return scale_coeff * f


def apply_update(W, O, lr, weight_decay, scale_coeff=0.2, mode="spectral", scale_shape=None):
    """W_t = W_{t-1} (1 - lr lambda) - lr * scale * O, in fp64; the scale is
    that of `scale_shape` (the whole parameter) when given, else W's shape."""
    W = np.asarray(W, dtype=np.float64)
    R, C = scale_shape if scale_shape is not None else W.shape
    s = update_scale(R, C, scale_coeff, mode)
    return W * (1.0 - lr * weight_decay) - lr * s * np.asarray(O, dtype=np.float64)


def muon_step(W, g, m, *, lr, momentum, weight_decay=0.0, nesterov=True,
              ns_steps=5, coeffs=NS_COEFFS, eps=NS_EPS, scale_coeff=0.2, mode="spectral",
              split_rows=None, orthogonalize=True):
    """One Muon step for one 2-D matrix, everything in fp64.

    split_rows: row counts of blocks orthogonalised separately (QKV split);
    orthogonalize=False gives plain momentum SGD (W -= lr * scale_coeff *
    gtilde, no Newton-Schulz and no shape factor).
    Returns (W_new, m_new, O) where O is the (unscaled) direction.
    Inputs are not modified.
    """
    m_new, gt = momentum_update(m, g, momentum, nesterov)
    if not orthogonalize:
        W = np.asarray(W, dtype=np.float64)
        return W * (1.0 - lr * weight_decay) - lr * scale_coeff * gt, m_new, gt
    if split_rows:
        assert sum(split_rows) == gt.shape[0]
        edges = np.cumsum([0] + list(split_rows))
        O = np.concatenate([newton_schulz(gt[a:b], ns_steps, coeffs, eps) for a, b in zip(edges[:-1], edges[1:])])
    else:
        O = newton_schulz(gt, ns_steps, coeffs, eps)
    W_new = apply_update(W, O, lr, weight_decay, scale_coeff, mode, scale_shape=np.shape(W))
    return W_new, m_new, O


def polar_svd(G):
    """U V^T from the thin SVD G = U S V^T (the exact orthogonalisation that
    Newton-Schulz approximates, §5.1).  Sanity reference only."""
    U, _, Vt = np.linalg.svd(np.asarray(G, dtype=np.float64), full_matrices=False)
    return U @ Vt


def ns_flops(rows, cols, steps=5):
    """Multiply-add flops of the iteration as counted by the pages: for the
    wide orientation m <= n, 4 m^2 n + 2 m^3 per iteration."""
    m, n = sorted((int(rows), int(cols)))
    return steps * (4 * m * m * n + 2 * m ** 3)
