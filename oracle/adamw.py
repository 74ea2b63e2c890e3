"""AdamW oracle (test infrastructure only; see ``oracle/__init__``).

Definitions followed
--------------------
"02 · Optimizer：算法与 infra" §2 (Adam, Kingma & Ba Algorithm 1), per element,
step t = 1, 2, ...::

    m_t   = beta1 * m_{t-1} + (1 - beta1) * g_t
    v_t   = beta2 * v_{t-1} + (1 - beta2) * g_t^2
    mhat  = m_t / (1 - beta1^t)
    vhat  = v_t / (1 - beta2^t)
    update = mhat / (sqrt(vhat) + eps)            # eps OUTSIDE the sqrt

§3 (AdamW, decoupled weight decay, Loshchilov & Hutter Algorithm 2)::

    theta_t = theta_{t-1} - lr * (update + lambda * theta_{t-1})

written here as ``theta * (1 - lr*lambda) - lr * update`` (the decay acts on
theta_{t-1}).  The L2 variant of §3 instead feeds ``g + lambda*theta_{t-1}``
through the moments and applies no decoupled decay; it exists only for the
decay experiment of "优化器：AdamW、Muon 与分布式优化器" ("AdamW：解耦的权重衰减").

The model copy is the fp32 master rounded to bf16 (§9.2 "参数写回": fp32 ->
bf16 cast of the master after the step), round-to-nearest-even.

Readings where the pages are silent
-----------------------------------
* Precision: master weights, gradients and moments are fp32 (§9.1 "fp32
  master copy").  ``adamw_step_fp32`` evaluates each element in fp32 in the
  literal order of the formulas above, every operation rounded once (numpy
  never contracts a*b+c into an FMA).  ``adamw_step_fp64`` is the same
  formula in fp64.
* Step scalars: 1-beta1, 1-beta2, 1-beta1^t, 1-beta2^t and 1-lr*lambda are
  formed in fp64 from the fp32 hyper-parameters and rounded once to fp32
  (``step_scalars``).
* bf16: round to nearest, ties to even, on the fp32 bit pattern; overflow
  rounds to +-inf; subnormals are kept; every NaN becomes 0x7FC0.
"""

from __future__ import annotations

import numpy as np


# --------------------------------------------------------------------------
# bf16 round-to-nearest-even
# --------------------------------------------------------------------------

def bf16_rne(x) -> np.ndarray:
    """fp32 -> bf16 bit patterns (uint16), round to nearest, ties to even.

    The bf16 value keeps the top 16 bits of the fp32 pattern.  The discarded
    low 16 bits decide the rounding: above half-way rounds up, below rounds
    down, exactly half-way rounds to the candidate whose last kept bit is 0.
    Carrying out of the mantissa bumps the exponent, so the largest finite
    values round to infinity.  NaNs map to the quiet NaN 0x7FC0.
    """
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    hi = bits >> np.uint64(16)
    lo = bits & np.uint64(0xFFFF)
    half = np.uint64(0x8000)
    round_up = (lo > half) | ((lo == half) & ((hi & np.uint64(1)) == np.uint64(1)))
    out = hi + round_up.astype(np.uint64)
    is_nan = ((bits & np.uint64(0x7F800000)) == np.uint64(0x7F800000)) & \
             ((bits & np.uint64(0x007FFFFF)) != np.uint64(0))
    out = np.where(is_nan, np.uint64(0x7FC0), out)
    return (out & np.uint64(0xFFFF)).astype(np.uint16)


def bf16_to_f32(b) -> np.ndarray:
    """bf16 bit patterns -> fp32 values (exact: append 16 zero bits)."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


# --------------------------------------------------------------------------
# step scalars
# --------------------------------------------------------------------------

def step_scalars(lr, beta1, beta2, eps, weight_decay, t):
    """Per-step scalars in fp64 from the fp32 hyper-parameters, rounded to fp32.

    Returns a dict of np.float32: lr, beta1, beta2, eps, one_minus_beta1,
    one_minus_beta2, bias_c1 = 1 - beta1^t, bias_c2 = 1 - beta2^t and
    decay = 1 - lr*lambda (§2 bias correction; §3 decoupled decay factor).
    """
    if int(t) < 1:
        raise ValueError("Adam step t counts from 1")
    f = lambda x: np.float64(np.float32(x))          # the fp32 hyper-parameter, exactly
    lr64, b1, b2, wd = f(lr), f(beta1), f(beta2), f(weight_decay)
    return dict(
        lr=np.float32(lr64),
        beta1=np.float32(b1),
        beta2=np.float32(b2),
        eps=np.float32(f(eps)),
        one_minus_beta1=np.float32(1.0 - b1),
        one_minus_beta2=np.float32(1.0 - b2),
        bias_c1=np.float32(1.0 - b1 ** int(t)),
        bias_c2=np.float32(1.0 - b2 ** int(t)),
        decay=np.float32(1.0 - lr64 * wd),
    )


# --------------------------------------------------------------------------
# AdamW, fp32 (the pages' precision), literal order
# --------------------------------------------------------------------------

def adamw_step_fp32(p, g, m, v, *, lr, beta1, beta2, eps, weight_decay, t):
    """One AdamW step on fp32 arrays, in place; returns the bf16 model copy.

    p: fp32 master weights theta_{t-1} -> theta_t
    g: fp32 main_grad g_t (read only)
    m, v: fp32 first / second raw moments, updated in place
    """
    for a in (p, g, m, v):
        assert a.dtype == np.float32
    s = step_scalars(lr, beta1, beta2, eps, weight_decay, t)
    with np.errstate(all="ignore"):
        m[...] = s["beta1"] * m + s["one_minus_beta1"] * g
        v[...] = s["beta2"] * v + s["one_minus_beta2"] * (g * g)
        mhat = m / s["bias_c1"]
        vhat = v / s["bias_c2"]
        update = mhat / (np.sqrt(vhat) + s["eps"])
        p[...] = p * s["decay"] - s["lr"] * update
    return bf16_rne(p)


# --------------------------------------------------------------------------
# Adam(W), fp64
# --------------------------------------------------------------------------

def adamw_step_fp64(p, g, m, v, *, lr, beta1, beta2, eps, weight_decay, t, l2=False):
    """One step in fp64, in place.  ``l2=False``: AdamW (decoupled decay, §3
    Algorithm 2).  ``l2=True``: Adam with the decay folded into the gradient
    (g' = g + lambda*theta_{t-1}), no decoupled term."""
    for a in (p, m, v):
        assert a.dtype == np.float64
    if int(t) < 1:
        raise ValueError("Adam step t counts from 1")
    g = np.asarray(g, dtype=np.float64)
    if l2:
        g = g + weight_decay * p
    m[...] = beta1 * m + (1.0 - beta1) * g
    v[...] = beta2 * v + (1.0 - beta2) * g * g
    mhat = m / (1.0 - beta1 ** int(t))
    vhat = v / (1.0 - beta2 ** int(t))
    update = mhat / (np.sqrt(vhat) + eps)
    if l2:
        p[...] = p - lr * update
    else:
        p[...] = p - lr * (update + weight_decay * p)
