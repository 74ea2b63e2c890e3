"""Pin checks for the oracle, written as functions of the step routine they
check, so that the same check runs on the oracle (must pass) and on copies of
it with a planted mistake (must fail).  Each check cites the passage whose
printed value, closed form or special case it uses."""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


# --------------------------------------------------------------------------
# AdamW pins.  ``step64(p, g, m, v, *, lr, beta1, beta2, eps, weight_decay,
# t, l2)`` is an fp64 Adam(W) step, in place.
# --------------------------------------------------------------------------

def decay_experiment(step64):
    """The adamw_decay.py experiment of "优化器：AdamW、Muon 与分布式优化器"
    ("AdamW：解耦的权重衰减"): two weights, alternating-sign gradients of
    scale 0.01 and 10, lr 1e-2, wd 0.1, 1000 steps.  Returns the final
    weights for (Adam + L2, AdamW) and the failures against the print."""
    gold = load_golden("adamw_decay_experiment.json")
    st = gold["setup"]
    res = {}
    for name, l2 in (("adam_l2", True), ("adamw", False)):
        p = np.array(st["w0"], dtype=np.float64)
        m = np.zeros(2)
        v = np.zeros(2)
        scale = np.array(st["grad_scale"], dtype=np.float64)
        for t in range(st["steps"]):
            g = scale * (-1.0) ** t
            step64(p, g, m, v, lr=st["lr"], beta1=st["beta1"], beta2=st["beta2"],
                   eps=st["eps"], weight_decay=st["weight_decay"], t=t + 1, l2=l2)
        res[name] = p.copy()
    fails = []
    nd = gold["printed_decimals"]
    for name in ("adam_l2", "adamw"):
        got = [round(float(x), nd) + 0.0 for x in res[name]]
        if got != gold["printed"][name]:
            fails.append(f"{name}: got {got}, printed {gold['printed'][name]}")
    closed = (1 - st["lr"] * st["weight_decay"]) ** st["steps"]
    if round(closed, nd) != gold["printed"]["decay_only_closed_form"]:
        fails.append("closed form")
    return res, fails


def zero_grad_decay(step64):
    """g = 0 for every step: m = v = 0, the Adam term is 0/(0+eps) = 0 and
    only the decoupled decay acts, so theta_t = theta_0 (1 - lr lambda)^t
    exactly ("02 · Optimizer：算法与 infra" §3, Algorithm 2)."""
    rng = np.random.default_rng(7)
    p0 = rng.standard_normal(64)
    p = p0.copy()
    m = np.zeros(64)
    v = np.zeros(64)
    lr, wd, T = 3e-3, 0.05, 200
    for t in range(1, T + 1):
        step64(p, np.zeros(64), m, v, lr=lr, beta1=0.9, beta2=0.999, eps=1e-8,
               weight_decay=wd, t=t, l2=False)
    want = p0 * (1 - lr * wd) ** T
    err = np.max(np.abs(p - want) / np.abs(want))
    return [] if err < 1e-12 else [f"zero-grad decay rel err {err:.3g}"]


def first_step_closed_form(step64):
    """At t = 1 with zero initial moments, bias correction gives
    mhat = g and vhat = g^2 exactly, so theta_1 = theta_0 (1 - lr lambda)
    - lr g / (|g| + eps), m_1 = (1-beta1) g and v_1 = (1-beta2) g^2
    ("02 · Optimizer：算法与 infra" §2, the bias-correction definitions)."""
    rng = np.random.default_rng(11)
    n = 257
    p0 = rng.standard_normal(n)
    g = rng.standard_normal(n) * np.exp(rng.uniform(-12, 2, n))
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.999, 1e-8, 0.01
    p, m, v = p0.copy(), np.zeros(n), np.zeros(n)
    step64(p, g, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=wd, t=1, l2=False)
    fails = []
    want_p = p0 * (1 - lr * wd) - lr * g / (np.abs(g) + eps)
    if not np.allclose(p, want_p, rtol=1e-12, atol=1e-15):
        fails.append("theta_1")
    if not np.allclose(m, (1 - b1) * g, rtol=1e-14, atol=0):
        fails.append("m_1")
    if not np.allclose(v, (1 - b2) * g * g, rtol=1e-14, atol=0):
        fails.append("v_1")
    return fails


def constant_grad_closed_form(step64):
    """Constant gradient c from zero moments: m_t = c (1 - beta1^t) and
    v_t = c^2 (1 - beta2^t), so the bias-corrected moments are exactly c and
    c^2 at every t; with lambda = 0, theta_t = theta_0 - t lr c / (|c| + eps)
    ("02 · Optimizer：算法与 infra" §2: bias correction removes the zero-init
    bias at every step)."""
    c = np.array([3e-4, -2.5, 1e-7, 40.0])
    lr, b1, b2, eps, T = 1e-2, 0.9, 0.999, 1e-8, 50
    p0 = np.array([0.5, -1.0, 2.0, 0.0])
    p, m, v = p0.copy(), np.zeros(4), np.zeros(4)
    for t in range(1, T + 1):
        step64(p, c, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, t=t, l2=False)
    want = p0 - T * lr * c / (np.abs(c) + eps)
    fails = []
    if not np.allclose(p, want, rtol=1e-10, atol=1e-12):
        fails.append("theta_T")
    if not np.allclose(m, c * (1 - b1 ** T), rtol=1e-12, atol=0):
        fails.append("m_T")
    if not np.allclose(v, c * c * (1 - b2 ** T), rtol=1e-12, atol=0):
        fails.append("v_T")
    return fails


def late_step_no_bias(step64):
    """For large t, beta^t -> 0 and mhat -> m (§2): at t = 10^6 the step
    equals the uncorrected update theta - lr m / (sqrt(v) + eps)."""
    rng = np.random.default_rng(3)
    n = 100
    p0 = rng.standard_normal(n)
    g = rng.standard_normal(n) * 1e-3
    m0 = rng.standard_normal(n) * 1e-3
    v0 = rng.uniform(0, 1e-6, n)
    lr, b1, b2, eps = 1e-3, 0.9, 0.999, 1e-8
    p, m, v = p0.copy(), m0.copy(), v0.copy()
    step64(p, g, m, v, lr=lr, beta1=b1, beta2=b2, eps=eps, weight_decay=0.0, t=10 ** 6, l2=False)
    m1 = b1 * m0 + (1 - b1) * g
    v1 = b2 * v0 + (1 - b2) * g * g
    want = p0 - lr * m1 / (np.sqrt(v1) + eps)
    return [] if np.allclose(p, want, rtol=1e-12, atol=1e-15) else ["late step"]


def adamw_pin_failures(step64):
    fails = []
    fails += decay_experiment(step64)[1]
    fails += zero_grad_decay(step64)
    fails += first_step_closed_form(step64)
    fails += constant_grad_closed_form(step64)
    fails += late_step_no_bias(step64)
    return fails


# --------------------------------------------------------------------------
# Newton-Schulz / Muon pins.  ``ns(G, steps)`` is a Newton-Schulz routine.
# --------------------------------------------------------------------------

COEFFS = (3.4445, -4.7750, 2.0315)


def phi_iterate(s, steps, coeffs=COEFFS):
    """The scalar quintic phi(s) = a s + b s^3 + c s^5 applied ``steps``
    times ("02 · Optimizer：算法与 infra" §5.2: with X = U S V^T every
    iteration applies the same odd polynomial to each singular value)."""
    a, b, c = coeffs
    s = np.asarray(s, dtype=np.float64)
    for _ in range(steps):
        s = a * s + b * s ** 3 + c * s ** 5
    return s


def random_orthonormal(rng, n, k):
    q, r = np.linalg.qr(rng.standard_normal((n, k)))
    return q * np.sign(np.diag(r))


def spectral_form(ns, shape, steps, seed):
    """NS(U S V^T) = U phi^k(S / (||S||_2 + eps)) V^T for arbitrary
    orthonormal U, V (§5.2), on a non-symmetric input of the given shape.
    Checks a wide, a tall and a square case with distinct singular values."""
    R, C = shape
    k = min(R, C)
    rng = np.random.default_rng(seed)
    U = random_orthonormal(rng, R, k)
    V = random_orthonormal(rng, C, k)
    S = np.sort(rng.uniform(0.05, 3.0, k))[::-1]
    G = (U * S) @ V.T
    X = ns(G, steps)
    want = (U * phi_iterate(S / (np.sqrt(np.sum(S * S)) + 1e-7), steps)) @ V.T
    err = np.linalg.norm(X - want) / np.linalg.norm(want)
    return [] if err < 1e-10 else [f"spectral form {shape} err {err:.3g}"]


def orthogonalize_print(ns):
    """orthogonalize.py of "优化器：AdamW、Muon 与分布式优化器": a 256 x 1024
    input with spectrum logspace(0, -2, 256); the printed singular-value
    ranges, in-band fractions, energy and RMS figures."""
    gold = load_golden("ns_orthogonalize_spectrum.json")
    pr = gold["printed"]
    rng = np.random.default_rng(0)
    U = random_orthonormal(rng, 256, 256)
    V = random_orthonormal(rng, 1024, 256)
    S = np.logspace(0, -2, 256)
    G = (U * S) @ V.T
    fails = []
    lo, hi = gold["setup"]["band_open_interval"]
    for k in (1, 3, 5):
        s = np.linalg.svd(ns(G, k), compute_uv=False)
        want = pr[f"steps_{k}"]
        got = (f"{s.min():.2f}", f"{s.max():.2f}", f"{np.mean((s > lo) & (s < hi)):.0%}")
        printed = (f"{want['sv_min']:.2f}", f"{want['sv_max']:.2f}", f"{want['frac_in_band_percent']}%")
        if got != printed:
            fails.append(f"k={k}: {got} vs printed {printed}")
    X = ns(G, 5)
    before = float(np.sum(S[:8] ** 2) / np.sum(S ** 2))
    after = float(np.linalg.norm(X @ V[:, :8]) ** 2 / np.linalg.norm(X) ** 2)
    # the script prints these with the formats :.0%, :.1%, :.4f and :.2f
    if f"{before:.0%}" != f"{pr['top8_energy_before_percent']}%":
        fails.append(f"top-8 energy before {before:.4f}")
    if f"{after:.1%}" != f"{pr['top8_energy_after_percent']}%":
        fails.append(f"top-8 energy after {after:.4f}")
    rms = float(np.sqrt(np.mean(X ** 2)))
    if f"{rms:.4f}" != f"{pr['rms_after_ns']:.4f}":
        fails.append(f"rms {rms:.5f}")
    if f"{rms * 0.2 * math.sqrt(1024):.2f}" != f"{pr['rms_after_scaling_0p2_sqrt_1024']:.2f}":
        fails.append("scaled rms")
    if f"{1024 ** -0.5:.4f}" != f"{pr['rms_reference_one_over_sqrt_1024']:.4f}":
        fails.append("reference rms")
    return fails


def rank_one(ns):
    """A rank-one input u v^T has one singular value ||u|| ||v|| = ||G||_F, so
    the normalised input has sigma = 1/(1 + eps/||G||_F) and the output is
    phi^5(sigma) u v^T / (||u|| ||v||) (§5.2)."""
    rng = np.random.default_rng(5)
    u = rng.standard_normal(40)
    v = rng.standard_normal(24)
    G = np.outer(u, v)
    nf = np.linalg.norm(u) * np.linalg.norm(v)
    want = phi_iterate(nf / (nf + 1e-7), 5) * G / nf
    X = ns(G, 5)
    err = np.linalg.norm(X - want) / np.linalg.norm(want)
    return [] if err < 1e-10 else [f"rank one err {err:.3g}"]


def ns_pin_failures(ns):
    fails = []
    fails += spectral_form(ns, (48, 80), 5, 1)
    fails += spectral_form(ns, (80, 48), 5, 2)
    fails += spectral_form(ns, (32, 32), 3, 3)
    fails += rank_one(ns)
    fails += orthogonalize_print(ns)
    return fails
