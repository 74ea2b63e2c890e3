"""CPU tests that pin the oracle to what the pages and the mathematics fix.

Each pin is run on the oracle (must pass) and on copies of it with a planted
mistake (must fail), so a plausible slip -- eps inside the sqrt, a missing bias
correction, coupled decay, a transposed operand, a wrong coefficient -- cannot
survive.  No GPU is used."""

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import adamw as OA
from oracle import muon as OM
import oracle_pins as P


# ---------------------------------------------------------------- AdamW ----

def test_adamw_fp64_pins():
    assert P.adamw_pin_failures(OA.adamw_step_fp64) == []


def _fp32_as_step64(p, g, m, v, *, lr, beta1, beta2, eps, weight_decay, t, l2=False):
    """Run the fp32 oracle on fp64 buffers (round in, compute, widen out)."""
    assert not l2
    p32, g32, m32, v32 = (np.asarray(x, dtype=np.float32).copy() for x in (p, g, m, v))
    OA.adamw_step_fp32(p32, g32, m32, v32, lr=lr, beta1=beta1, beta2=beta2, eps=eps,
                       weight_decay=weight_decay, t=t)
    p[...], m[...], v[...] = p32, m32, v32


def test_adamw_fp32_decay_experiment():
    """The printed decay experiment also holds for the fp32 oracle (the AdamW
    half; the pages' precision for master weights is fp32)."""
    gold = P.load_golden("adamw_decay_experiment.json")
    st = gold["setup"]
    p = np.ones(2, np.float32)
    m = np.zeros(2, np.float32)
    v = np.zeros(2, np.float32)
    for t in range(st["steps"]):
        g = (np.array(st["grad_scale"]) * (-1.0) ** t).astype(np.float32)
        OA.adamw_step_fp32(p, g, m, v, lr=st["lr"], beta1=st["beta1"], beta2=st["beta2"],
                           eps=st["eps"], weight_decay=st["weight_decay"], t=t + 1)
    assert [round(float(x), 3) for x in p] == gold["printed"]["adamw"]


def test_adamw_fp32_matches_fp64():
    """fp32 literal-order oracle agrees with the fp64 one to fp32 rounding."""
    rng = np.random.default_rng(1)
    n = 4099
    p32 = rng.standard_normal(n).astype(np.float32)
    m32 = np.zeros(n, np.float32)
    v32 = np.zeros(n, np.float32)
    p64, m64, v64 = p32.astype(np.float64), m32.astype(np.float64), v32.astype(np.float64)
    hp = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)
    for t in range(1, 21):
        g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
        OA.adamw_step_fp32(p32, g, m32, v32, t=t, **hp)
        h64 = {k: float(np.float32(x)) for k, x in hp.items()}
        OA.adamw_step_fp64(p64, g.astype(np.float64), m64, v64, t=t, **h64)
    for a, b in ((p32, p64), (m32, m64), (v32, v64)):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert rel < 1e-6


def test_step_scalars():
    s = OA.step_scalars(1e-3, 0.9, 0.999, 1e-8, 0.1, 1)
    assert s["bias_c1"] == np.float32(1.0 - np.float64(np.float32(0.9)))
    assert s["one_minus_beta1"] == s["bias_c1"]            # 1 - beta1^1
    assert s["decay"] == np.float32(1.0 - np.float64(np.float32(1e-3)) * np.float64(np.float32(0.1)))
    with pytest.raises(ValueError):
        OA.step_scalars(1e-3, 0.9, 0.999, 1e-8, 0.1, 0)


def test_fp32_first_step_closed_form_bits():
    """t = 1 in fp32: mhat = m/(1-beta1) recovers g to within one rounding of
    the product and the quotient, so theta_1 is within a few ulps of the
    closed form theta_0 (1 - lr lambda) - lr g/(|g| + eps)."""
    rng = np.random.default_rng(2)
    n = 1000
    p = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-2).astype(np.float32)
    p0 = p.astype(np.float64).copy()
    m = np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    OA.adamw_step_fp32(p, g, m, v, lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, t=1)
    g64 = g.astype(np.float64)
    want = p0 * (1 - 1e-3 * 0.01) - 1e-3 * g64 / (np.abs(g64) + 1e-8)
    assert np.max(np.abs(p - want)) < 4 * np.spacing(np.float32(4.0))


# --- planted mistakes: every one must be caught by some AdamW pin ---------

def _mutant(kind):
    """An fp64 Adam(W) step with one planted mistake."""
    if kind == "coupled_decay":                   # AdamW computed as Adam + L2
        def step(p, g, m, v, *, l2=False, **kw):
            return OA.adamw_step_fp64(p, g, m, v, l2=True, **kw)
        return step

    def step(p, g, m, v, *, lr, beta1, beta2, eps, weight_decay, t, l2=False):
        g = np.asarray(g, dtype=np.float64)
        if l2:
            g = g + weight_decay * p
        m[...] = beta1 * m + (1 - beta1) * g
        v[...] = beta2 * v + (1 - beta2) * g * g
        bc1, bc2 = 1 - beta1 ** t, 1 - beta2 ** t
        if kind == "no_bias_correction":
            bc1 = bc2 = 1.0
        if kind == "bias_t_plus_1":
            bc1, bc2 = 1 - beta1 ** (t + 1), 1 - beta2 ** (t + 1)
        mhat, vhat = m / bc1, v / bc2
        if kind == "eps_inside_sqrt":
            upd = mhat / np.sqrt(vhat + eps)
        else:
            upd = mhat / (np.sqrt(vhat) + eps)
        if l2:
            p[...] = p - lr * upd
        elif kind == "decay_without_lr":
            p[...] = p - lr * upd - weight_decay * p
        elif kind == "decay_after_update":
            p[...] = (p - lr * upd) * (1 - lr * weight_decay)
        else:
            p[...] = p - lr * (upd + weight_decay * p)
    return step


@pytest.mark.parametrize("kind", ["no_bias_correction", "bias_t_plus_1", "eps_inside_sqrt",
                                  "coupled_decay", "decay_without_lr", "decay_after_update"])
def test_adamw_pins_catch_planted_mistakes(kind):
    assert P.adamw_pin_failures(_mutant(kind)) != []


# ----------------------------------------------------------------- bf16 ----

def _structured_patterns():
    hi = np.arange(1 << 16, dtype=np.uint32) << np.uint32(16)
    lows = np.array([0, 1, 0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x1234, 0xC000], dtype=np.uint32)
    return (hi[:, None] | lows[None, :]).reshape(-1)


def test_bf16_rne_matches_torch_conversion():
    """The library routine torch.Tensor.to(bfloat16) on the CPU rounds to
    nearest-even; on every exponent, sign and rounding case (below, at and
    above half-way, with odd and even kept bits) the oracle agrees, NaNs
    aside (checked separately)."""
    bits = _structured_patterns()
    x = bits.view(np.float32)
    ours = OA.bf16_rne(x)
    ref = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.all(ours[nan] == 0x7FC0)


def test_bf16_rne_special_values():
    cases = {
        0x3F800000: 0x3F80,   # 1.0 exact
        0x3F808000: 0x3F80,   # tie, kept bit even -> down
        0x3F818000: 0x3F82,   # tie, kept bit odd -> up
        0x3F808001: 0x3F81,   # just above half
        0x3F807FFF: 0x3F80,   # just below half
        0x7F7FFFFF: 0x7F80,   # largest finite rounds to +inf
        0xFF7FFFFF: 0xFF80,   # and to -inf
        0x7F800000: 0x7F80,   # +inf
        0x80000000: 0x8000,   # -0
        0x00000001: 0x0000,   # tiniest subnormal rounds to +0
        0x00008000: 0x0000,   # subnormal tie to even (0)
        0x00018000: 0x0002,   # subnormal tie to even (up)
        0x007FFFFF: 0x0080,   # largest subnormal carries into the exponent
        0x7FC00000: 0x7FC0,   # qNaN
        0xFFC00001: 0x7FC0,   # negative NaN: canonical
        0x7F800001: 0x7FC0,   # sNaN: canonical
    }
    x = np.array(list(cases), dtype=np.uint32).view(np.float32)
    got = OA.bf16_rne(x)
    assert [int(v) for v in got] == list(cases.values())
    # bf16 -> fp32 -> bf16 is the identity on non-NaN patterns
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = OA.bf16_to_f32(b)
    keep = ~np.isnan(f)
    assert np.array_equal(OA.bf16_rne(f)[keep], b[keep])


# ------------------------------------------------------------ Newton-Schulz --

def test_ns_pins():
    assert P.ns_pin_failures(OM.newton_schulz) == []


def _ns_mutant(kind):
    def ns(G, steps=5):
        a, b, c = OM.NS_COEFFS
        if kind == "coeffs_rotated":
            a, b, c = b, c, a
        X = np.asarray(G, dtype=np.float64)
        X = X / (np.linalg.norm(X) + 1e-7) if kind != "spectral_norm" else X / np.linalg.norm(X, 2)
        tr = X.shape[0] > X.shape[1] and kind != "no_transpose"
        if tr:
            X = X.T
        for _ in range(steps):
            A = X @ X.T
            B = b * A + c * (A if kind == "quintic_as_cubic" else A @ A)
            X = a * X + (X @ B if kind == "bx_swapped" else B @ X)
        return X.T if tr and kind != "forget_transpose_back" else X
    return ns


@pytest.mark.parametrize("kind", ["coeffs_rotated", "spectral_norm", "quintic_as_cubic",
                                  "bx_swapped", "forget_transpose_back"])
def test_ns_pins_catch_planted_mistakes(kind):
    try:
        fails = P.ns_pin_failures(_ns_mutant(kind))
    except ValueError:          # a shape mismatch is a caught mistake too
        fails = ["shape error"]
    assert fails != []


def test_ns_flop_formula():
    """4 m^2 n + 2 m^3 per iteration for m <= n ("优化器：AdamW、Muon 与分布式
    优化器", Newton-Schulz cost note); the exercise quotes 4.1e11 for a 4096^2
    matrix per iteration."""
    assert OM.ns_flops(4096, 4096, 1) == 6 * 4096 ** 3
    assert f"{OM.ns_flops(4096, 4096, 1):.1e}" == "4.1e+11"
    assert OM.ns_flops(1024, 4096, 5) == OM.ns_flops(4096, 1024, 5)


# ------------------------------------------------------------------- Muon ----

def test_momentum_forms_agree():
    """The EMA/lerp form ("02 · Optimizer：算法与 infra" §1) and the sum form
    of "优化器：AdamW、Muon 与分布式优化器" (M <- mu M + G, update NS(G + mu M))
    feed Newton-Schulz with inputs that differ by the factor (1 - mu), which
    the normalisation removes: the outputs agree up to the eps term."""
    rng = np.random.default_rng(4)
    mu = 0.95
    m_lerp = np.zeros((24, 40))
    M_sum = np.zeros((24, 40))
    for _ in range(6):
        g = rng.standard_normal((24, 40))
        m_lerp, gt = OM.momentum_update(m_lerp, g, mu, nesterov=True)
        M_sum = mu * M_sum + g
        assert np.allclose(gt, (1 - mu) * (g + mu * M_sum), rtol=1e-12, atol=1e-14)
        O1 = OM.newton_schulz(gt)
        O2 = OM.newton_schulz(g + mu * M_sum)
        assert np.linalg.norm(O1 - O2) / np.linalg.norm(O2) < 1e-6
    # plain momentum (no Nesterov) returns the buffer itself
    m2, gt2 = OM.momentum_update(np.ones(3), np.zeros(3), 0.9, nesterov=False)
    assert np.allclose(m2, 0.9) and np.allclose(gt2, m2)


def test_update_rms_lemma():
    """A full-rank semi-orthogonal A x B matrix has RMS 1/sqrt(max(A, B))
    ("02 · Optimizer：算法与 infra" §5.4 Lemma 1), so the scaled update of
    Eq. 4 has RMS 0.2 * lr exactly when O = U V^T."""
    rng = np.random.default_rng(8)
    for shape in ((32, 96), (96, 32), (50, 50)):
        O = OM.polar_svd(rng.standard_normal(shape))
        assert abs(np.sqrt(np.mean(O ** 2)) - 1 / math.sqrt(max(shape))) < 1e-12
        W = rng.standard_normal(shape)
        Wn = OM.apply_update(W, O, lr=0.02, weight_decay=0.0)
        assert abs(np.sqrt(np.mean((Wn - W) ** 2)) - 0.2 * 0.02) < 1e-12


def test_decoupled_decay_in_muon_update():
    """Eq. 3: W_t = W_{t-1} - lr (scaled O + lambda W_{t-1})."""
    rng = np.random.default_rng(9)
    W = rng.standard_normal((8, 12))
    O = rng.standard_normal((8, 12))
    Wn = OM.apply_update(W, O, lr=0.1, weight_decay=0.3)
    assert np.allclose(Wn, W - 0.1 * (0.2 * math.sqrt(12) * O + 0.3 * W), rtol=1e-14)


def test_ns_vs_svd_polar():
    """Five quintic steps keep the singular vectors of U V^T (§5.2) but not
    unit singular values: on a well-conditioned input every singular value
    lands in the printed band and the distance to U V^T is the spectral
    residual alone."""
    rng = np.random.default_rng(10)
    G = rng.standard_normal((64, 160))
    X = OM.newton_schulz(G)
    P_ = OM.polar_svd(G)
    U, S, Vt = np.linalg.svd(G, full_matrices=False)
    s_ns = np.linalg.svd(X, compute_uv=False)
    phi = P.phi_iterate(S / (np.linalg.norm(G) + 1e-7), 5)
    assert np.allclose(np.sort(s_ns), np.sort(phi), rtol=1e-9)
    assert np.allclose(X, (U * phi) @ Vt, atol=1e-10)
    assert np.linalg.norm(X - P_) / np.linalg.norm(P_) < 0.35
    assert 0.6 < s_ns.min() and s_ns.max() < 1.3


def test_muon_step_composes():
    """muon_step = momentum -> Newton-Schulz -> scaled decoupled update."""
    rng = np.random.default_rng(12)
    W = rng.standard_normal((40, 24)) * 0.02
    g = rng.standard_normal((40, 24)) * 1e-2
    m = rng.standard_normal((40, 24)) * 1e-2
    Wn, mn, O = OM.muon_step(W, g, m, lr=0.02, momentum=0.95, weight_decay=0.1)
    m_want = m + 0.05 * (g - m)
    gt = g + 0.95 * (m_want - g)
    assert np.allclose(mn, m_want, rtol=1e-14)
    assert np.allclose(O, OM.newton_schulz(gt), rtol=1e-12)
    assert np.allclose(Wn, W * (1 - 0.002) - 0.02 * 0.2 * math.sqrt(40) * O, rtol=1e-13)


def test_oracle_header_says_test_infrastructure():
    assert "TEST INFRASTRUCTURE ONLY" in oracle.__doc__


# ------------------------------------------------------------- clipping ----

from oracle import clip as OC  # noqa: E402


def _clip_pin_failures(total_norm, clip_scale):
    """Pins of the clipping definition ("02 · Optimizer：算法与 infra" §11.1):
    a 3-4-5 triangle, a norm below the threshold, a disabled clip, and the
    post-clip norm landing on max_norm up to the 1e-6 guard."""
    fails = []
    g = [np.array([3.0]), np.array([[4.0]])]           # two tensors: the norm is global
    if abs(total_norm(g) - 5.0) > 1e-15:
        fails.append("3-4-5 norm")
    if abs(clip_scale(g, 1.0) - 1.0 / (5.0 + 1e-6)) > 1e-15:
        fails.append("coefficient")
    if clip_scale(g, 10.0) != 1.0:
        fails.append("below threshold must not scale")
    if clip_scale(g, 0.0) != 1.0 or clip_scale(g, -1.0) != 1.0:
        fails.append("max_norm <= 0 disables")
    rng = np.random.default_rng(0)
    gs = [rng.standard_normal(s) for s in ((7,), (3, 5), (11, 2))]
    s = clip_scale(gs, 0.5)
    clipped = total_norm([x * s for x in gs])
    if not (0.5 - 1e-5 < clipped <= 0.5):
        fails.append(f"post-clip norm {clipped}")
    # the coefficient is the same for every tensor (global, not per-tensor)
    per = [clip_scale([x], 0.5) for x in gs]
    if all(abs(p - s) < 1e-12 for p in per):
        fails.append("per-tensor norm")
    return fails


def test_clip_pins():
    assert _clip_pin_failures(OC.total_norm, OC.clip_scale) == []


@pytest.mark.parametrize("kind", ["no_sqrt", "per_tensor", "always_scale", "eps_missing_sign"])
def test_clip_pins_catch_planted_mistakes(kind):
    def tn(grads):
        s = sum(float(np.sum(np.asarray(g, np.float64) ** 2)) for g in grads)
        return s if kind == "no_sqrt" else float(np.sqrt(s))

    def cs(grads, max_norm):
        if max_norm <= 0:
            return 1.0
        if kind == "per_tensor":
            return max_norm / (tn(grads[:1]) + 1e-6)
        coeff = max_norm / (tn(grads) + (-1e-6 if kind == "eps_missing_sign" else 1e-6))
        return coeff if (coeff < 1.0 or kind == "always_scale") else 1.0
    assert _clip_pin_failures(tn, cs) != []


# ------------------------------------------------------- Muon variants ----

def test_scale_modes_follow_the_printed_formulas():
    """§14.6 of "02 · Optimizer：算法与 infra": spectral = max(m,n)**0.5,
    shape_scaling = max(1, m/n)**0.5, unit_rms_norm = (m/n)**0.5, with
    m = fan_out (rows) and n = fan_in (cols)."""
    for (m, n), want in {(4096, 1024): (64.0, 2.0, 2.0), (1024, 4096): (64.0, 1.0, 0.5),
                         (14336, 4096): (math.sqrt(14336), math.sqrt(3.5), math.sqrt(3.5))}.items():
        got = tuple(OM.update_scale(m, n, 1.0, mode) for mode in OM.SCALE_MODES)
        assert np.allclose(got, want, rtol=1e-15)
    assert OM.update_scale(256, 512, 0.2) == 0.2 * math.sqrt(512)


def test_coefficient_schedule_is_composition_of_quintics():
    """With a different (a, b, c) in each iteration, every singular value goes
    through the composition of the per-iteration quintics (§5.2's
    per-singular-value argument does not need equal coefficients); a schedule
    of identical triples equals the single triple."""
    rng = np.random.default_rng(13)
    U = P.random_orthonormal(rng, 30, 30)
    V = P.random_orthonormal(rng, 50, 30)
    S = np.linspace(0.05, 1.0, 30)
    G = (U * S) @ V.T
    sched = [(3.4445, -4.7750, 2.0315), (3.0, -3.2, 1.2), (2.5, -2.0, 0.5), (1.875, -1.25, 0.375)]
    s = S / (np.linalg.norm(S) + 1e-7)
    for a, b, c in sched:
        s = a * s + b * s ** 3 + c * s ** 5
    assert np.allclose(OM.newton_schulz(G, 4, sched), (U * s) @ V.T, atol=1e-12)
    assert np.array_equal(OM.newton_schulz(G, 3, [P.COEFFS] * 3), OM.newton_schulz(G, 3))


def test_split_blocks_are_orthogonalised_separately():
    """QKV split (§5.5, §14.4): each row block is orthogonalised on its own, so
    the split result differs from the whole-matrix result but each block
    equals Newton-Schulz of that block; the scale uses the full shape."""
    rng = np.random.default_rng(14)
    W = rng.standard_normal((48, 32)) * 0.02
    g = rng.standard_normal((48, 32)) * 1e-2
    m = np.zeros((48, 32))
    Wn, _, O = OM.muon_step(W, g, m, lr=0.02, momentum=0.95, split_rows=[16, 16, 16])
    gt = OM.momentum_update(m, g, 0.95)[1]
    for a in (0, 16, 32):
        assert np.allclose(O[a:a + 16], OM.newton_schulz(gt[a:a + 16]), atol=1e-13)
    assert np.allclose(Wn, W - 0.02 * 0.2 * math.sqrt(48) * O, atol=1e-15)
    whole = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)[2]
    assert np.linalg.norm(whole - O) > 1e-3


def test_plain_momentum_sgd():
    """Without orthogonalisation the step is theta -= lr * gtilde (§1)."""
    W = np.ones((3, 4))
    g = np.full((3, 4), 2.0)
    m = np.zeros((3, 4))
    Wn, mn, _ = OM.muon_step(W, g, m, lr=0.1, momentum=0.5, orthogonalize=False, scale_coeff=1.0)
    # m = 0.5 * 2 = 1; gtilde = lerp(2, 1, 0.5) = 1.5
    assert np.allclose(mn, 1.0) and np.allclose(Wn, 1 - 0.1 * 1.5)


@pytest.mark.parametrize("sizes", [[3, 2], [2, 2, 1], [1, 2, 2], [5], [2, 3]])
@pytest.mark.parametrize("shape", [(64, 200), (200, 64), (96, 96)])
def test_grouped_iterations_are_exact_algebra(sizes, shape):
    """The grouped evaluation of the Newton-Schulz iterations (reading R20 of
    the design): within a group every C_k = a I + b A_k + c A_k^2 is a
    polynomial in the group's first Gram matrix, so A_{k+1} = C_k (A_k C_k)
    and X_{k0+g} = (C_{k0+g-1} ... C_k0) X_k0.  In fp64 that equals the
    iteration as printed ("优化器：AdamW、Muon 与分布式优化器", newton_schulz)
    to rounding, for every split of the five iterations and for a
    coefficient schedule."""
    rng = np.random.default_rng(sum(sizes) * 1000 + shape[0])
    G = rng.standard_normal(shape)
    for coeffs in (OM.NS_COEFFS, [(3.4445, -4.775, 2.0315), (3.2, -4.4, 1.9), (3.0, -4.0, 1.7),
                                  (2.8, -3.6, 1.55), (2.2, -2.1, 0.9)]):
        sched = [tuple(coeffs)] * 5 if np.isscalar(coeffs[0]) else list(coeffs)
        X = G / (np.linalg.norm(G) + 1e-7)
        tr = shape[0] > shape[1]
        if tr:
            X = X.T
        I = np.eye(X.shape[0])
        k = 0
        for g in sizes:
            A = X @ X.T
            a, b, c = sched[k]
            C = a * I + b * A + c * (A @ A)
            M = C
            for j in range(1, g):
                A = C @ (A @ C)
                a, b, c = sched[k + j]
                C = a * I + b * A + c * (A @ A)
                M = C @ M
            X = M @ X
            k += g
        got = X.T if tr else X
        want = OM.newton_schulz(G, 5, coeffs)
        assert np.abs(got - want).max() <= 1e-10 * np.abs(want).max()
