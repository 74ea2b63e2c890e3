"""AdamW parity on the GPU, through the C ABI: the kernel must be bit-exact
against the fp32 oracle (same literal operation order, each operation rounded
once), and the bf16 model copy bit-exact against the oracle's
round-to-nearest-even of the GPU's own master weights."""

import numpy as np
import pytest

from gpu_helpers import (AdamwState, assert_bits_equal, bf16_host, dev, host, require_gpu, torch)
import mixed_precision_optimizer_gb300 as mp
from oracle import adamw as OA
import synthetic as S

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.1)


def oracle_step(st: AdamwState, t, hp=HP):
    return OA.adamw_step_fp32(st.h["p"], st.h["g"], st.h["m"], st.h["v"], t=t, **hp)


def check(st: AdamwState, what):
    for k in ("p", "m", "v"):
        assert_bits_equal(host(st.d[k]), st.h[k], f"{what}.{k}")
    if st.model is not None:
        got = bf16_host(st.model)
        assert np.array_equal(got, OA.bf16_rne(host(st.d["p"]))), f"{what}: bf16 vs GPU master"
        assert np.array_equal(got, OA.bf16_rne(st.h["p"])), f"{what}: bf16 vs oracle master"


def random_state(rng, n, with_model=True):
    p = rng.standard_normal(n).astype(np.float32)
    g = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    v = rng.uniform(0, 1e-6, n).astype(np.float32)
    return AdamwState(p, g, m, v, with_model)


RAGGED = [1, 2, 3, 7, 8, 9, 15, 16, 17, 127, 1000, 16383, 16384, 16385, 3 * 16384 + 5, 100003]


def test_ragged_sizes_multi_tensor_bit_exact():
    rng = np.random.default_rng(100)
    states = [random_state(rng, n, with_model=(i % 3 != 2)) for i, n in enumerate(RAGGED)]
    for t in (1, 2, 3, 10):
        for st in states:
            st.h["g"][...] = (rng.standard_normal(st.h["g"].size) * 1e-3).astype(np.float32)
            st.d["g"].copy_(dev(st.h["g"]))
        mp.adamw_step([s.param() for s in states], mp.adamw_hp(step=t, **HP))
        for st in states:
            oracle_step(st, t)
        torch.cuda.synchronize()
        for i, st in enumerate(states):
            check(st, f"t={t} n={RAGGED[i]}")


def test_zero_size_and_empty_list():
    rng = np.random.default_rng(1)
    st = random_state(rng, 33)
    z = torch.zeros(0, device="cuda")
    empty = mp.Param(z, z, z, z, torch.zeros(0, dtype=torch.bfloat16, device="cuda"))
    mp.adamw_step([empty, st.param(), empty], mp.adamw_hp(step=1, **HP))
    mp.adamw_step([], mp.adamw_hp(step=1, **HP))
    oracle_step(st, 1)
    torch.cuda.synchronize()
    check(st, "with empty")


def _views(buf_len, offs, n):
    """Device views of length n at element offsets offs = (p, g, m, v, model)."""
    rng = np.random.default_rng(sum(offs) + n)
    base = {
        "p": rng.standard_normal(buf_len).astype(np.float32),
        "g": (rng.standard_normal(buf_len) * 1e-3).astype(np.float32),
        "m": (rng.standard_normal(buf_len) * 1e-3).astype(np.float32),
        "v": rng.uniform(0, 1e-6, buf_len).astype(np.float32),
    }
    dbase = {k: dev(a) for k, a in base.items()}
    model_buf = torch.zeros(buf_len, dtype=torch.bfloat16, device="cuda")
    keys = ("p", "g", "m", "v")
    d = {k: dbase[k][o:o + n] for k, o in zip(keys, offs[:4])}
    h = {k: base[k][o:o + n].copy() for k, o in zip(keys, offs[:4])}
    model = model_buf[offs[4]:offs[4] + n]
    return d, h, model, dbase, model_buf


@pytest.mark.parametrize("offs", [(1, 1, 1, 1, 1), (3, 3, 3, 3, 3), (2, 2, 2, 2, 6), (0, 1, 2, 3, 0),
                                  (5, 5, 5, 5, 2), (4, 4, 4, 4, 4)])
@pytest.mark.parametrize("n", [5, 40000])
def test_unaligned_views(offs, n):
    """Views at element offsets: equal offsets (mod 4 for fp32, consistent
    with the bf16 offset mod 8) take the peeled-head vector path; the rest
    take the element-at-a-time path.  Both must match the oracle and leave
    the memory around the view untouched."""
    d, h, model, dbase, model_buf = _views(n + 16, offs, n)
    before = {k: host(v).copy() for k, v in dbase.items()}
    mb_before = bf16_host(model_buf).copy()
    p = mp.Param(d["p"], d["g"], d["m"], d["v"], model)
    mp.adamw_step([p], mp.adamw_hp(step=3, **HP))
    OA.adamw_step_fp32(h["p"], h["g"], h["m"], h["v"], t=3, **HP)
    torch.cuda.synchronize()
    for k in ("p", "m", "v"):
        assert_bits_equal(host(d[k]), h[k], k)
    assert np.array_equal(bf16_host(model), OA.bf16_rne(h["p"]))
    # outside the views nothing changed
    for k, o in zip(("p", "g", "m", "v"), offs[:4]):
        after = host(dbase[k])
        mask = np.ones(after.size, bool)
        mask[o:o + n] = False
        assert np.array_equal(after[mask], before[k][mask]), k
    mb = bf16_host(model_buf)
    mask = np.ones(mb.size, bool)
    mask[offs[4]:offs[4] + n] = False
    assert np.array_equal(mb[mask], mb_before[mask])


def test_more_tensors_than_one_launch():
    """Lists longer than one launch's parameter-space table (400 tensors)."""
    rng = np.random.default_rng(5)
    sizes = rng.integers(1, 3000, 1001)
    states = [random_state(rng, int(n), with_model=bool(i % 2)) for i, n in enumerate(sizes)]
    mp.adamw_step([s.param() for s in states], mp.adamw_hp(step=7, **HP))
    for st in states:
        oracle_step(st, 7)
    torch.cuda.synchronize()
    for i, st in enumerate(states):
        check(st, f"tensor {i}")


def test_special_values():
    vals = np.array([0.0, -0.0, 1e-45, -1e-40, 1.17549435e-38, 3.4e38, -3.4e38, np.inf, -np.inf, np.nan,
                     1.0, -1.0, 65504.0, 1e-8, 2.0 ** -126, 2.0 ** -149], dtype=np.float32)
    n = vals.size
    grid = np.stack(np.meshgrid(np.arange(n), np.arange(n), indexing="ij"), -1).reshape(-1, 2)
    p = vals[grid[:, 0]]
    g = vals[grid[:, 1]]
    m = np.resize(vals[::-1], p.size).astype(np.float32)
    v = np.abs(np.resize(vals, p.size)).astype(np.float32)
    st = AdamwState(p, g, m, v)
    for hp in (HP, dict(HP, weight_decay=0.0), dict(lr=0.5, beta1=0.0, beta2=0.0, eps=0.0, weight_decay=1.0)):
        mp.adamw_step([st.param()], mp.adamw_hp(step=2, **hp))
        OA.adamw_step_fp32(st.h["p"], st.h["g"], st.h["m"], st.h["v"], t=2, **hp)
        torch.cuda.synchronize()
        check(st, f"special {hp}")


def test_tiny_mixed_adamw_vector_10_steps():
    """The 512-element AdamW vector of the tiny mixed workload: init ones,
    N(0, 1e-2) gradients, lr 1e-3, wd 0.01, 10 steps, bit-exact every step."""
    w = S.tiny_mixed()
    spec = w.tensors[1]
    st = AdamwState(S.init_value(spec, 1), np.zeros(spec.shape, np.float32),
                    np.zeros(spec.shape, np.float32), np.zeros(spec.shape, np.float32))
    hp = dict(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
              weight_decay=w.adamw.weight_decay)
    for t in range(1, w.steps + 1):
        st.h["g"][...] = S.grad_value(spec, 1, t)
        st.d["g"].copy_(dev(st.h["g"]))
        mp.adamw_step([st.param()], mp.adamw_hp(step=t, **hp))
        OA.adamw_step_fp32(st.h["p"], st.h["g"], st.h["m"], st.h["v"], t=t, **hp)
        torch.cuda.synchronize()
        check(st, f"step {t}")


def test_adamw_8m_100_steps_bit_exact():
    """The two-matrix AdamW workload (4096x1024 + 1024x4096, init N(0,1),
    gradients N(0, 1e-3)) at full size for all 100 steps."""
    w = S.adamw_8m()
    hp = dict(lr=w.adamw.lr, beta1=w.adamw.beta1, beta2=w.adamw.beta2, eps=w.adamw.eps,
              weight_decay=w.adamw.weight_decay)
    states = []
    for i, spec in enumerate(w.tensors):
        z = np.zeros(spec.shape, np.float32)
        states.append(AdamwState(S.init_value(spec, i), z, z.copy(), z.copy()))
    for t in range(1, w.steps + 1):
        for i, (st, spec) in enumerate(zip(states, w.tensors)):
            st.h["g"][...] = S.grad_value(spec, i, t)
            st.d["g"].copy_(dev(st.h["g"]))
        mp.adamw_step([s.param() for s in states], mp.adamw_hp(step=t, **hp))
        for st in states:
            oracle_step(st, t, hp)
        if t in (1, 2, 50, w.steps):
            torch.cuda.synchronize()
            for i, st in enumerate(states):
                check(st, f"step {t} tensor {i}")


def test_bf16_writeback_every_fp32_pattern():
    """lr = 0, lambda = 0, zero gradient and moments leave p unchanged
    (p*1 - 0*0), so the step writes bf16_rne(p) for every p: all 2^32 fp32
    bit patterns, in chunks, compared with the oracle's rounding of the GPU's
    own master weights."""
    chunk = 1 << 28
    p = torch.empty(chunk, dtype=torch.float32, device="cuda")
    z = torch.zeros(chunk, dtype=torch.float32, device="cuda")
    m = torch.zeros_like(z)
    v = torch.zeros_like(z)
    model = torch.empty(chunk, dtype=torch.bfloat16, device="cuda")
    hp = mp.adamw_hp(lr=0.0, weight_decay=0.0, step=1)
    idx = torch.arange(chunk, dtype=torch.int64, device="cuda")
    for c in range(1 << 32 >> 28):
        bits = (idx + c * chunk).to(torch.int64)
        p.view(torch.int32).copy_(bits.to(torch.int32) if c < 8 else (bits - (1 << 32)).to(torch.int32))
        m.zero_()
        v.zero_()
        mp.adamw_step([mp.Param(p, z, m, v, model)], hp)
        got = bf16_host(model)
        want = OA.bf16_rne(host(p))
        bad = np.nonzero(got != want)[0]
        assert bad.size == 0, f"chunk {c}: {bad.size} mismatches, first bits {c * chunk + bad[0]:#x}"
