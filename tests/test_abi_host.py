"""Host-side tests of the C ABI: the library loads without a GPU, exports
every function include/mpopt.h declares, and rejects bad arguments on the
host before anything is enqueued.  Pointers here are fake aligned addresses
that are never dereferenced (every case returns before a CUDA call)."""

import ctypes
import os
import re

import pytest

import mixed_precision_optimizer_gb300 as mp
from mixed_precision_optimizer_gb300 import build_lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_lib.build()
    return mp.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "mpopt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(opt_[a-z_0-9]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(mp.EXPORTED)
    out = os.popen(f"nm -D --defined-only {mp.LIB_PATH}").read()
    exported = set(re.findall(r"\bT (opt_\w+)", out))
    assert exported == set(names), exported ^ set(names)


def test_strerror_and_version(L):
    for code, name in mp.STATUS_NAMES.items():
        assert L.opt_strerror(code)
    assert L.opt_strerror(99) == b"unknown status"
    assert L.opt_abi_version() >> 16 == 2


FAKE = 1 << 20     # 1 MiB: an aligned address, never dereferenced


def tensor(rows, cols, ndim=2, kind=mp.KIND_AUTO, flags=0, base=FAKE, model=True, sq=True):
    t = mp.OptTensor()
    t.main_param, t.main_grad, t.exp_avg = base, base + (1 << 30), base + (2 << 30)
    t.exp_avg_sq = base + (3 << 30) if sq else None
    t.model_param = base + (4 << 30) if model else None
    t.rows, t.cols, t.ndim, t.kind, t.flags = rows, cols, ndim, kind, flags
    return t


def arr(*ts):
    a = (mp.OptTensor * len(ts))()
    for i, t in enumerate(ts):
        a[i] = t
    return a


def adamw(L, ts, hp=None, ws=None, nb=0):
    hp = hp or mp.adamw_hp()
    return L.opt_adamw_step(ctypes.byref(hp), arr(*ts), len(ts), ws, nb, None)


def test_adamw_argument_errors(L):
    E = mp.STATUS_NAMES
    inv, mis = 1, 3
    assert adamw(L, [tensor(1, 10, 1)], mp.adamw_hp(step=0)) == inv           # t counts from 1
    assert adamw(L, [tensor(1, 10, 1)], mp.adamw_hp(beta1=1.0)) == inv
    assert adamw(L, [tensor(1, 10, 1)], mp.adamw_hp(beta2=-0.1)) == inv
    assert adamw(L, [tensor(1, 10, 1)], mp.adamw_hp(lr=float("nan"))) == inv
    assert adamw(L, [tensor(1, 10, 1)], mp.adamw_hp(eps=float("inf"))) == inv
    assert adamw(L, [tensor(1, 10, 1, sq=False)]) == inv                        # v missing
    t = tensor(1, 10, 1)
    t.main_grad = None
    assert adamw(L, [t]) == inv
    assert adamw(L, [tensor(1, 10, 1, base=FAKE + 2)]) == mis                   # fp32 not 4-B aligned
    t = tensor(1, 10, 1)
    t.model_param = FAKE + 1
    assert adamw(L, [t]) == mis                                                 # bf16 not 2-B aligned
    assert adamw(L, [tensor(-1, 10, 1)]) == inv
    assert adamw(L, [tensor(1, 10, 1, kind=7)]) == inv
    assert L.opt_adamw_step(ctypes.byref(mp.adamw_hp()), None, 3, None, 0, None) == inv
    assert L.opt_adamw_step(None, arr(tensor(1, 10, 1)), 1, None, 0, None) == inv
    # nothing to do: empty list and zero-size tensors succeed without a GPU
    assert L.opt_adamw_step(ctypes.byref(mp.adamw_hp()), None, 0, None, 0, None) == 0
    t = tensor(0, 5, 2)
    t.main_param = None
    assert adamw(L, [t]) == 0
    assert E[inv] == "OPT_ERR_INVALID_ARG"


def test_muon_argument_errors(L):
    inv = 1
    hp = mp.muon_hp()
    ws = ctypes.c_void_p(FAKE)
    big = 1 << 40
    assert L.opt_muon_step(ctypes.byref(hp), arr(tensor(8, 16, 1)), ws, big, None) == inv   # not 2-D
    assert L.opt_muon_step(ctypes.byref(mp.muon_hp(ns_steps=17)), arr(tensor(8, 16)), ws, big, None) == inv
    assert L.opt_muon_step(ctypes.byref(mp.muon_hp(ns_steps=-1)), arr(tensor(8, 16)), ws, big, None) == inv
    assert L.opt_muon_step(ctypes.byref(mp.muon_hp(momentum=1.0)), arr(tensor(8, 16)), ws, big, None) == inv
    assert L.opt_muon_step(ctypes.byref(mp.muon_hp(eps=-1.0)), arr(tensor(8, 16)), ws, big, None) == inv
    assert L.opt_muon_step(ctypes.byref(mp.muon_hp(coeffs=(1.0, float("nan"), 1.0))), arr(tensor(8, 16)),
                           ws, big, None) == inv
    assert L.opt_muon_step(None, arr(tensor(8, 16)), ws, big, None) == inv
    bad = mp.muon_hp()
    bad.scale_mode = 3
    assert L.opt_muon_step(ctypes.byref(bad), arr(tensor(8, 16)), ws, big, None) == inv
    bad = mp.muon_hp()
    bad.flags = 8                                           # not a defined flag
    assert L.opt_muon_step(ctypes.byref(bad), arr(tensor(8, 16)), ws, big, None) == inv
    sched = mp.muon_hp(ns_steps=2, schedule=[(1.0, 2.0, 3.0), (1.0, float("inf"), 3.0)])
    assert L.opt_muon_step(ctypes.byref(sched), arr(tensor(8, 16)), ws, big, None) == inv
    t = tensor(8, 16)
    t.scale_rows = 24                                       # scale shape needs both dims
    assert L.opt_muon_step(ctypes.byref(hp), arr(t), ws, big, None) == inv
    assert L.opt_muon_step(ctypes.byref(hp), None, ws, big, None) == inv
    # workspace: missing, misaligned, too small
    assert L.opt_muon_step(ctypes.byref(hp), arr(tensor(8, 16)), None, 0, None) == 4
    assert L.opt_muon_step(ctypes.byref(hp), arr(tensor(8, 16)), ctypes.c_void_p(FAKE + 64), big, None) == 4
    need = L.opt_workspace_size(arr(tensor(8, 16)), 1, mp.KIND_MUON)
    assert L.opt_muon_step(ctypes.byref(hp), arr(tensor(8, 16)), ws, need - 1, None) == 4


def test_workspace_size_formula(L):
    # one matrix 300 x 200: wide orientation A=200 -> 256, B=300 -> 512
    # fp16 iterate twice (ping-pong); fp16 Gram; fp16 polynomial; norm
    # partials of 8192 elements each; one inverse norm
    Ap, Bp = 256, 512
    al = lambda x: (x + 1023) // 1024 * 1024
    ab, aa, blocks = Ap * Bp, Ap * Ap, -(-(300 * 200) // 8192)
    want = 256 + 2 * al(ab * 2) + al(aa * 2) + al(aa * 2) + al(blocks * 4) + al(4)
    assert L.opt_workspace_size(arr(tensor(300, 200)), 1, mp.KIND_MUON) == want
    # AdamW needs none
    assert L.opt_workspace_size(arr(tensor(1, 1000, 1), tensor(30, 40)), 2, mp.KIND_ADAMW) == 0
    # auto routing: 2-D -> Muon unless flagged embedding/output; 1-D -> AdamW
    assert L.opt_workspace_size(arr(tensor(1, 1000, 1)), 1, mp.KIND_AUTO) == 0
    assert L.opt_workspace_size(arr(tensor(300, 200, flags=1)), 1, mp.KIND_AUTO) == 0
    assert L.opt_workspace_size(arr(tensor(300, 200)), 1, mp.KIND_AUTO) == want
    # same (min, max) shape in both orientations shares one class: two matrices
    two = L.opt_workspace_size(arr(tensor(300, 200), tensor(200, 300)), 2, mp.KIND_AUTO)
    assert two > want
    # clipping adds the header (if absent) and one float per 16K gradient elements
    assert L.opt_workspace_size(arr(tensor(1, 1000, 1)), 1, mp.KIND_AUTO | mp.WORKSPACE_CLIP) == 256 + 1024
    assert L.opt_workspace_size(arr(tensor(300, 200)), 1, mp.KIND_AUTO | mp.WORKSPACE_CLIP) == want + 1024
    # grouped iterations: two more fp16 [Ap][Ap] buffers, on request for any shape
    assert L.opt_workspace_size(arr(tensor(300, 200)), 1, mp.KIND_MUON | mp.WORKSPACE_GROUPED) == want + 2 * al(aa * 2)
    # invalid list -> 0
    assert L.opt_workspace_size(arr(tensor(300, 200, ndim=3)), 1, mp.KIND_MUON) == 0
    assert L.opt_workspace_size(arr(tensor(300, 200)), 1, 9) == 0


def test_grouped_iterations_by_default_where_they_pay(L):
    """Shapes whose padded max side is at least twice the padded min side, with
    a min side of 1024 or more, take grouped Newton-Schulz iterations by
    default, and their workspace holds the two extra fp16 [Ap][Ap] buffers;
    other shapes get them only when sized for grouping."""
    al = lambda x: (x + 1023) // 1024 * 1024

    def plain(R, C):
        A, B = min(R, C), max(R, C)
        Ap, Bp = -(-A // 256) * 256, -(-B // 256) * 256
        blocks = max(-(-(A * B) // 8192), (Ap // 64) * (Bp // 64))
        return 256 + 2 * al(Ap * Bp * 2) + 2 * al(Ap * Ap * 2) + al(blocks * 4) + al(20), al(Ap * Ap * 2)

    for (R, C), grouped in (((1024, 4096), True), ((4096, 1024), True), ((1024, 2048), True),
                            ((4096, 14336), True), ((1000, 2000), True), ((768, 2048), False),
                            ((1024, 1024), False), ((4096, 4096), False), ((1024, 1700), False)):
        base, aa = plain(R, C)
        got = L.opt_workspace_size(arr(tensor(R, C)), 1, mp.KIND_MUON)
        assert got == base + (2 * aa if grouped else 0), (R, C)
        assert L.opt_workspace_size(arr(tensor(R, C)), 1, mp.KIND_MUON | mp.WORKSPACE_GROUPED) == base + 2 * aa


def test_ns_plan_grouping_rules(L):
    """opt_ns_plan (host only) reports how a matrix's iterations are grouped:
    groups of at most three, the larger first, for the shapes grouped by
    default (padded max side >= 2 x padded min side, min side >= 1024) or
    every shape with OPT_MUON_NS_GROUPED; one at a time otherwise."""
    hp = mp.muon_hp()
    assert mp.ns_plan(4096, 14336, hp) == [3, 2] and mp.ns_plan(14336, 4096, hp) == [3, 2]
    assert mp.ns_plan(1024, 4096, hp) == [3, 2]
    for shape in ((4096, 4096), (768, 2048), (1024, 1700), (300, 700), (1, 64)):
        assert mp.ns_plan(*shape, hp) == [1] * 5, shape
        assert mp.ns_plan(*shape, mp.muon_hp(ns_order="grouped")) == [3, 2], shape
    assert mp.ns_plan(4096, 14336, mp.muon_hp(ns_order="per_iteration")) == [1] * 5
    for steps, sizes in ((1, [1]), (2, [2]), (3, [3]), (4, [2, 2]), (6, [3, 3]), (7, [3, 2, 2]),
                         (8, [3, 3, 2]), (16, [3, 3, 3, 3, 2, 2])):
        assert mp.ns_plan(300, 700, mp.muon_hp(ns_steps=steps, ns_order="grouped")) == sizes, steps
    assert mp.ns_plan(4096, 14336, mp.muon_hp(ns_steps=0)) == []
    assert mp.ns_plan(4096, 14336, mp.muon_hp(orthogonalize=False)) == []


def test_ns_plan_splits_groups_that_could_leave_fp16(L):
    """A group is split into single iterations when the product of its
    polynomials' largest values over the reachable singular values exceeds
    4096.  With b = c = 0 an iteration multiplies every singular value by a:
    a = 15 three times bounds the group by 15^3 = 3375 (grouped), a = 16 by
    4096 plus the bound's margin (split).  The printed coefficients bound a
    group of three by about 42."""
    g = lambda a: mp.muon_hp(ns_order="grouped", schedule=[(a, 0.0, 0.0)] * 3 + [(1.0, 0.0, 0.0)] * 2)
    assert mp.ns_plan(300, 700, g(15.0)) == [3, 2]
    assert mp.ns_plan(300, 700, g(16.0)) == [1, 1, 1, 2]
    assert mp.ns_plan(300, 700, g(-16.0)) == [1, 1, 1, 2]           # |p| counts
    big_late = mp.muon_hp(ns_order="grouped", schedule=[(1.0, 0.0, 0.0)] * 3 + [(100.0, 0.0, 0.0)] * 2)
    assert mp.ns_plan(300, 700, big_late) == [3, 1, 1]
    # the printed coefficients, and a schedule whose quintics keep [0, 1]
    # bounded, stay grouped; one whose singular values near 1 grow without
    # bound (envelope 42 after four iterations) has its second group split
    assert mp.ns_plan(300, 700, mp.muon_hp(ns_order="grouped")) == [3, 2]
    bounded = [(3.4445, -4.7750, 2.0315), (3.2, -4.4, 1.9), (3.0, -4.0, 1.7), (2.8, -3.6, 1.55), (2.2, -2.1, 0.9)]
    assert mp.ns_plan(300, 700, mp.muon_hp(ns_order="grouped", schedule=bounded)) == [3, 2]
    growing = [(3.4445, -4.7750, 2.0315), (3.0, -3.8, 1.7), (2.8, -3.4, 1.5), (3.2, -4.3, 1.9), (2.5, -2.9, 1.3)]
    assert mp.ns_plan(300, 700, mp.muon_hp(ns_order="grouped", schedule=growing)) == [3, 1, 1]


def test_ns_plan_errors(L):
    hp = mp.muon_hp()
    out, n = (ctypes.c_int32 * 8)(), ctypes.c_int32(0)
    assert L.opt_ns_plan(0, 10, ctypes.byref(hp), out, 8, ctypes.byref(n)) == 1
    assert L.opt_ns_plan(10, 10, None, out, 8, ctypes.byref(n)) == 1
    assert L.opt_ns_plan(10, 10, ctypes.byref(hp), None, 8, ctypes.byref(n)) == 1
    assert L.opt_ns_plan(10, 10, ctypes.byref(hp), out, 4, ctypes.byref(n)) == 1     # capacity < ns_steps
    bad = mp.muon_hp()
    bad.flags = mp.MUON_NS_GROUPED | mp.MUON_NS_PER_ITERATION
    assert L.opt_ns_plan(10, 10, ctypes.byref(bad), out, 8, ctypes.byref(n)) == 1
    assert L.opt_ns_plan(10, 10, ctypes.byref(hp), out, 5, ctypes.byref(n)) == 0 and n.value == 5


def test_ns_order_flags(L):
    """At most one evaluation-order flag; unknown flag bits are refused.  The
    hyper-parameters are checked before the workspace, so an accepted flag
    set reaches the missing-workspace error (4) and a refused one stops at 1."""
    for flags, want in ((0, 4), (mp.MUON_NS_GROUPED, 4), (mp.MUON_NS_PER_ITERATION, 4),
                        (mp.MUON_NS_GROUPED | mp.MUON_NS_PER_ITERATION, 1), (8, 1),
                        (mp.MUON_NO_ORTHOGONALIZE | mp.MUON_NS_GROUPED, 4)):
        hp = mp.muon_hp()
        hp.flags = flags
        assert L.opt_muon_step(ctypes.byref(hp), arr(tensor(8, 16)), None, 0, None) == want, flags
    assert mp.muon_hp(ns_order="grouped").flags == mp.MUON_NS_GROUPED
    assert mp.muon_hp(ns_order="per_iteration", orthogonalize=False).flags == (
        mp.MUON_NS_PER_ITERATION | mp.MUON_NO_ORTHOGONALIZE)


def test_clipped_step_argument_errors(L):
    hpa = mp.adamw_hp()
    f = L.opt_mixed_step_clipped
    one = arr(tensor(1, 10, 1))
    assert f(None, ctypes.byref(hpa), float("nan"), None, None, one, 1, None, 0, None) == 1
    assert f(None, ctypes.byref(hpa), 1.0, ctypes.c_void_p(FAKE + 2), None, one, 1, None, 0, None) == 3
    assert f(None, ctypes.byref(hpa), 1.0, None, None, one, 1, None, 0, None) == 4      # needs workspace
    assert f(None, ctypes.byref(mp.adamw_hp(step=0)), 1.0, None, None, one, 1, None, 0, None) == 1


def test_newton_schulz_argument_errors(L):
    ws = ctypes.c_void_p(FAKE)
    f = L.opt_newton_schulz
    c = mp.NS_COEFFS
    assert f(FAKE, FAKE, 8, 16, 17, *c, 1e-7, ws, 1 << 40, None) == 1
    assert f(None, FAKE, 8, 16, 5, *c, 1e-7, ws, 1 << 40, None) == 1
    assert f(FAKE + 2, FAKE, 8, 16, 5, *c, 1e-7, ws, 1 << 40, None) == 3
    assert f(FAKE, FAKE, 8, 16, 5, *c, -1.0, ws, 1 << 40, None) == 1
    assert f(FAKE, FAKE, 0, 16, 5, *c, 1e-7, ws, 1 << 40, None) == 0     # empty: nothing to do
    assert f(FAKE, FAKE, 8, 16, 5, *c, 1e-7, None, 0, None) == 4


def test_binding_rejects_wrong_tensors():
    import torch
    p = torch.zeros(4)
    with pytest.raises(ValueError):
        mp.Param(p, p, p, p).to_c()               # CPU tensors are refused
    with pytest.raises(TypeError):
        mp.Param(p.double(), p, p, p).to_c()


def test_library_has_no_cpu_fallback():
    """The product path imports nothing from the oracle."""
    pkg = os.path.join(ROOT, "mixed_precision_optimizer_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".h")):
                src = open(os.path.join(dirpath, f), encoding="utf-8").read()
                assert "oracle" not in src.replace("the oracle", ""), f


def test_copy_from_host_argument_errors(L):
    """Checked on the host before any CUDA call: null pointers, alignment,
    and an empty copy that does nothing."""
    assert L.opt_copy_from_host(None, ctypes.c_void_p(FAKE), 16, None) == 1
    assert L.opt_copy_from_host(ctypes.c_void_p(FAKE), None, 16, None) == 1
    assert L.opt_copy_from_host(ctypes.c_void_p(FAKE + 2), ctypes.c_void_p(FAKE), 16, None) == 3
    assert L.opt_copy_from_host(ctypes.c_void_p(FAKE), ctypes.c_void_p(FAKE), 14, None) == 3
    assert L.opt_copy_from_host(None, None, 0, None) == 0
