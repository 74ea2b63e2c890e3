"""Helpers for the GPU parity tests: move seeded host arrays to the device,
read results back, and compare them with the oracle."""

from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import mixed_precision_optimizer_gb300 as mp
from mixed_precision_optimizer_gb300 import build_lib


def require_gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    build_lib.build()
    mp.lib()


def dev(a: np.ndarray):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t) -> np.ndarray:
    return t.detach().cpu().numpy()


def bits32(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def bf16_host(t) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what=""):
    """Bit-exact fp32 comparison; any NaN matches any NaN (NaN payloads are
    not part of the method)."""
    g, w = bits32(got).ravel(), bits32(want).ravel()
    gn, wn = np.isnan(got.ravel()), np.isnan(want.ravel())
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    bad = np.nonzero((g != w) & ~gn)[0]
    assert bad.size == 0, (f"{what}: {bad.size} of {g.size} differ; first at {bad[0]}: "
                           f"got {got.ravel()[bad[0]]!r} want {want.ravel()[bad[0]]!r}")


class AdamwState:
    """p, g, m, v (fp32) and the bf16 model copy for one tensor, on the host
    (oracle side) and on the device (library side)."""

    def __init__(self, p, g, m, v, with_model=True):
        self.h = dict(p=p.astype(np.float32), g=g.astype(np.float32), m=m.astype(np.float32),
                      v=v.astype(np.float32))
        self.d = {k: dev(a) for k, a in self.h.items()}
        self.model = torch.zeros(p.shape, dtype=torch.bfloat16, device="cuda") if with_model else None

    def param(self):
        return mp.Param(self.d["p"], self.d["g"], self.d["m"], self.d["v"], self.model)


def singular_values(O) -> np.ndarray:
    """Singular values of a matrix, ascending: square roots of the
    eigenvalues of the Gram matrix of its wide orientation (fp64; clipped at
    zero, so near-zero singular values are exact to about 1e-7)."""
    O = np.asarray(O, dtype=np.float64)
    X = O if O.shape[0] <= O.shape[1] else O.T
    ev = np.linalg.eigvalsh(X @ X.T)
    return np.sqrt(np.clip(ev, 0.0, None))


# Square matrices: a noise-dominated square gradient has singular values near
# zero that five quintic steps do not lift into [0.6, 1.3], even in exact
# arithmetic, so the bound on the update's spectrum becomes: the sorted
# singular values of the output match those of the fp64 oracle's output, each
# within SQUARE_SV_TOL (the distance between the two spectra as
# distributions; it also bounds any histogram of them: counts differ only by
# values within SQUARE_SV_TOL of a bin edge), and none exceeds SQUARE_SV_MAX.
SQUARE_SV_TOL = 0.05
SQUARE_SV_MAX = 1.3


def assert_square_spectrum(got, want, what=""):
    sg, sw = singular_values(got), singular_values(want)
    dev_max = float(np.max(np.abs(sg - sw)))
    assert dev_max <= SQUARE_SV_TOL, f"{what}: sorted singular values differ by up to {dev_max:.3g}"
    assert sg.max() <= SQUARE_SV_MAX, f"{what}: largest singular value {sg.max():.4f}"
    edges = np.linspace(0.0, 1.4, 15)
    hg, _ = np.histogram(sg, edges)
    hw, _ = np.histogram(sw, edges)
    near = sum(int(np.sum(np.abs(sw - e) <= SQUARE_SV_TOL)) for e in edges)
    assert int(np.abs(hg - hw).sum()) <= 2 * near, f"{what}: histograms {hg} vs {hw}"
    return dev_max
