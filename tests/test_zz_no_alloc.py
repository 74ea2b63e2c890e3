"""opt_newton_schulz_noalloc: Newton-Schulz for callers that cannot allocate
device memory (a host runtime that owns every allocation and gives extensions
no allocator, or a fixed memory budget).  Its scratch is an array built into
the library instead of a caller workspace.  This file checks, through the C
ABI, that two calls in a row give the workspace entry point's result within
the Newton-Schulz tolerance of the other tests, and that sizes beyond the
built-in scratch are refused.  It is named to be collected last so that a run
stopping at the first failure has already run every other test."""

import ctypes

import numpy as np
import pytest

from gpu_helpers import dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import muon as OM

pytestmark = pytest.mark.gpu

NS_TOL = 2e-2


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def rel(a, b):
    return float(np.linalg.norm(np.asarray(a, np.float64) - b) / np.linalg.norm(b))


def with_workspace(Gd, steps):
    out = torch.empty_like(Gd)
    ws = mp.alloc_workspace(mp.newton_schulz_workspace_size(*Gd.shape))
    mp.newton_schulz(Gd, out, steps=steps, workspace=ws)
    return out


def without_allocation(Gd, steps):
    out = torch.empty_like(Gd)
    a, b, c = mp.NS_COEFFS
    st = mp.lib().opt_newton_schulz_noalloc(ctypes.c_void_p(Gd.data_ptr()), ctypes.c_void_p(out.data_ptr()),
                                            Gd.shape[0], Gd.shape[1], steps, a, b, c, 1e-7,
                                            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == mp.OPT_OK, mp.lib().opt_last_cuda_error()
    # no device-side wait of the call ran out (status word of the built-in array)
    assert mp.lib().opt_noalloc_device_status(ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)) == mp.OPT_OK
    return out


def test_noalloc_matches_workspace_entry_point_two_calls():
    # the largest accepted shape first, then a smaller tall one: the second
    # call must not depend on what the first left in the shared scratch
    for shape, seed, steps in (((1024, 4096), 1, 5), ((700, 300), 2, 5)):
        G = np.random.default_rng(seed).standard_normal(shape).astype(np.float32)
        Gd = dev(G)
        ref = with_workspace(Gd, steps)
        got = without_allocation(Gd, steps)
        torch.cuda.synchronize()
        r, g = host(ref).astype(np.float64), host(got).astype(np.float64)
        assert rel(g, r) < NS_TOL
        assert rel(g, OM.newton_schulz(G.astype(np.float64), steps)) < NS_TOL


def test_noalloc_refuses_oversize():
    L = mp.lib()
    a, b, c = mp.NS_COEFFS
    for rows, cols in ((1025, 2000), (100, 4097), (4097, 100)):
        st = L.opt_newton_schulz_noalloc(ctypes.c_void_p(1 << 20), ctypes.c_void_p(1 << 20), rows, cols, 5,
                                         a, b, c, 1e-7, None)
        assert st == 2                      # OPT_ERR_UNSUPPORTED
        assert b"exceeds the built-in scratch" in L.opt_last_cuda_error()
