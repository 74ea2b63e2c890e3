"""opt_copy_from_host: a host-to-device copy of page-locked memory by SM
loads, used where gradients arrive in host memory.  Checked through the C ABI:
bit-exact copies of every size class (empty, 4-byte words only, ragged 16-byte
tails, large), the 4-byte path for buffers that are not 16-byte aligned, the
refused arguments, and a copy on a second stream while a Muon step runs."""

import ctypes

import numpy as np
import pytest

from gpu_helpers import dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import muon as OM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def pinned_words(n, seed):
    src = torch.empty(n, dtype=torch.int32, pin_memory=True)
    src.copy_(torch.from_numpy(np.random.default_rng(seed).integers(-2 ** 31, 2 ** 31 - 1, n, dtype=np.int64)
                               .astype(np.int32)))
    return src


@pytest.mark.parametrize("n", [0, 1, 3, 4, 5, 1023, 4096 + 3, 1 << 20, (64 << 20) + 7])
@pytest.mark.parametrize("offset", [0, 1])
def test_copy_is_bit_exact(n, offset):
    """offset 1 shifts both buffers by one 4-byte word: no 16-byte accesses."""
    src = pinned_words(n + offset, n)[offset:]
    dst_buf = torch.full((n + offset,), -7, dtype=torch.int32, device="cuda")
    dst = dst_buf[offset:]
    mp.copy_from_host(dst, src)
    torch.cuda.synchronize()
    assert np.array_equal(host(dst), src.numpy())
    if offset:
        assert int(dst_buf[0]) == -7                  # nothing written before dst


def test_copy_mixed_alignment_and_float_payloads():
    """A 16-byte aligned source into a 4-byte aligned destination, and fp32
    payloads with NaN, infinities and subnormals: bits are moved, not values."""
    vals = np.array([np.nan, np.inf, -np.inf, 1e-45, -0.0, 3.5, 65504.0] * 1000, dtype=np.float32)
    src = torch.empty(len(vals), dtype=torch.float32, pin_memory=True)
    src.copy_(torch.from_numpy(vals))
    dst_buf = torch.zeros(len(vals) + 1, dtype=torch.float32, device="cuda")
    mp.copy_from_host(dst_buf[1:], src)
    torch.cuda.synchronize()
    assert np.array_equal(host(dst_buf[1:]).view(np.uint32), vals.view(np.uint32))


def test_copy_refuses_bad_arguments():
    L = mp.lib()
    dst = torch.empty(64, dtype=torch.int32, device="cuda")
    pinned = pinned_words(64, 1)
    pageable = torch.zeros(64, dtype=torch.int32)
    on_device = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    assert L.opt_copy_from_host(p(dst), p(pageable), 256, None) == mp.OPT_ERR_INVALID_ARG
    assert L.opt_copy_from_host(p(dst), p(on_device), 256, None) == mp.OPT_ERR_INVALID_ARG
    assert L.opt_copy_from_host(p(pinned), p(pinned), 256, None) == mp.OPT_ERR_INVALID_ARG   # dst on the host
    assert L.opt_copy_from_host(None, p(pinned), 256, None) == mp.OPT_ERR_INVALID_ARG
    assert L.opt_copy_from_host(ctypes.c_void_p(dst.data_ptr() + 2), p(pinned), 252, None) == mp.OPT_ERR_MISALIGNED
    assert L.opt_copy_from_host(p(dst), p(pinned), 6, None) == mp.OPT_ERR_MISALIGNED
    assert L.opt_copy_from_host(p(dst), p(pinned), 0, None) == mp.OPT_OK
    with pytest.raises(ValueError):
        mp.copy_from_host(dst, pinned[:32])


def test_copy_beside_a_muon_step():
    """A 256 MB copy on a second stream while a Muon step of a 1024 x 4096
    matrix runs on the first: both results are exact / within the bar."""
    n = 64 << 20
    src = pinned_words(n, 3)
    dst = torch.empty(n, dtype=torch.int32, device="cuda")
    shape = (1024, 4096)
    rng = np.random.default_rng(4)
    W = (rng.standard_normal(shape) * 0.02).astype(np.float32)
    g = (rng.standard_normal(shape) * 1e-2).astype(np.float32)
    m = np.zeros(shape, np.float32)
    Wd = dev(W)
    p = mp.Param(Wd, dev(g), dev(m), None, torch.zeros(shape, dtype=torch.bfloat16, device="cuda"))
    ws = mp.alloc_workspace(mp.workspace_size([p], "muon"))
    side = torch.cuda.Stream()
    torch.cuda.synchronize()
    mp.muon_step(p, mp.muon_hp(), ws)
    mp.copy_from_host(dst, src, stream=side)
    torch.cuda.synchronize()
    assert np.array_equal(host(dst), src.numpy())
    assert mp.device_status(ws) == mp.OPT_OK
    Wn, _, _ = OM.muon_step(W, g, m, lr=0.02, momentum=0.95)
    W1 = host(Wd).astype(np.float64)
    assert np.linalg.norm((W - W1) - (W - Wn)) / np.linalg.norm(W - Wn) < 2e-2
