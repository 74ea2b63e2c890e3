"""The bounded device-side waits of the tensor-core kernels.

Every mbarrier wait in the Newton-Schulz GEMM gives up after about 2 s,
records a code in the workspace header and makes every role of its CTA pair
leave its loop.  opt_selftest_wait_timeout withholds one TMA stage of the
first X X^T launch, so the MMA issuer's wait for that stage runs out.  Nothing
faults: the host reads the timeout status, and the same workspace then serves
a normal call whose result matches the oracle."""

import time

import numpy as np
import pytest

from gpu_helpers import dev, host, require_gpu, torch
import mixed_precision_optimizer_gb300 as mp
from oracle import muon as OM

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_withheld_stage_times_out_and_the_workspace_recovers():
    rng = np.random.default_rng(11)
    G = rng.standard_normal((512, 1024)).astype(np.float32)
    Gd = dev(G)
    out = torch.empty_like(Gd)
    ws = mp.alloc_workspace(mp.newton_schulz_workspace_size(*G.shape))

    t0 = time.monotonic()
    mp.selftest_wait_timeout(Gd, out, ws)
    assert mp.device_status(ws) == mp.OPT_ERR_DEVICE_TIMEOUT
    elapsed = time.monotonic() - t0
    assert 1.0 < elapsed < 60.0          # one wait ran out (about 2 s); nothing hung
    code = int(ws[:4].view(torch.int32).item())
    assert 1 <= code <= 7                # which wait gave up first (the kernel's status codes)

    # the context and the workspace are still usable
    mp.newton_schulz(Gd, out, workspace=ws)
    assert mp.device_status(ws) == mp.OPT_OK
    want = OM.newton_schulz(G.astype(np.float64), 5)
    got = host(out).astype(np.float64)
    assert np.linalg.norm(got - want) / np.linalg.norm(want) < 2e-2
