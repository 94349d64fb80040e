"""Failure detection on the GPU without a fault.  Every pipeline wait of the
expert GEMMs is bounded (the stage rings' mbarrier waits, and the one-launch
decode layer's wait of a down stage for its gate/up tile, a count): past its limit
it records BI_DEVERR_WAIT_TIMEOUT in the device error word and the kernel
unwinds.  Here a probe kernel waits on a barrier phase that nothing
completes, or a count that nothing raises; the wait must give up after about
a second, the host must read the status, and the context must keep running
the path afterwards."""
import time

import pytest
import torch

from tests import synthetic as syn

pytestmark = pytest.mark.gpu

WAIT_TIMEOUT = 3  # BI_DEVERR_WAIT_TIMEOUT


@pytest.mark.parametrize("which", [0, 1])
def test_bounded_wait_gives_up_and_context_survives(cuda, which):
    import invariant_moe_gb300 as bm
    assert bm.device_error() == 0
    t0 = time.perf_counter()
    bm.bi_wait_timeout_probe(which)
    code = bm.device_error()  # synchronises the device
    elapsed = time.perf_counter() - t0
    assert code == WAIT_TIMEOUT
    assert 0.9 < elapsed < 30.0, elapsed
    assert bm.device_error() == 0  # reading the word cleared it

    # the same context still runs the path
    x = syn.normal((8, 4096), 1.0, 7).to(cuda)
    w = syn.normal((256, 4096), 1.0 / 64, 8).to(cuda)
    y = bm.bi_router_gemm(x, w)
    y_again = bm.bi_router_gemm(x, w)
    torch.cuda.synchronize()
    assert torch.isfinite(y).all() and torch.equal(y, y_again)
