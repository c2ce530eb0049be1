"""Device-side failure detection without a GPU fault: a bounded wait on a
barrier that never completes gives up with MOE_ERR_TIMEOUT after the limit,
and the context keeps computing correctly afterwards."""
import numpy as np
import pytest

import synth
from harness import DeviceLayer, check_out, check_route, oracle_out, torch

pytestmark = pytest.mark.gpu

MOE_OK, MOE_ERR_TIMEOUT = 0, 5


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch().cuda.is_available():
        pytest.skip("no CUDA device")


def test_bounded_wait_times_out_and_context_survives():
    import mxfp4_routed_expert_moe_gb300 as moe
    for cycles in (1_000, 2_000_000):  # ~0.5 us and ~1 ms at 2 GHz
        assert moe.wait_selftest(cycles) == MOE_ERR_TIMEOUT
    # The same context still runs the layer correctly.
    inp = synth.make_inputs(synth.WORKLOADS["tiny"])
    L = DeviceLayer(inp)
    out, ids, w = L.forward()
    torch().cuda.synchronize()
    assert L.status() == MOE_OK
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), "after timeout")


def test_wait_selftest_rejects_bad_limits():
    import mxfp4_routed_expert_moe_gb300 as moe
    for bad in (0, -5, 5_000_000_000):
        with pytest.raises(moe.MoeError):
            moe.wait_selftest(bad)
