"""Device-side failure detection without a GPU fault: a bounded wait on a
barrier that never completes gives up with MOE_ERR_TIMEOUT after the limit;
the product kernels' own waits give up under a diagnostic limit and take
their abort paths; and the context keeps computing correctly afterwards."""
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


# Shapes that run each product kernel family: the 1-token-class decode path
# (router GEMV, tensor-core gate/up with the fused routing prologue, CUDA-core
# down with the fused combine), the decode path above 64 tokens (router GEMM,
# tensor-core gate/up and down, separate combine), and the prefill path (the
# tcgen05 GEMMs with Tensor-Memory A, the TMA-fed down).
ABORT_CASES = [
    ("decode", 1, (4, 256, 8, 2, 128)),
    ("decode_batch", 1, (80, 256, 8, 2, 128)),
    ("prefill", 2, (130, 256, 8, 2, 128)),
]


@pytest.mark.parametrize("label,path,shape", ABORT_CASES, ids=[c[0] for c in ABORT_CASES])
def test_product_kernel_waits_give_up_and_next_call_is_correct(label, path, shape):
    """With the diagnostic wait limit at 1 cycle, a real wait of the layer's
    kernels (a bulk copy landing, a ring stage, a hand-over between roles)
    gives up: the call reports MOE_ERR_TIMEOUT, each CTA takes its abort path
    (drains its copies, releases Tensor Memory) and exits.  With the default
    limit restored, the next call on the same context and workspace matches
    the oracle."""
    import mxfp4_routed_expert_moe_gb300 as moe
    T, H, E, k, I = shape
    inp = synth.make_inputs(synth.Workload(f"abort_{label}", T, H, E, k, I), seed=13)
    L = DeviceLayer(inp)
    try:
        moe.set_wait_limit(1)
        L.forward(path=path)
        torch().cuda.synchronize()
        status = L.status()
    finally:
        moe.set_wait_limit(0)
    assert status == MOE_ERR_TIMEOUT, moe.status_string(status)
    out, ids, w = L.forward(path=path)
    torch().cuda.synchronize()
    assert L.status() == MOE_OK
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), f"{label} after abort")


def test_set_wait_limit_rejects_bad_values():
    import mxfp4_routed_expert_moe_gb300 as moe
    for bad in (-1, 5_000_000_000):
        with pytest.raises(moe.MoeError):
            moe.set_wait_limit(bad)
    moe.set_wait_limit(0)
