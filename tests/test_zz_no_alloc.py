"""moe_forward_static_scratch: the layer with the library's own static device
scratch as workspace.  Its results must match moe_forward with a caller
workspace (same launch sequence), call after call, and shapes whose workspace
exceeds the scratch must be refused before anything runs.  Collected last so
that it also runs after every other GPU test in the same process."""
import numpy as np
import pytest

import synth
from harness import DeviceLayer, torch


def test_oversize_shape_is_refused_before_launch():
    import mxfp4_routed_expert_moe_gb300 as moe
    shp = moe.shape(64, 7168, 896, 1408, 16)
    assert moe.workspace_bytes(64, 7168, 896, 1408, 16) > moe.STATIC_SCRATCH_BYTES
    x = torch().zeros(8, dtype=torch().bfloat16)  # only its dtype is read: the call must return first
    with pytest.raises(moe.MoeError) as err:
        moe.forward_static_scratch(shp, x, None, None, None, None, None, False, stream=0)
    assert err.value.status == 3  # MOE_ERR_WORKSPACE


def _compare(name, wl, path):
    t = torch()
    inp = synth.make_inputs(wl)
    L = DeviceLayer(inp)
    moe = L.moe
    ref, ids_ref, w_ref = L.forward(path=path)
    status = t.full((1,), -1, dtype=t.int32, device="cuda")
    for call in range(2):
        out = t.full((wl.T, wl.H), float("nan"), dtype=t.float32, device="cuda")
        ids = t.empty((wl.T, wl.k), dtype=t.int32, device="cuda")
        w = t.empty((wl.T, wl.k), dtype=t.float32, device="cuda")
        moe.forward_static_scratch(L.shape, L.x, L.wr, L.br, L.table.desc, L.shared, out, False, ids_out=ids,
                                   w_out=w, path=path, status_dev=status)
        t.cuda.synchronize()
        assert int(status.item()) == 0, f"{name} call {call}: device status {int(status.item())}"
        assert t.equal(ids, ids_ref), f"{name} call {call}: ids differ"
        assert float((w - w_ref).abs().max()) <= 1e-6
        if path == 1:
            # The decode path sums in a fixed order: bitwise the same result.
            assert t.equal(out, ref), f"{name} call {call}: output differs from moe_forward"
        else:
            # The prefill path combines with fp32 atomics (order not fixed).
            a, b = out.cpu().numpy().astype(np.float64), ref.cpu().numpy().astype(np.float64)
            rel = np.linalg.norm(a - b) / np.linalg.norm(b)
            assert rel <= 1e-5, f"{name} call {call}: rel-L2 {rel:.2e} against moe_forward"


@pytest.mark.gpu
@pytest.mark.parametrize("name,path", [("tiny", 1), ("decode_e32", 1), ("pf_small", 2)])
def test_static_scratch_matches_forward(name, path):
    if not torch().cuda.is_available():
        pytest.skip("no CUDA device")
    wl = synth.WORKLOADS.get(name) or synth.Workload("pf_small_T100_H256_E8_k2_I128", 100, 256, 8, 2, 128)
    _compare(name, wl, path)
