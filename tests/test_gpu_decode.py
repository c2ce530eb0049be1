"""GPU parity of routing and the decode (weight-streaming GEMV) path against the
fp64 oracle, through the C ABI.  Workloads: the tiny fp32 layer, 1-token
decode and 8-token wide decode at full size, and small edge shapes."""
import numpy as np
import pytest

import synth
from harness import (DeviceLayer, check_buckets, check_out, check_route, oracle_out, torch)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_routed_expert_moe_gb300 as moe
    moe.lib()  # raises if the library is missing: no fallback


def _small_workload(name, T, H, E, k, I, x_dtype="bf16"):
    return synth.Workload(name, T, H, E, k, I, x_dtype=x_dtype)


def _rigged_inputs(wl, seed, rig=None):
    inp = synth.make_inputs(wl, seed)
    if rig:
        rig(inp)
    return inp


@pytest.mark.parametrize("name", ["tiny", "decode", "wide", "decode_i1536"])
def test_route_parity(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    L = DeviceLayer(inp)
    ids, w, off, srt = L.route()
    torch().cuda.synchronize()
    assert L.status() == 0
    ids, w, off, srt = (a.cpu().numpy() for a in (ids, w, off, srt))
    amb, _ = check_route(inp, ids, w)
    print(f"{name}: {int(amb.sum())} of {inp.wl.T} tokens have a near-tie among their first k+1 scores")
    check_buckets(ids, off, srt, inp.wl.E)


@pytest.mark.parametrize("name", ["tiny", "decode", "wide", "decode_i1536"])
def test_forward_decode_parity(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=1)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    assert toks.size >= inp.wl.T - 1
    ref = oracle_out(inp, toks)
    check_out(out.cpu().numpy()[toks], ref, name)


def test_wide_decode_shares_experts():
    inp = synth.make_inputs(synth.WORKLOADS["wide"])
    L = DeviceLayer(inp)
    _, ids, _ = L.forward()
    torch().cuda.synchronize()
    ids = ids.cpu().numpy()
    shared, private = synth.planted_sets(inp.wl)
    assert len(set(ids.ravel())) == 72
    for t in range(inp.wl.T):
        assert set(ids[t]) == set(shared) | set(private[t])


def test_batch_invariance_wide_vs_single():
    """A token's route and output in an 8-token decode are bitwise those of
    its 1-token decode."""
    t = torch()
    wl = synth.WORKLOADS["wide"]
    inp = synth.make_inputs(wl)
    L = DeviceLayer(inp)
    out8, ids8, w8 = L.forward(path=1)
    wl1 = synth.Workload("wide_single", 1, wl.H, wl.E, wl.k, wl.I)
    shp1 = L.moe.shape(1, wl.H, wl.E, wl.I, wl.k)
    ws1 = t.empty(L.moe.workspace_bytes(1, wl.H, wl.E, wl.I, wl.k), dtype=t.uint8, device="cuda")
    for tok in range(wl.T):
        x1 = L.x[tok:tok + 1].contiguous()
        out1 = t.zeros((1, wl.H), dtype=t.float32, device="cuda")
        ids1 = t.empty((1, wl.k), dtype=t.int32, device="cuda")
        w1 = t.empty((1, wl.k), dtype=t.float32, device="cuda")
        L.moe.forward(shp1, x1, L.wr, None, L.table.desc, None, out1, False, ws1, ids_out=ids1, w_out=w1, path=1)
        t.cuda.synchronize()
        assert t.equal(ids1[0], ids8[tok])
        assert t.equal(w1[0], w8[tok])
        assert t.equal(out1[0], out8[tok]), f"token {tok} differs"
    del wl1


def test_accumulate_adds_residual():
    t = torch()
    inp = synth.make_inputs(synth.WORKLOADS["tiny"])
    L = DeviceLayer(inp)
    out0, _, _ = L.forward(path=1)
    res = t.randn(out0.shape, device="cuda", generator=t.Generator("cuda").manual_seed(3))
    out1 = res.clone()
    L.forward(path=1, accumulate=True, out=out1)
    t.cuda.synchronize()
    assert t.equal(out1, out0 + res)
    ref = oracle_out(inp, np.arange(inp.wl.T), residual=res.cpu().numpy())
    check_out(out1.cpu().numpy(), ref, "accumulate")


def test_experts_only_calls_match_forward():
    t = torch()
    inp = synth.make_inputs(synth.WORKLOADS["wide"])
    L = DeviceLayer(inp)
    out_f, _, _ = L.forward(path=1)
    ids, w, off, srt = L.route()
    wl = inp.wl
    out_a = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    out_b = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, srt, out_a, False, L.ws, path=1)
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, None, None, out_b, False, L.ws, path=1)
    t.cuda.synchronize()
    assert L.status() == 0
    assert t.equal(out_a, out_f)
    assert t.equal(out_b, out_f)


EDGE = [
    # name, T, H, E, k, I
    ("t1_k1", 1, 64, 4, 1, 64),
    ("e_eq_k", 3, 64, 4, 4, 96),
    ("odd_t", 7, 96, 16, 3, 160),
    ("k32", 2, 128, 40, 32, 32),
    ("t64", 64, 64, 24, 4, 64),
    ("f32_many", 33, 128, 12, 2, 64),
    # Tensor-core gate/up kernel (bf16 activations, H % 128 == 0): more tokens
    # than router CTAs, items with several 8-pair passes, 1..4 consumer warps.
    ("mma_t64_passes", 64, 512, 16, 4, 256),
    ("mma_t40_all_shared", 40, 256, 8, 8, 128),
    ("mma_h384_odd_warps", 5, 384, 12, 3, 128),
    ("mma_h128_one_warp", 9, 128, 6, 2, 64),
]


@pytest.mark.parametrize("name,T,H,E,k,I", EDGE)
def test_edge_shapes_decode(name, T, H, E, k, I):
    wl = _small_workload(name, T, H, E, k, I, x_dtype="f32" if name.startswith("f32") else "bf16")
    inp = synth.make_inputs(wl, seed=5)
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=1)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    ref = oracle_out(inp, toks)
    check_out(out.cpu().numpy()[toks], ref, name)


def test_zero_load_and_hot_expert():
    """Every token routes to expert 5 first; most experts get no pair."""
    wl = _small_workload("hot", 20, 64, 32, 2, 64)
    inp = synth.make_inputs(wl, seed=9)
    inp.br = np.zeros(wl.E, dtype=np.float32)
    inp.br[5] = 100.0
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=1)
    ids_r, w_r, off, srt = L.route()
    torch().cuda.synchronize()
    ids_n = ids.cpu().numpy()
    assert np.all(ids_n[:, 0] == 5)
    check_route(inp, ids_n, w.cpu().numpy())
    check_buckets(ids_r.cpu().numpy(), off.cpu().numpy(), srt.cpu().numpy(), wl.E)
    assert (np.diff(off.cpu().numpy()) == 0).sum() > 0
    check_out(out.cpu().numpy(), oracle_out(inp, np.arange(wl.T)), "hot")


def test_exact_ties_pick_lower_index():
    wl = _small_workload("ties", 4, 64, 10, 3, 64)
    inp = synth.make_inputs(wl, seed=2)
    inp.wr[7] = inp.wr[2]
    inp.wr[9] = inp.wr[2]
    L = DeviceLayer(inp)
    ids, w, _, _ = L.route()
    torch().cuda.synchronize()
    ids = ids.cpu().numpy()
    w = w.cpu().numpy()
    for t in range(wl.T):
        pos = {int(e): j for j, e in enumerate(ids[t])}
        if 7 in pos:
            assert 2 in pos and pos[2] < pos[7]
        if 9 in pos:
            assert 7 in pos and pos[7] < pos[9]
        if 2 in pos and 7 in pos:
            assert w[t, pos[2]] == w[t, pos[7]]
    check_route(inp, ids, w)


@pytest.mark.parametrize("H", [64, 256], ids=["cuda_core_gateup", "tensor_core_gateup"])
def test_bad_expert_id_sets_device_status(H):
    t = torch()
    wl = _small_workload("badid", 4, H, 8, 2, 128)
    inp = synth.make_inputs(wl, seed=1)
    L = DeviceLayer(inp)
    ids = t.tensor([[0, 1], [2, 99], [3, 4], [5, 6]], dtype=t.int32, device="cuda")
    w = t.full((4, 2), 0.5, dtype=t.float32, device="cuda")
    out = t.zeros((4, H), dtype=t.float32, device="cuda")
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, None, None, out, False, L.ws, path=1)
    assert L.status() == L.moe.MOE_ERR_DEVICE_CHECK
    # The next call on the same workspace starts clean.
    ids[1, 1] = 7
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, None, None, out, False, L.ws, path=1)
    assert L.status() == 0


def test_device_generator_matches_host_generator():
    t = torch()
    wl = synth.WORKLOADS["decode"]
    inp = synth.make_inputs(synth.Workload("gen", 1, wl.H, 3, 1, wl.I))
    import mxfp4_routed_expert_moe_gb300 as moe
    table = moe.ExpertTable(3, wl.H, wl.I, "cuda")
    synth.fill_experts_device(inp, table.blob.data_ptr(), t.cuda.current_stream().cuda_stream)
    t.cuda.synchronize()
    names = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")
    for e in (0, 2):
        ex = inp.expert(e)
        for j, n in enumerate(names):
            assert np.array_equal(table.tensor(e, j).cpu().numpy(), ex[n]), (e, n)


def test_misaligned_expert_descriptor_is_flagged_not_read():
    """An expert whose descriptor holds a misaligned tensor pointer is flagged
    (MOE_ERR_DEVICE_CHECK) and never dereferenced; the next clean call is ok."""
    t = torch()
    wl = _small_workload("misal", 4, 256, 8, 2, 128)
    inp = synth.make_inputs(wl, seed=4)
    inp.br = np.zeros(wl.E, dtype=np.float32)
    inp.br[3] = 100.0
    L = DeviceLayer(inp)
    good = L.table.desc.clone()
    bad = good.clone()
    bad[3, 0] += 8  # gate.q of expert 3, no longer 16-byte aligned
    L.table.desc.copy_(bad)
    out, ids, w = L.forward(path=1)
    assert L.status() == L.moe.MOE_ERR_DEVICE_CHECK
    assert np.all(ids.cpu().numpy()[:, 0] == 3)
    L.table.desc.copy_(good)
    out, ids, w = L.forward(path=1)
    assert L.status() == 0
    check_out(out.cpu().numpy(), oracle_out(inp, np.arange(wl.T)), "after misaligned")


def test_special_scale_codes_decode():
    """E8M0 code 0 (2^-127, subnormal) and 255 (NaN) in the expert scales take
    the exact scale conversion: finite results match the oracle, and a token
    routed to an expert with a NaN scale comes out NaN where the oracle's does."""
    wl = _small_workload("mma_specials", 6, 256, 8, 2, 128)
    inp = synth.make_inputs(wl, seed=11)
    for e in range(wl.E):
        ex = inp.expert(e)
        ex["gate_s"].reshape(-1)[::7] = 0
        ex["up_s"].reshape(-1)[3::11] = 0
    inp.expert(3)["up_s"].reshape(-1)[5] = 255
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=1)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    ref = oracle_out(inp, toks)
    got = out.cpu().numpy()[toks].astype(np.float64)
    nan_ref = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan_ref)
    fin = ~nan_ref.any(axis=1)
    assert fin.any()
    check_out(got[fin], ref[fin], "special scales")
    routed3 = (ids.cpu().numpy()[toks] == 3).any(axis=1)
    assert np.array_equal(nan_ref.all(axis=1), routed3)
