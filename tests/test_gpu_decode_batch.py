"""GPU parity of the decode path on batches above 64 tokens (bf16
activations): routed by the tiled router GEMM and the bucketing kernels, then
the staged decode kernels (tensor-core gate/up and down) and the
slot-ordered combine as a kernel of its own.  Above 2048 routed pairs the kernels read the pair list
from the workspace instead of shared memory."""
import numpy as np
import pytest

import synth
from harness import DeviceLayer, check_out, check_route, oracle_out, torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_routed_expert_moe_gb300 as moe
    moe.lib()  # raises if the library is missing: no fallback


BATCH = [
    # name, T, H, E, k, I
    ("t65_pairs_in_smem", 65, 256, 16, 8, 128),          # 520 pairs: shared-memory pair list
    ("t129_pairs_in_ws", 129, 512, 32, 16, 256),         # 2064 pairs: workspace pair list, ~8 passes per item
    ("t300_three_warps", 300, 384, 40, 7, 256),          # 3 consumer warps, ragged buckets
    ("t1024_max_one_warp", 1024, 128, 64, 4, 128),       # the largest decode batch, 1 consumer warp
]


def _check_forward(inp, name, path=1):
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=path)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    assert toks.size >= inp.wl.T - 2
    ref = oracle_out(inp, toks)
    check_out(out.cpu().numpy()[toks], ref, name)
    return L, out, ids, w


@pytest.mark.parametrize("name,T,H,E,k,I", BATCH)
def test_decode_batch_parity(name, T, H, E, k, I):
    import mxfp4_routed_expert_moe_gb300 as moe
    assert moe.select_path(T, H, E, I, k, path=moe.PATH_DECODE) == moe.PATH_DECODE
    inp = synth.make_inputs(synth.Workload(name, T, H, E, k, I), seed=7)
    _check_forward(inp, name)


def test_decode_batch_full_size_sampled():
    """256 tokens of the full layer (H=7168, 896 experts, top-16, I=1408) on
    the decode path, which the automatic choice takes there; sampled tokens
    against the oracle, the route of every token."""
    import mxfp4_routed_expert_moe_gb300 as moe
    base = synth.WORKLOADS["decode"]
    wl = synth.Workload("batch_T256_H7168_E896_k16_I1408", 256, base.H, base.E, base.k, base.I)
    assert moe.select_path(wl.T, wl.H, wl.E, wl.I, wl.k) == moe.PATH_DECODE
    inp = synth.make_inputs(wl)
    L = DeviceLayer(inp)
    out, ids, w = L.forward()
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    toks = toks[np.linspace(0, toks.size - 1, 3).astype(int)]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), wl.name)


def test_decode_batch_matches_prefill_path():
    """Both expert paths agree on a 200-token batch (same routes)."""
    t = torch()
    inp = synth.make_inputs(synth.Workload("both_paths", 200, 512, 48, 16, 256), seed=3)
    L = DeviceLayer(inp)
    ids, w, off, srt = L.route()
    wl = inp.wl
    o1 = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    o2 = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, srt, o1, False, L.ws, path=1)
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, srt, o2, False, L.ws, path=2)
    t.cuda.synchronize()
    assert L.status() == 0
    a, b = o1.cpu().numpy().astype(np.float64), o2.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-3


def test_decode_batch_experts_calls_match_forward():
    """moe_mxfp4_experts on the decode path, with the caller's buckets (a
    checked copy of the pair list) and without them, equals moe_forward
    bitwise, with the pair list in the workspace (2400 pairs)."""
    t = torch()
    inp = synth.make_inputs(synth.Workload("experts_only", 300, 384, 40, 8, 256), seed=12)
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


def test_decode_batch_invariance():
    """Given the same routes, a token's decode output is bitwise the same in a
    300-token batch (workspace pair list), a 150-token and an 80-token batch
    (shared-memory pair list): above 64 tokens one set of kernels serves
    every batch size."""
    t = torch()
    wl = synth.Workload("invariance", 300, 512, 32, 8, 256)
    inp = synth.make_inputs(wl, seed=21)
    L = DeviceLayer(inp)
    out_all, ids, w = L.forward(path=1)
    t.cuda.synchronize()
    assert L.status() == 0
    for lo, n in ((100, 150), (7, 80)):
        shp = L.moe.shape(n, wl.H, wl.E, wl.I, wl.k)
        ws = t.empty(L.moe.workspace_bytes(n, wl.H, wl.E, wl.I, wl.k), dtype=t.uint8, device="cuda")
        out = t.zeros((n, wl.H), dtype=t.float32, device="cuda")
        L.moe.mxfp4_experts(shp, L.x[lo:lo + n].contiguous(), L.table.desc, ids[lo:lo + n].contiguous(),
                            w[lo:lo + n].contiguous(), None, None, out, False, ws, path=1)
        t.cuda.synchronize()
        assert L.moe.device_status(ws) == 0
        assert t.equal(out, out_all[lo:lo + n]), f"tokens {lo}..{lo + n - 1} differ"


def test_decode_batch_bad_pair_entry_is_flagged():
    """A caller pair list with an entry outside [0, T*k) is flagged
    (MOE_ERR_DEVICE_CHECK) on the decode path with the pair list in the
    workspace; that entry is not used; the next clean call is ok."""
    t = torch()
    inp = synth.make_inputs(synth.Workload("badpair", 300, 256, 24, 8, 128), seed=5)
    L = DeviceLayer(inp)
    ids, w, off, srt = L.route()
    wl = inp.wl
    out = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    bad = srt.clone()
    bad[17] = wl.T * wl.k + 5
    bad[1000] = -3
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, bad, out, False, L.ws, path=1)
    assert L.status() == L.moe.MOE_ERR_DEVICE_CHECK
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, srt, out, False, L.ws, path=1)
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), "after bad pair entry")


def test_router_split_contraction_routes():
    """The CUDA-core router GEMM (the tensor-core screen takes H % 64 == 0,
    so H = 4128 runs on it) splits its contraction when the batch has few
    tiles (here 16 splits: 100 tokens, 64 experts) and adds the splits'
    double-float partial sums in order; routes, weights and buckets match the
    oracle, with a per-expert bias."""
    from harness import check_buckets
    wl = synth.Workload("split_router", 100, 4128, 64, 8, 128)
    inp = synth.make_inputs(wl, seed=8)
    inp.br = (np.arange(wl.E, dtype=np.float32) % 7 - 3.0) * 0.05
    L = DeviceLayer(inp)
    ids, w, off, srt = L.route()
    torch().cuda.synchronize()
    assert L.status() == 0
    ids, w, off, srt = (a.cpu().numpy() for a in (ids, w, off, srt))
    check_route(inp, ids, w)
    check_buckets(ids, off, srt, wl.E)


@pytest.mark.parametrize("T,H,E", [(100, 4096, 64), (333, 1024, 200), (70, 512, 2048)],
                         ids=["T100_E64", "T333_E200_ragged", "T70_E2048"])
def test_router_screen_routes(T, H, E):
    """Batches above 64 tokens (bf16) are routed by the tensor-core screen
    plus exact scores for the candidate experts: routes and weights match the
    oracle (ids exact up to near-ties of the exact arithmetic), buckets are a
    stable sort, with a per-expert bias; ragged token and expert tiles, and
    2048 experts."""
    from harness import check_buckets
    wl = synth.Workload(f"screen_T{T}_E{E}", T, H, E, 16 if E >= 16 else 8, 128)
    inp = synth.make_inputs(wl, seed=31)
    inp.br = (np.arange(wl.E, dtype=np.float32) % 11 - 5.0) * 0.03
    L = DeviceLayer(inp)
    ids, w, off, srt = L.route()
    torch().cuda.synchronize()
    assert L.status() == 0
    ids, w, off, srt = (a.cpu().numpy() for a in (ids, w, off, srt))
    check_route(inp, ids, w)
    check_buckets(ids, off, srt, wl.E)


@pytest.mark.parametrize("T", [5, 200])
def test_decode_path_with_shared_expert(T):
    """A bf16 shared expert on the decode path (run after the routed experts
    on the prefill kernels, alone) matches the oracle, and agrees with the
    prefill path, which takes it with the routed tiles."""
    wl = synth.Workload(f"shared_T{T}", T, 256, 16, 4, 128, shared=True)
    inp = synth.make_inputs(wl, seed=4)
    L, out, ids, w = _check_forward(inp, wl.name, path=1)
    o2, _, _ = L.forward(path=2)
    torch().cuda.synchronize()
    assert L.status() == 0
    a, b = out.cpu().numpy().astype(np.float64), o2.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-3


def test_prefill_workload_decode_path_with_shared_expert():
    """The 512-token layer with the shared expert on the decode path (the
    automatic choice takes the prefill path at about 9 routed pairs per
    expert): the routed experts on the decode kernels, the shared expert on
    the prefill kernels; sampled tokens against the oracle."""
    import mxfp4_routed_expert_moe_gb300 as moe
    wl = synth.WORKLOADS["prefill"]
    assert moe.select_path(wl.T, wl.H, wl.E, wl.I, wl.k, shared=True) == moe.PATH_PREFILL
    inp = synth.make_inputs(wl)
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=moe.PATH_DECODE)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    toks = toks[np.linspace(0, toks.size - 1, 3).astype(int)]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), "prefill workload, decode path + shared")
