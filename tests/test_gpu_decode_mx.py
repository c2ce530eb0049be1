"""GPU parity of the persistent block-scaled decode kernel (MOE_PATH_DECODE_MX:
routing, gate/up + SwiGLU, down and the slot-ordered combine in one launch
on tcgen05 block-scaled MMAs) against the fp64 oracle, through the C ABI:
the 1-token and 8-token layers at full size, I = 1536, small shapes with an
odd number of down slices and several items per CTA, batch invariance,
experts-only calls, the residual, special E8M0 codes, a misaligned
descriptor and the shared expert."""
import numpy as np
import pytest

import synth
from harness import DeviceLayer, check_out, check_route, oracle_out, torch

pytestmark = pytest.mark.gpu

MX = 3  # MOE_PATH_DECODE_MX


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_routed_expert_moe_gb300 as moe
    moe.lib()  # raises if the library is missing: no fallback
    assert moe.PATH_DECODE_MX == MX


def _forward_checked(inp, name, sample=None):
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=MX)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    assert toks.size >= inp.wl.T - 1
    if sample:
        toks = toks[np.linspace(0, toks.size - 1, sample).astype(int)]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), name)
    return L, out, ids, w


def test_select_path_takes_explicit_choice_only():
    import mxfp4_routed_expert_moe_gb300 as moe
    wl = synth.WORKLOADS["decode"]
    assert moe.select_path(wl.T, wl.H, wl.E, wl.I, wl.k, path=MX) == MX
    assert moe.select_path(wl.T, wl.H, wl.E, wl.I, wl.k) == moe.PATH_DECODE
    with pytest.raises(moe.MoeError):
        moe.select_path(9, wl.H, wl.E, wl.I, wl.k, path=MX)  # more than 8 tokens


@pytest.mark.parametrize("name", ["decode", "wide", "decode_i1536", "decode_e32"])
def test_forward_parity_full_size(name):
    inp = synth.make_inputs(synth.WORKLOADS[name])
    _forward_checked(inp, name, sample=None if inp.wl.T <= 8 else 3)


SMALL = [
    # name, T, H, E, k, I
    ("t3_h512_i256", 3, 512, 16, 4, 256),
    ("t8_i384_odd_down_slices", 8, 256, 64, 8, 384),
    ("t5_e4_all_shared", 5, 384, 4, 4, 256),
    ("t2_k32", 2, 256, 40, 32, 256),
]


@pytest.mark.parametrize("name,T,H,E,k,I", SMALL)
def test_forward_parity_small(name, T, H, E, k, I):
    inp = synth.make_inputs(synth.Workload(name, T, H, E, k, I), seed=6)
    inp.br = (np.arange(E, dtype=np.float32) % 5 - 2.0) * 0.04
    _forward_checked(inp, name)


def test_agrees_with_decode_path():
    """Same routes; outputs of the two decode kernel families agree to the
    oracle tolerance."""
    inp = synth.make_inputs(synth.WORKLOADS["wide"])
    L = DeviceLayer(inp)
    a, ids_a, _ = L.forward(path=MX)
    b, ids_b, _ = L.forward(path=1)
    torch().cuda.synchronize()
    assert L.status() == 0
    assert torch().equal(ids_a, ids_b)
    a, b = a.cpu().numpy().astype(np.float64), b.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(b) < 1e-3


def test_batch_invariance_wide_vs_single():
    """A token's route and output in an 8-token step are bitwise those of its
    1-token step."""
    t = torch()
    wl = synth.WORKLOADS["wide"]
    inp = synth.make_inputs(wl)
    L = DeviceLayer(inp)
    out8, ids8, w8 = L.forward(path=MX)
    shp1 = L.moe.shape(1, wl.H, wl.E, wl.I, wl.k)
    ws1 = t.empty(L.moe.workspace_bytes(1, wl.H, wl.E, wl.I, wl.k), dtype=t.uint8, device="cuda")
    for tok in range(wl.T):
        x1 = L.x[tok:tok + 1].contiguous()
        out1 = t.zeros((1, wl.H), dtype=t.float32, device="cuda")
        ids1 = t.empty((1, wl.k), dtype=t.int32, device="cuda")
        w1 = t.empty((1, wl.k), dtype=t.float32, device="cuda")
        L.moe.forward(shp1, x1, L.wr, None, L.table.desc, None, out1, False, ws1, ids_out=ids1, w_out=w1, path=MX)
        t.cuda.synchronize()
        assert L.moe.device_status(ws1) == 0
        assert t.equal(ids1[0], ids8[tok])
        assert t.equal(w1[0], w8[tok])
        assert t.equal(out1[0], out8[tok]), f"token {tok} differs"


def test_experts_only_calls_match_forward():
    """moe_mxfp4_experts on this path, with the caller's buckets and without
    them, equals moe_forward bitwise."""
    t = torch()
    inp = synth.make_inputs(synth.WORKLOADS["wide"])
    L = DeviceLayer(inp)
    out_f, _, _ = L.forward(path=MX)
    ids, w, off, srt = L.route()
    wl = inp.wl
    out_a = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    out_b = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off, srt, out_a, False, L.ws, path=MX)
    L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, None, None, out_b, False, L.ws, path=MX)
    t.cuda.synchronize()
    assert L.status() == 0
    assert t.equal(out_a, out_f)
    assert t.equal(out_b, out_f)


def test_accumulate_adds_residual():
    t = torch()
    inp = synth.make_inputs(synth.Workload("acc_mx", 4, 256, 8, 2, 256), seed=2)
    L = DeviceLayer(inp)
    out0, _, _ = L.forward(path=MX)
    res = t.randn(out0.shape, device="cuda", generator=t.Generator("cuda").manual_seed(3))
    out1 = res.clone()
    L.forward(path=MX, accumulate=True, out=out1)
    t.cuda.synchronize()
    assert t.equal(out1, out0 + res)
    check_out(out1.cpu().numpy(), oracle_out(inp, np.arange(inp.wl.T), residual=res.cpu().numpy()), "accumulate")


def test_special_scale_codes():
    """E8M0 code 0 (2^-127) and 255 (NaN) in gate/up and down scales: finite
    rows match the oracle, rows of tokens routed to an expert with a NaN scale
    come out NaN where the oracle's do."""
    wl = synth.Workload("mx_specials", 6, 256, 8, 2, 256)
    inp = synth.make_inputs(wl, seed=11)
    for e in range(wl.E):
        ex = inp.expert(e)
        ex["gate_s"].reshape(-1)[::7] = 0
        ex["up_s"].reshape(-1)[3::11] = 0
        ex["down_s"].reshape(-1)[5::13] = 0
    inp.expert(3)["up_s"].reshape(-1)[5] = 255
    inp.expert(6)["down_s"].reshape(-1)[40] = 255
    L = DeviceLayer(inp)
    out, ids, w = L.forward(path=MX)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    ref = oracle_out(inp, toks)
    got = out.cpu().numpy()[toks].astype(np.float64)
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    fin = ~np.isnan(ref)
    assert fin.any()
    check_out(np.where(fin, got, 0.0), np.where(fin, ref, 0.0), "special scales")


def test_misaligned_expert_descriptor_is_flagged_not_read():
    """An expert whose codes are not 32-byte aligned gets no tensor map: the
    call reports MOE_ERR_DEVICE_CHECK without reading them; the next clean
    call is ok."""
    wl = synth.Workload("mx_misal", 4, 256, 8, 2, 256)
    inp = synth.make_inputs(wl, seed=4)
    inp.br = np.zeros(wl.E, dtype=np.float32)
    inp.br[3] = 100.0
    L = DeviceLayer(inp)
    good = L.table.desc.clone()
    bad = good.clone()
    bad[3, 0] += 16  # gate.q of expert 3: 16- but not 32-byte aligned
    L.table.desc.copy_(bad)
    L.forward(path=MX)
    torch().cuda.synchronize()
    assert L.status() == L.moe.MOE_ERR_DEVICE_CHECK
    L.table.desc.copy_(good)
    out, ids, w = L.forward(path=MX)
    torch().cuda.synchronize()
    assert L.status() == 0
    check_out(out.cpu().numpy(), oracle_out(inp, np.arange(wl.T)), "after misaligned")


def test_shared_expert():
    """The shared expert (prefill kernels, after the persistent kernel) on
    this path matches the oracle."""
    wl = synth.Workload("mx_shared", 3, 256, 16, 4, 256, shared=True)
    inp = synth.make_inputs(wl, seed=4)
    _forward_checked(inp, wl.name)
