"""GPU parity of the prefill path (grouped MXFP4 GEMM on tcgen05 tensor cores)
against the fp64 oracle, through the C ABI: small shapes that span several
row, token and contraction tiles with ragged token tails, the bf16 shared
expert, accumulation into a residual, routes given by the caller, and the
full-size prefill workloads on sampled tokens."""
import numpy as np
import pytest

import synth
from harness import DeviceLayer, check_buckets, check_out, check_route, oracle_out, torch

pytestmark = pytest.mark.gpu

PREFILL = 2


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    t = torch()
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    import mxfp4_routed_expert_moe_gb300 as moe
    moe.lib()  # raises if the library is missing: no fallback


def _forward_check(inp, path=PREFILL, tokens=None, accumulate=False):
    L = DeviceLayer(inp)
    t = torch()
    wl = inp.wl
    residual = None
    out0 = None
    if accumulate:
        residual = synth.normal(synth.key(inp.seed, 999), wl.T * wl.H).reshape(wl.T, wl.H).astype(np.float32)
        out0 = t.from_numpy(residual).cuda()
    out, ids, w = L.forward(path=path, accumulate=accumulate, out=out0)
    t.cuda.synchronize()
    assert L.status() == 0, L.moe.status_string(L.status())
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    if tokens is not None:
        toks = np.intersect1d(toks, np.asarray(tokens))
    assert toks.size > 0
    ref = oracle_out(inp, toks, residual=residual)
    rel, mx = check_out(out.cpu().numpy()[toks], ref, wl.name)
    return L, rel, mx


# (T, H, E, k, I): several contraction slices (H/64, I/64), several 128-row
# tiles of I and H, ragged token tiles, experts with several token tiles.
SMALL = [
    (130, 256, 8, 2, 128),     # one row tile of I, 2 of H; ~32 tokens per expert
    (300, 384, 8, 2, 256),     # 6 slices of H, 3 row tiles of H, 2 of I
    (1000, 256, 4, 2, 128),    # ~500 tokens per expert: 4 token tiles, ragged tail
    (96, 512, 64, 4, 384),     # many experts with 0-12 tokens
    (70, 256, 16, 16, 128),    # k = E: every expert active, 70 tokens each
]


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "T{}_H{}_E{}_k{}_I{}".format(*s))
def test_prefill_small(shape):
    T, H, E, k, I = shape
    inp = synth.make_inputs(synth.Workload("pf_small", T, H, E, k, I))
    _, rel, mx = _forward_check(inp)
    print(f"{shape}: rel-L2 {rel:.2e}, max-abs/rms {mx:.2e}")


def test_prefill_shared_expert_small():
    inp = synth.make_inputs(synth.Workload("pf_shared", 200, 256, 8, 2, 256, shared=True))
    _forward_check(inp)


def test_prefill_accumulate_small():
    inp = synth.make_inputs(synth.Workload("pf_acc", 150, 256, 8, 2, 128))
    _forward_check(inp, accumulate=True)


def test_prefill_short_batch():
    # The prefill path on a batch the automatic choice would send to decode.
    inp = synth.make_inputs(synth.Workload("pf_short", 5, 256, 8, 2, 128))
    _forward_check(inp)


def test_prefill_matches_decode_path():
    """Both expert paths agree with each other (and the oracle) on one batch."""
    inp = synth.make_inputs(synth.Workload("pf_vs_dec", 64, 512, 16, 4, 256))
    L = DeviceLayer(inp)
    t = torch()
    o1, i1, w1 = L.forward(path=1)
    o2, i2, w2 = L.forward(path=PREFILL)
    t.cuda.synchronize()
    assert L.status() == 0
    # The two paths route with different kernels (GEMV vs GEMM): same ids,
    # weights equal within the route tolerance.
    assert t.equal(i1, i2)
    assert float((w1 - w2).abs().max()) <= 2e-6
    a, b = o1.cpu().numpy().astype(np.float64), o2.cpu().numpy().astype(np.float64)
    assert np.linalg.norm(a - b) / np.linalg.norm(a) < 1e-3


def test_prefill_experts_given_route():
    """moe_mxfp4_experts on the prefill path with the caller's buckets and with
    buckets rebuilt from ids."""
    inp = synth.make_inputs(synth.Workload("pf_given", 257, 256, 8, 2, 128))
    L = DeviceLayer(inp)
    t = torch()
    wl = inp.wl
    ids, w, off, srt = L.route()
    outs = []
    for given in (True, False):
        out = t.zeros((wl.T, wl.H), dtype=t.float32, device="cuda")
        L.moe.mxfp4_experts(L.shape, L.x, L.table.desc, ids, w, off if given else None, srt if given else None,
                            out, False, L.ws, path=PREFILL)
        outs.append(out)
    t.cuda.synchronize()
    assert L.status() == 0
    check_buckets(ids.cpu().numpy(), off.cpu().numpy(), srt.cpu().numpy(), wl.E)
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    ref = oracle_out(inp, toks)
    for out in outs:
        check_out(out.cpu().numpy()[toks], ref, "given route")


def test_prefill_skewed_load():
    """One expert takes every token (router bias), the rest share the second
    slot: a 600-token bucket next to small ones."""
    wl = synth.Workload("pf_skew", 600, 256, 32, 2, 128)
    inp = synth.make_inputs(wl)
    br = np.zeros(wl.E, dtype=np.float32)
    br[7] = 100.0
    inp.br = br
    _forward_check(inp)


@pytest.mark.parametrize("name,tokens", [("prefill", [0, 255, 511]), ("long", [0, 2047, 4095])])
def test_prefill_full_size_sampled(name, tokens):
    """Full-size prefill workloads in the launch configuration the benchmark
    times; the oracle checks a few tokens (routing for all of them)."""
    inp = synth.make_inputs(synth.WORKLOADS[name])
    _, rel, mx = _forward_check(inp, tokens=tokens)
    print(f"{name}: rel-L2 {rel:.2e}, max-abs/rms {mx:.2e} on tokens {tokens}")


def test_prefill_unaligned_codes_flagged_not_read():
    """The prefill gate/up GEMM reads code matrices with tensor-map copies,
    which need 32-byte aligned rows: an expert whose gate codes are 16- but not
    32-byte aligned is flagged (MOE_ERR_DEVICE_CHECK) and its codes are never
    copied; the next clean call on the same workspace matches the oracle."""
    wl = synth.Workload("pf_unaligned", 130, 256, 8, 2, 128)
    inp = synth.make_inputs(wl, seed=8)
    L = DeviceLayer(inp)
    good = L.table.desc.clone()
    bad = good.clone()
    bad[3, 0] += 16  # gate.q of expert 3: 16-byte aligned, not 32
    L.table.desc.copy_(bad)
    L.forward(path=PREFILL)
    torch().cuda.synchronize()
    assert L.status() == L.moe.MOE_ERR_DEVICE_CHECK
    L.table.desc.copy_(good)
    out, ids, w = L.forward(path=PREFILL)
    torch().cuda.synchronize()
    assert L.status() == 0
    _, same = check_route(inp, ids.cpu().numpy(), w.cpu().numpy())
    toks = np.nonzero(same)[0]
    check_out(out.cpu().numpy()[toks], oracle_out(inp, toks), "after unaligned codes")
