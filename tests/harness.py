"""Shared helpers of the GPU parity tests: put a workload on the device, call
the library through its C ABI, and compare with the fp64 oracle."""
from __future__ import annotations

import numpy as np

import oracle
import synth

# Tolerances (fixed by the parity contract): ids and buckets exact; route
# weights |dw| <= 1e-6; outputs rel-L2 <= 1e-3 and max-abs <= 1e-2 * rms(out).
W_TOL = 1e-6
REL_L2_TOL = 1e-3
MAXABS_RMS_TOL = 1e-2
DEVICE_FILL_BYTES = 256 << 20  # experts above this total are made by the device generator


def torch():
    import torch as _t
    return _t


class DeviceLayer:
    """A workload's inputs resident on the GPU (experts in one ExpertTable)."""

    def __init__(self, inp: synth.LayerInputs, device: str = "cuda"):
        import mxfp4_routed_expert_moe_gb300 as moe
        t = torch()
        wl = inp.wl
        self.inp, self.wl, self.device = inp, wl, device
        self.moe = moe
        self.table = moe.ExpertTable(wl.E, wl.H, wl.I, device)
        if wl.E * wl.expert_bytes > DEVICE_FILL_BYTES:
            offs, stride = synth.expert_blob_layout(wl)
            assert (offs, stride) == moe.ExpertTable.blob_layout(wl.H, wl.I)
            synth.fill_experts_device(inp, self.table.blob.data_ptr(), t.cuda.current_stream().cuda_stream)
        else:
            for e in range(wl.E):
                self.table.load_host(e, inp.expert(e))
        if wl.x_dtype == "f32":
            self.x = t.from_numpy(inp.x).to(device)
        else:
            self.x = t.from_numpy(inp.x.view(np.int16)).to(device).view(t.bfloat16)
        self.wr = t.from_numpy(inp.wr).to(device)
        self.br = None if inp.br is None else t.from_numpy(inp.br).to(device)
        self.shared = None
        if inp.shared is not None:
            self.shared = tuple(t.from_numpy(a.view(np.int16)).to(device).view(t.bfloat16) for a in inp.shared)
        self.shape = moe.shape(wl.T, wl.H, wl.E, wl.I, wl.k)
        self.ws = t.empty(moe.workspace_bytes(wl.T, wl.H, wl.E, wl.I, wl.k), dtype=t.uint8, device=device)

    def forward(self, path=0, accumulate=False, out=None):
        t = torch()
        wl = self.wl
        if out is None:
            out = t.zeros((wl.T, wl.H), dtype=t.float32, device=self.device)
        ids = t.empty((wl.T, wl.k), dtype=t.int32, device=self.device)
        w = t.empty((wl.T, wl.k), dtype=t.float32, device=self.device)
        self.moe.forward(self.shape, self.x, self.wr, self.br, self.table.desc, self.shared, out, accumulate,
                         self.ws, ids_out=ids, w_out=w, path=path)
        return out, ids, w

    def route(self):
        t = torch()
        wl = self.wl
        ids = t.empty((wl.T, wl.k), dtype=t.int32, device=self.device)
        w = t.empty((wl.T, wl.k), dtype=t.float32, device=self.device)
        off = t.empty(wl.E + 1, dtype=t.int32, device=self.device)
        srt = t.empty(wl.T * wl.k, dtype=t.int32, device=self.device)
        self.moe.route(self.shape, self.x, self.wr, self.br, ids, w, off, srt, self.ws)
        return ids, w, off, srt

    def status(self):
        return self.moe.device_status(self.ws)


def oracle_route(inp: synth.LayerInputs):
    """Oracle scores, ids and weights, and per-score error bounds of the
    library's router arithmetic: products are summed in fp32 in chunks of at
    most 16 (error <= gamma_16 * sum |x W| over the chunk) and the chunk sums
    are carried in double-float (hi + lo), whose own error is below
    2^-40 * sum |x W|.  gamma_n = n u / (1 - n u), u = 2^-24."""
    wl = inp.wl
    s = oracle.router_logits(inp.x, inp.wr, inp.br)
    ids, w, _ = oracle.topk(s, wl.k)
    absx = np.abs(inp.x_f32).astype(np.float32)
    absw = np.abs(inp.wr).astype(np.float32)
    mag = (absx @ absw.T).astype(np.float64)
    if inp.br is not None:
        mag += np.abs(inp.br.astype(np.float64))[None, :]
    u = 2.0 ** -24
    n = 16
    bound = ((n * u / (1 - n * u)) + 2.0 ** -40) * mag * 1.01  # 1% margin: mag is evaluated in fp32
    return s, ids, w, bound


def check_route(inp, ids_gpu, w_gpu, w_tol=W_TOL):
    """Exact route parity up to near-ties.

    Oracle-sorted scores are split into tie groups: consecutive entries whose
    gap is below the sum of their error bounds.  At every slot j the GPU's
    expert must lie in the same tie group as the oracle's (so ids are equal
    unless two scores are indistinguishable in fp32).  Weights must agree
    within W_TOL whenever the GPU selected the oracle's set.  Returns the mask
    of tokens that had a near-tie among their first k+1 scores and the mask of
    tokens whose selected set equals the oracle's."""
    wl = inp.wl
    s, ids_o, w_o, bound = oracle_route(inp)
    T, k, E = wl.T, wl.k, wl.E
    amb = np.zeros(T, dtype=bool)
    same = np.zeros(T, dtype=bool)
    worst = 0.0
    for t in range(T):
        order = np.array(sorted(range(E), key=lambda e: (-s[t, e], e)))
        ss, bb = s[t, order], bound[t, order]
        group = np.zeros(E, dtype=np.int64)
        g = 0
        for j in range(1, E):
            if ss[j - 1] - ss[j] >= bb[j - 1] + bb[j]:
                g += 1
            group[j] = g
        gid = np.empty(E, dtype=np.int64)
        gid[order] = group
        amb[t] = len(set(group[: min(k + 1, E)])) < min(k + 1, E)
        assert len(set(ids_gpu[t])) == k, f"token {t}: repeated ids {ids_gpu[t]}"
        for j in range(k):
            assert gid[ids_gpu[t, j]] == gid[ids_o[t, j]], f"token {t} slot {j}: {ids_gpu[t]} vs {ids_o[t]}"
        if not amb[t]:
            assert np.array_equal(ids_gpu[t], ids_o[t])
        same[t] = set(ids_gpu[t]) == set(ids_o[t])
        if same[t]:
            ref = dict(zip(ids_o[t], w_o[t]))
            dw = max(abs(float(w_gpu[t, j]) - ref[ids_gpu[t, j]]) for j in range(k))
            worst = max(worst, dw)
    assert worst <= w_tol, f"route weight error {worst:.3e} > {w_tol}"
    return amb, same


def check_buckets(ids, offsets, sorted_idx, E):
    """Properties of the bucket layout of given ids: a stable counting sort."""
    T, k = ids.shape
    counts = np.bincount(ids.ravel(), minlength=E)
    np.testing.assert_array_equal(offsets, np.concatenate([[0], np.cumsum(counts)]))
    assert sorted(sorted_idx.tolist()) == list(range(T * k))
    flat = ids.ravel()
    for e in range(E):
        seg = sorted_idx[offsets[e]:offsets[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)


def check_out(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = got.astype(np.float64)
    err = got - ref
    rel = np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300)
    rms = np.sqrt(np.mean(ref * ref))
    mx = np.abs(err).max()
    assert rel <= REL_L2_TOL, f"{what} rel-L2 {rel:.3e} > {REL_L2_TOL}"
    assert mx <= MAXABS_RMS_TOL * rms, f"{what} max-abs {mx:.3e} > {MAXABS_RMS_TOL} * rms {rms:.3e}"
    return rel, mx / rms


def oracle_out(inp, tokens, residual=None):
    out, ids, w = oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, inp.wl.E, inp.wl.I, inp.wl.k,
                                    np.asarray(tokens), shared=inp.shared, residual=residual)
    return out
