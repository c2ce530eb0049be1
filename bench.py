"""Benchmark of the routed MXFP4 MoE layer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode|wide|batch256|prefill|long|decode_i1536|tiny]
    python bench.py --sweep [--sweep-i 1408|1536] [--steps K]

A step is one pass of the whole layer (moe_forward: router, top-k, bucketing,
MXFP4 experts, combine) over one batch of the workload.  The default workload
is 1-token decode (H=7168, 896 MXFP4 experts, top-16, I=1408).  Inputs are
synthetic and seeded; all 896 experts are resident in HBM.  Prints ONE JSON
line (rank 0).  For N > 1 (torchrun) every rank runs an independent replica
of the workload on its own GPU (the layer has no exchange step here), the
time is the max over ranks and `value` counts the tokens of all ranks.

With the default workload the same line also carries `prefill_long`: the
4096-token Zipf prefill (tensor-core grouped GEMMs) timed the same way, with
its own roofline, parity, cpu_baseline and e2e figures.

Before anything is timed, the layer's output on a few sampled tokens is
checked against the fp64 oracle (ids, route weights, outputs within the
parity tolerances); a mismatch prints the line with "value": null and exits 1.

--impl reference times the fp64 CPU oracle (the reference arm) on the host
cores, each step a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s & weight GB/s (decode) / TFLOP/s (prefill) vs GB300 roofline"
L2_FLUSH_BYTES = 256 << 20   # > 2x the 129 MB L2
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=1000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode")
    ap.add_argument("--path", default="auto", choices=["auto", "decode", "prefill", "decode_mx"],
                    help="expert path of the workload (default: the library's own choice)")
    ap.add_argument("--no-prefill-leg", action="store_true",
                    help="with the default 1-token decode workload, skip the 4096-token prefill leg")
    ap.add_argument("--no-graph", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true",
                    help="time both paths over batch sizes T (one JSON line per T and path) instead of one workload")
    ap.add_argument("--sweep-i", type=int, default=1408, choices=[1408, 1536], help="intermediate size of the sweep")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's time: every replica ran the same work, so the job
    took as long as its slowest member."""
    if world <= 1:
        return ms
    import torch
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(world: int, tokens_per_replica: int, ms: float) -> float:
    """Whole-job throughput of `world` replicas, each processing
    `tokens_per_replica` tokens per step of `ms` milliseconds (weak scaling)."""
    return world * tokens_per_replica / (ms / 1000.0)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


# ------------------------------------------------------------------ clocks --
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ device --
class Layer:
    """The workload resident on one GPU, called through the C ABI."""

    def __init__(self, wl, device: str, table=None, path=None):
        """wl: a workload or its name.  table: an ExpertTable already filled
        with this workload's experts (they depend on H, E, I and the seed
        only), else one is made and filled.  path: the library's path
        selector (default: its own choice by T)."""
        import torch

        import mxfp4_routed_expert_moe_gb300 as moe
        import synth
        self.torch, self.moe, self.synth = torch, moe, synth
        self.wl = wl = synth.WORKLOADS[wl] if isinstance(wl, str) else wl
        self.inp = inp = synth.make_inputs(wl)
        self.device = device
        self.path = moe.PATH_AUTO if path is None else path
        offs, stride = synth.expert_blob_layout(wl)
        assert (offs, stride) == moe.ExpertTable.blob_layout(wl.H, wl.I)
        if table is None:
            table = moe.ExpertTable(wl.E, wl.H, wl.I, device)
            synth.fill_experts_device(inp, table.blob.data_ptr(), torch.cuda.current_stream().cuda_stream)
        self.table = table
        if wl.x_dtype == "f32":
            self.x_host = torch.from_numpy(inp.x).pin_memory()
        else:
            self.x_host = torch.from_numpy(inp.x.view("int16")).view(torch.bfloat16).pin_memory()
        self.x = self.x_host.to(device)
        self.wr = torch.from_numpy(inp.wr).to(device)
        self.br = None if inp.br is None else torch.from_numpy(inp.br).to(device)
        self.shared = None
        if inp.shared is not None:
            self.shared = tuple(torch.from_numpy(a.view("int16")).view(torch.bfloat16).to(device) for a in inp.shared)
        self.shape = moe.shape(wl.T, wl.H, wl.E, wl.I, wl.k)
        self.ws = torch.empty(moe.workspace_bytes(wl.T, wl.H, wl.E, wl.I, wl.k), dtype=torch.uint8, device=device)
        self.out = torch.zeros((wl.T, wl.H), dtype=torch.float32, device=device)
        self.out_host = torch.empty((wl.T, wl.H), dtype=torch.float32).pin_memory()
        self.ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device=device)
        self.w = torch.empty((wl.T, wl.k), dtype=torch.float32, device=device)
        self.flush_buf = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_read = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=device)
        self.flush_sink = torch.empty((), dtype=torch.float32, device=device)
        torch.cuda.synchronize()

    def step(self):
        self.moe.forward(self.shape, self.x, self.wr, self.br, self.table.desc, self.shared, self.out, False,
                         self.ws, ids_out=self.ids, w_out=self.w, path=self.path)

    def flush_l2(self):
        # Write a buffer larger than L2, then read another one: the step
        # starts with an L2 holding only clean lines of unrelated data (the
        # write-backs of the written buffer happen here, not in the step).
        self.flush_buf.fill_(1.0)
        torch_ = self.torch
        torch_.amax(self.flush_read, dim=0, out=self.flush_sink)

    @property
    def decode_path(self) -> bool:
        wl, moe = self.wl, self.moe
        dt = moe.DT_F32 if wl.x_dtype == "f32" else moe.DT_BF16
        return moe.select_path(wl.T, wl.H, wl.E, wl.I, wl.k, dt, self.shared is not None,
                               self.path) in (moe.PATH_DECODE, moe.PATH_DECODE_MX)

    @property
    def persistent_decode(self) -> bool:
        """The explicit persistent block-scaled decode kernel (routing, gate/up,
        down and combine in one launch after the router)."""
        return self.path == self.moe.PATH_DECODE_MX

    def launches_per_step(self) -> int:
        # prefill: routing (see _router_launches), bucket count, bucket scatter, pair positions,
        # x->E4M3 rows, item tables, code maps, block-scaled gate/up, h->E4M3, block-scaled down; the shared
        # expert adds x->fp16, its row shifts, its gate/up, h->fp16 and its down
        if self.decode_path:
            # shared expert: x->fp16, its row shifts, item tables, and the two prefill GEMMs (with
            # the h->fp16 pass between them) on its tiles alone
            sh = 6 if self.shared is not None else 0
            if self.persistent_decode:
                return 2 + sh  # router (+ E4M3 activation terms, counters), the persistent kernel
            if self.wl.T <= self.moe.DECODE_MAX_T:
                return 3 + sh  # router (+ f16 activations), gate/up (+ fused top-k/bucketing), down (+ fused combine)
            # routing (below), bucket count, bucket scatter, x->fp16, gate/up, down, combine
            return 6 + self._router_launches() + sh
        return 9 + self._router_launches() + (5 if self.shared is not None else 0)

    def _router_launches(self) -> int:
        """Routing kernels of a batch above 64 tokens: the tensor-core screen (W split, screen
        GEMM, exact candidate scores with the top-k) for bf16 x, H % 64 == 0 and E <= 4096; else
        the CUDA-core GEMM (and its split reduction) and the top-k."""
        wl = self.wl
        if wl.x_dtype != "f32" and wl.H % 64 == 0 and wl.E <= 4096:
            return 3
        return 1 + (1 if self._router_splits() > 1 else 0) + 1

    def _router_splits(self) -> int:
        """Splits of the router GEMM's contraction (the library's rule)."""
        wl = self.wl
        if wl.T <= self.moe.DECODE_MAX_T:
            return 1
        tiles = ((wl.E + 63) // 64) * ((wl.T + 63) // 64)
        return max(1, min(-(-456 // tiles), wl.H // 256, 16))

    def dominant_stage(self):
        return self.moe.STAGE_GATEUP if self.decode_path else self.moe.STAGE_PF_GATEUP

    def active_experts(self) -> int:
        return len(set(self.ids.cpu().numpy().ravel().tolist()))

    def algorithmic_bytes_step(self, n_active: int) -> int:
        wl = self.wl
        xb = wl.T * wl.H * (4 if wl.x_dtype == "f32" else 2)
        b = n_active * wl.expert_bytes + wl.E * wl.H * 4 + xb + wl.T * wl.H * 4
        if self.shared is not None:
            b += 3 * wl.H * wl.I * 2
        return b

    def algorithmic_bytes_gateup(self, n_active: int) -> int:
        wl = self.wl
        xb = wl.T * wl.H * (4 if wl.x_dtype == "f32" else 2)
        return n_active * 2 * (wl.I * wl.H // 2 + wl.I * wl.H // 32) + xb + wl.T * wl.k * wl.I * 4

    def flops_gateup(self) -> int:
        """Algorithmic FLOPs of the prefill gate/up GEMM launch: routed pairs
        (and the shared expert) x 2 matrices x H x I multiply-adds."""
        wl = self.wl
        rows = wl.T * wl.k + (wl.T if self.shared is not None else 0)
        return 2 * rows * 2 * wl.H * wl.I

    def flops_step(self) -> int:
        return self.wl.T * self.wl.flops_per_token


def time_steps(layer, steps, warmup, use_graph):
    """Device time of each of `steps` steps (ms), L2 flushed before each."""
    torch = layer.torch
    fn = layer.step
    graph = None
    if use_graph:
        layer.step()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            layer.step()
        torch.cuda.current_stream().wait_stream(s)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            layer.step()
        fn = graph.replay
    for _ in range(warmup):
        layer.flush_l2()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        layer.flush_l2()
        a.record()
        fn()
        b.record()
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in ev], graph


def time_stage(layer, stage, reps):
    """Mean duration (ms) of one stage's kernel, bracketed by events the
    library records on the launching stream (profiling hook)."""
    torch = layer.torch
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record(); b.record()  # materialise the events
    torch.cuda.synchronize()
    times = []
    layer.moe.profile_events(stage, a, b)
    try:
        for _ in range(reps):
            layer.flush_l2()
            layer.step()
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b))
    finally:
        layer.moe.profile_events(stage, None, None)
    return statistics.mean(times)


def stage_breakdown(layer, reps=20):
    """Mean device time (ms) of each kernel stage of one step (profiling
    hook), and of an experts-only call given the route."""
    moe, torch = layer.moe, layer.torch
    out = {}
    stages = ([("router", moe.STAGE_ROUTE), ("gate_up", moe.STAGE_GATEUP), ("down", moe.STAGE_DOWN)]
              if layer.decode_path else
              [("router", moe.STAGE_ROUTE), ("gate_up", moe.STAGE_PF_GATEUP), ("down", moe.STAGE_PF_DOWN)])
    for name, st in stages:
        try:
            out[name] = time_stage(layer, st, reps)
        except Exception as exc:  # stage not launched on this path
            out[name] = None
    wl = layer.wl
    ids = torch.empty((wl.T, wl.k), dtype=torch.int32, device=layer.device)
    w = torch.empty((wl.T, wl.k), dtype=torch.float32, device=layer.device)
    off = torch.empty(wl.E + 1, dtype=torch.int32, device=layer.device)
    srt = torch.empty(wl.T * wl.k, dtype=torch.int32, device=layer.device)
    moe.route(layer.shape, layer.x, layer.wr, layer.br, ids, w, off, srt, layer.ws)
    o2 = torch.zeros_like(layer.out)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t = []
    for _ in range(reps):
        layer.flush_l2()
        a.record()
        moe.mxfp4_experts(layer.shape, layer.x, layer.table.desc, ids, w, off, srt, o2, False, layer.ws)
        b.record()
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    out["experts_call_given_route"] = statistics.mean(t)
    t = []
    for _ in range(reps):
        layer.flush_l2()
        a.record()
        moe.route(layer.shape, layer.x, layer.wr, layer.br, ids, w, off, srt, layer.ws)
        b.record()
        torch.cuda.synchronize()
        t.append(a.elapsed_time(b))
    out["route_call"] = statistics.mean(t)
    return out


def time_e2e(layer, steps, warmup, graph):
    """Same metric through the C ABI with host buffers: pinned H2D of the
    step's activations, the layer, D2H of its output, all inside the timing."""
    torch = layer.torch
    fn = graph.replay if graph is not None else layer.step
    for _ in range(warmup):
        layer.flush_l2()
        layer.x.copy_(layer.x_host, non_blocking=True)
        fn()
        layer.out_host.copy_(layer.out, non_blocking=True)
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for a, b in ev:
        layer.flush_l2()
        a.record()
        layer.x.copy_(layer.x_host, non_blocking=True)
        fn()
        layer.out_host.copy_(layer.out, non_blocking=True)
        b.record()
    torch.cuda.synchronize()
    return statistics.mean(a.elapsed_time(b) for a, b in ev)


FP8_OVER_BF16 = 2.0  # nominal dense fp8 / bf16 tensor rates of GB300 (4.5 / 2.25 PFLOP/s)

KERNEL_SOURCES = {
    "dec_gateup": ("common.cuh", "async.cuh", "route_small.cuh", "decode.cu"),
    "pf_gateup": ("common.cuh", "async.cuh", "tcgen05.cuh", "prefill.cu"),
}


def source_sha(kernel: str) -> str:
    src = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        p = os.path.join(ROOT, "mxfp4_routed_expert_moe_gb300", "csrc", f)
        if os.path.exists(p):
            src.update(open(p, "rb").read())
    return src.hexdigest()[:16]


def traffic_from_profiles(kernel: str, workload: str):
    """DRAM bytes per launch recorded by an ncu capture (a profiles/*.md line
    `traffic[<kernel>:<workload>]: bytes_per_launch=<n> source_sha=<sha>`), or
    None when the kernel's sources changed since the capture."""
    sha = source_sha(kernel)
    tag = f"{kernel}:{workload}"
    pdir = os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, sha
    for f in sorted(os.listdir(pdir)):
        if not f.endswith(".md"):
            continue
        text = open(os.path.join(pdir, f)).read()
        m = re.search(rf"traffic\[{re.escape(tag)}\]: bytes_per_launch=(\d+) source_sha=(\w+)", text)
        if m and m.group(2) == sha:
            return int(m.group(1)), sha
    return None, sha


# ------------------------------------------------------------------- oracle --
def cpu_model() -> str:
    """The host CPU's model name (lscpu, else /proc/cpuinfo)."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def sample_tokens(inp, n):
    """Up to n tokens spread over the batch whose oracle route has no near-tie:
    every gap between consecutive scores among the first k+1 is at least twice
    the error bound of the library's router arithmetic (products summed in fp32
    in chunks of at most 16, chunk sums carried in double-float)."""
    import numpy as np

    import oracle
    wl = inp.wl
    u = 2.0 ** -24
    gam = 16 * u / (1 - 16 * u) + 2.0 ** -40
    absw = np.abs(inp.wr).astype(np.float64)
    toks = []
    for i in range(8 * n + 16):
        tok = (i * 7919) % wl.T
        if tok in toks:
            continue
        sc = oracle.router_logits(inp.x[[tok]], inp.wr, inp.br)
        _, _, margin = oracle.topk(sc, wl.k)
        mag = absw @ np.abs(inp.x_f32[tok]).astype(np.float64)
        if inp.br is not None:
            mag = mag + np.abs(inp.br.astype(np.float64))
        if wl.k >= wl.E or margin[0] >= 2.0 * gam * 1.01 * float(mag.max()):
            toks.append(tok)
        if len(toks) == n:
            break
    return toks or [0]


def parity_check(layer, ntok):
    """The output of the layer's last step on sampled tokens against the fp64
    oracle: ids equal, route weights within 1e-6, outputs within rel-L2 1e-3
    and max-abs 1e-2 * rms (the parity tolerances)."""
    import numpy as np

    import oracle
    inp, wl = layer.inp, layer.wl
    toks = sample_tokens(inp, ntok)
    t0 = time.perf_counter()
    ref, rids, rw = oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, np.array(toks),
                                      shared=inp.shared, nthreads=oracle.default_threads())
    dt = time.perf_counter() - t0
    got = layer.out.cpu().numpy()[toks].astype(np.float64)
    ids = layer.ids.cpu().numpy()[toks]
    w = layer.w.cpu().numpy()[toks]
    ids_ok = bool(np.array_equal(ids, rids))
    dw = float(np.abs(w.astype(np.float64) - rw).max()) if ids_ok else None
    err = got - ref
    rel = float(np.linalg.norm(err) / max(float(np.linalg.norm(ref)), 1e-300))
    rms = float(np.sqrt(np.mean(ref * ref)))
    mx = float(np.abs(err).max()) / rms if rms > 0 else float("inf")
    ok = bool(ids_ok and dw <= 1e-6 and rel <= 1e-3 and mx <= 1e-2)
    return {"ok": ok, "when": "before the timed region", "tokens": [int(t) for t in toks], "ids_equal": ids_ok,
            "max_abs_dw": dw, "rel_l2": rel, "max_abs_over_rms": mx, "oracle_seconds": round(dt, 3)}


def cpu_baseline(layer, seconds: float):
    """The fp64 oracle as it stands on the host cores, on a bounded sample of
    the workload: whole tokens of the layer, repeated until `seconds` elapsed
    (at most 64); then the same sample timed again with every expert already
    materialised on the host (the first pass includes their generation).  For
    workloads of at most 64 tokens, also one token on one thread."""
    import numpy as np

    import oracle
    inp, wl = layer.inp, layer.wl
    threads = oracle.default_threads()
    tokens = []
    t0 = time.perf_counter()
    i = 0
    while True:
        tok = (i * 7919) % wl.T
        oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, np.array([tok]), shared=inp.shared,
                          nthreads=threads)
        tokens.append(tok)
        i += 1
        if time.perf_counter() - t0 >= seconds or i >= 64:
            break
    t0 = time.perf_counter()
    for tok in tokens:
        oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, np.array([tok]), shared=inp.shared,
                          nthreads=threads)
    dt = time.perf_counter() - t0
    cb = {"value": len(tokens) / dt, "unit": "tokens/s", "cores": threads, "kind": "oracle",
          "sample": f"{len(tokens)} token(s) of {wl.name} through the whole layer (fp64, {threads} threads)",
          "seconds": round(dt, 3), "cpu_model": cpu_model()}
    if wl.T <= 64:
        t0 = time.perf_counter()
        oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, np.array([tokens[0]]),
                          shared=inp.shared, nthreads=1)
        d1 = time.perf_counter() - t0
        cb["single_thread"] = {"value": 1.0 / d1, "unit": "tokens/s", "cores": 1,
                               "sample": f"1 token of {wl.name} through the whole layer (fp64, 1 thread)",
                               "seconds": round(d1, 3)}
    return cb


def reference_arm(args, rank, world):
    """The fp64 oracle as the reference implementation, K timed steps."""
    import numpy as np

    import oracle
    import synth
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload]
    inp = synth.make_inputs(wl)
    threads = oracle.default_threads()
    toks = lambda i: np.array([(i * 7919) % wl.T])
    # Materialise the experts of the sampled tokens first (input generation).
    n_total = args.steps + args.warmup
    t0 = time.perf_counter()
    oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, toks(0), shared=inp.shared, nthreads=threads)
    t_tok = time.perf_counter() - t0
    budget = 150.0
    # Per-step sample: one token through the layer if the run fits the budget,
    # else the expert MLPs of a subset of one token's routed slots (the
    # route is still computed every step).
    slots = wl.k if n_total * t_tok <= budget else max(1, int(wl.k * budget / (n_total * t_tok)))
    s = oracle.router_logits(inp.x[toks(0)], inp.wr, inp.br, threads)
    ids0, _, _ = oracle.topk(s, wl.k)
    for e in ids0[0]:
        inp.expert(int(e))
    x0 = inp.x_f32[toks(0)[0]].astype(np.float64)

    def one_step(i):
        if slots == wl.k:
            oracle.moe_tokens(inp.x, inp.wr, inp.br, inp.expert, wl.E, wl.I, wl.k, toks(0), shared=inp.shared,
                              nthreads=threads)
        else:
            s = oracle.router_logits(inp.x[toks(0)], inp.wr, inp.br, threads)
            ids, _, _ = oracle.topk(s, wl.k)
            from concurrent.futures import ThreadPoolExecutor
            with ThreadPoolExecutor(max_workers=slots) as ex:
                list(ex.map(lambda j: oracle.expert_mlp(wl.H, wl.I, x0, inp.expert(int(ids[0, (i + j) % wl.k]))),
                            range(slots)))

    for i in range(args.warmup):
        one_step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        one_step(i)
    dt = time.perf_counter() - t0
    tokens_per_step = slots / wl.k
    value = args.steps * tokens_per_step / dt
    sample = (f"1 token of {wl.name} per step through the whole layer" if slots == wl.k else
              f"per step: route + {slots} of the {wl.k} routed expert MLPs of 1 token of {wl.name}")
    line = {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
            "impl": "reference",
            "config": {"workload": wl.name, "tokens_per_step": tokens_per_step},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# -------------------------------------------------------------------- sweep --
SWEEP_T = (1, 2, 4, 8, 16, 32, 48, 64, 96, 128, 192, 256, 384, 512, 768, 1024)


def sweep(args, device):
    """Both paths over batch sizes T: uniform routing, H=7168, E=896 experts
    resident, k=16, I=--sweep-i.  The decode path takes bf16 batches up to
    DECODE_BATCH_MAX_T tokens and the prefill path any T.  One JSON line per
    (T, path): tokens/s, the step's algorithmic bytes per second against the
    measured HBM rate, its FLOP rate, and whether the library's automatic
    choice takes that path.  Graph replay, L2 flushed before every step
    (outside the timing)."""
    import dataclasses

    import mxfp4_routed_expert_moe_gb300 as moe
    import synth
    base = synth.WORKLOADS["decode" if args.sweep_i == 1408 else "decode_i1536"]
    hbm, bf16, _, peak_src = peaks()
    table = None
    for T in SWEEP_T:
        wl = dataclasses.replace(base, name=f"sweep_T{T}_H{base.H}_E{base.E}_k{base.k}_I{base.I}", T=T)
        paths = [("decode", moe.PATH_DECODE)] if T <= moe.DECODE_BATCH_MAX_T else []
        paths.append(("prefill", moe.PATH_PREFILL))
        auto = moe.select_path(T, wl.H, wl.E, wl.I, wl.k)
        for pname, path in paths:
            layer = Layer(wl, device, table=table, path=path)
            table = layer.table
            layer.step()
            layer.torch.cuda.synchronize()
            st = layer.moe.device_status(layer.ws)
            if st != 0:
                raise SystemExit(f"T={T} {pname}: device status {st} ({layer.moe.status_string(st)})")
            n_active = layer.active_experts()
            step_ms, _ = time_steps(layer, args.steps, max(args.warmup, 3), not args.no_graph)
            ms = statistics.mean(step_ms)
            b = layer.algorithmic_bytes_step(n_active)
            line = {"sweep": wl.name, "T": T, "I": wl.I, "path": pname, "tokens_per_s": T / (ms / 1000.0),
                    "ms_per_step": ms, "active_experts": n_active, "step_bytes": b,
                    "weight_gbps": b / (ms / 1000.0) / 1e9, "frac_hbm": b / (ms / 1000.0) / 1e9 / hbm,
                    "tflops": layer.flops_step() / (ms / 1000.0) / 1e12, "steps": args.steps, "auto": path == auto,
                    "peak_source": peak_src, "cuda_graph": not args.no_graph}
            print(json.dumps(line), flush=True)
            del layer


# --------------------------------------------------------------------- main --
PATHS = {"auto": None, "decode": 1, "prefill": 2, "decode_mx": 3}


def step_stats(step_ms):
    q = sorted(step_ms)

    def pct(p):
        return q[min(len(q) - 1, max(0, int(round(p / 100.0 * (len(q) - 1)))))]

    return {"n": len(q), "mean": statistics.mean(q), "median": statistics.median(q), "p10": pct(10), "p90": pct(90),
            "min": q[0], "max": q[-1]}


def all_ranks_ok(ok: bool, world: int, device: str) -> bool:
    if world <= 1:
        return ok
    import torch
    t = torch.tensor([1 if ok else 0], dtype=torch.int32, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MIN)
    return bool(t.item())


def measure(layer, args, rank, world, local, device, steps, cpu_seconds, parity_tokens):
    """One workload: parity on sampled tokens, then `steps` timed steps (L2
    flushed before each), the dominant kernel's roofline, the per-stage
    breakdown, the end-to-end figure and (rank 0) the oracle's CPU baseline.
    Returns (fields, parity); fields is None when parity failed."""
    torch = layer.torch
    wl = layer.wl
    layer.step()
    torch.cuda.synchronize()
    st = layer.moe.device_status(layer.ws)
    if st != 0:
        raise SystemExit(f"{wl.name}: device status {st} ({layer.moe.status_string(st)})")
    n_active = layer.active_experts()
    parity = parity_check(layer, parity_tokens) if rank == 0 else {"ok": True, "checked_on": "rank 0"}
    if not all_ranks_ok(parity["ok"], world, device):
        return None, parity

    clocks = ClockSampler(local)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_wall = time.perf_counter()
    step_ms, graph = time_steps(layer, steps, max(args.warmup, 3), not args.no_graph)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(statistics.mean(step_ms), world, device)
    stats = step_stats(step_ms)
    if steps < 50:
        # Distribution over at least 50 steps (reported beside the K-step mean).
        stats["over_50_steps"] = step_stats(time_steps(layer, 50, 3, not args.no_graph)[0])

    hbm, bf16, bf16_sus, peak_src = peaks()
    stage = layer.dominant_stage()
    st_ms = time_stage(layer, stage, reps=20)
    e2e_ms = time_e2e(layer, max(20, min(steps, 200)), 3, graph)
    breakdown = stage_breakdown(layer)
    nograph_ms = statistics.mean(time_steps(layer, 50 if wl.T <= 64 else 10, 3, False)[0]) if not args.no_graph else ms
    if layer.decode_path and layer.persistent_decode:
        # One launch streams every routed expert's gate, up and down weights.
        ex_bytes = n_active * wl.expert_bytes
        achieved = ex_bytes / (st_ms / 1000.0) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": None, "kernel": "k_dec_mx (persistent block-scaled decode: routing, gate/up, down, combine)",
                "bytes_per_launch": ex_bytes, "launch_ms": st_ms, "peak_source": f"{peak_src} (hbm_gbs, burst)"}
    elif layer.decode_path:
        gu_bytes = layer.algorithmic_bytes_gateup(n_active)
        achieved = gu_bytes / (st_ms / 1000.0) / 1e9
        traffic, sha = traffic_from_profiles("dec_gateup", wl.name)
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic, "kernel": "k_dec_gateup (MXFP4 gate/up GEMV + SwiGLU)",
                "bytes_per_launch": gu_bytes, "launch_ms": st_ms, "peak_source": f"{peak_src} (hbm_gbs, burst)"}
    else:
        # The gate/up MMAs are tcgen05 kind::mxf8f6f4 (E2M1 weights x E4M3 activation terms), an
        # 8-bit-class contraction: its peak is the measured bf16 rate times the nominal fp8 / bf16
        # ratio (4.5 / 2.25).  Each algorithmic product takes two MMA products (the activation's
        # two E4M3 terms), so the MMA rate executed is twice `achieved`.
        fl = layer.flops_gateup()
        achieved = fl / (st_ms / 1000.0) / 1e12
        fp8 = bf16 * FP8_OVER_BF16
        traffic, sha = traffic_from_profiles("pf_gateup", wl.name)
        roof = {"bound": "tensor", "achieved": achieved, "peak": fp8, "unit": "TFLOP/s", "frac": achieved / fp8,
                "traffic": traffic, "kernel": "k_pf_mx<gate/up> (tcgen05 block-scaled grouped GEMM + SwiGLU)",
                "flops_per_launch": fl, "launch_ms": st_ms, "mma_terms": 2,
                "frac_of_bf16_peak": achieved / bf16,
                "hbm_frac_of_step": layer.algorithmic_bytes_step(n_active) / (ms / 1000.0) / 1e9 / hbm,
                "peak_source": f"{peak_src} (bf16_tflops burst x {FP8_OVER_BF16:g}, the nominal fp8 / bf16 ratio: "
                               "the MMAs are kind::mxf8f6f4)"}
    step_bytes = layer.algorithmic_bytes_step(n_active)
    step_flops = layer.flops_step()
    fields = {
        "value": job_tokens_per_s(world, wl.T, ms), "unit": "tokens/s", "ms_per_step": ms,
        "step_ms_stats": stats,
        "config": {"workload": wl.name, "T": wl.T, "H": wl.H, "E": wl.E, "k": wl.k, "I": wl.I,
                   "x_dtype": wl.x_dtype, "path": ("decode_mx" if layer.persistent_decode else "decode") if layer.decode_path else "prefill",
                   "path_arg": args.path, "cuda_graph": not args.no_graph,
                   "l2": "flushed before every step (256 MiB write, then 256 MiB read; outside the step timing)",
                   "active_experts": n_active, "parallelism": f"replicas x{world}"},
        "weight_gbps": step_bytes / (ms / 1000.0) / 1e9,
        "step_roofline": {"bytes": step_bytes, "frac_hbm": step_bytes / (ms / 1000.0) / 1e9 / hbm,
                          "flops": step_flops, "tflops": step_flops / (ms / 1000.0) / 1e12,
                          "frac_bf16": step_flops / (ms / 1000.0) / 1e12 / bf16},
        "no_graph_ms_per_step": nograph_ms,
        "stage_ms": breakdown,
        "roofline": roof,
        "clocks": clk,
        "e2e": {"value": job_tokens_per_s(world, wl.T, e2e_ms), "unit": "tokens/s",
                "h2d_bytes_per_step": layer.x.numel() * layer.x.element_size(),
                "d2h_bytes_per_step": layer.out.numel() * 4, "ms_per_step": e2e_ms},
        "gpu_launches": layer.launches_per_step() * steps,
        "wall_s_timed_region": t_wall,
        "parity": parity,
    }
    if rank == 0:
        fields["cpu_baseline"] = cpu_baseline(layer, cpu_seconds)
    return fields, parity


def main():
    args = parse_args()
    rank, world, local = dist_env()
    if args.impl == "reference":
        reference_arm(args, rank, world)
        return
    if args.sweep:
        import torch
        torch.cuda.set_device(0)
        sweep(args, "cuda:0")
        return
    import torch
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    device = f"cuda:{torch.cuda.current_device()}"
    layer = Layer(args.workload, device, path=PATHS[args.path])
    wl = layer.wl
    fields, parity = measure(layer, args, rank, world, local, device, args.steps, args.cpu_seconds, 3)
    base = {"metric": METRIC, "n_gpus": world, "steps": args.steps, "warmup": max(args.warmup, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": ("f32 activations" if wl.x_dtype == "f32" else "bf16 activations") +
                     ", MXFP4 weights, fp32 accumulate",
            "data": "synthetic (seeded; 896 experts resident in HBM)"}
    if fields is None:
        if rank == 0:
            print(json.dumps(dict(base, value=None, unit="tokens/s", parity=parity,
                                  error="parity against the oracle failed: nothing timed")), flush=True)
        raise SystemExit(1)
    line = dict(base, **fields)
    if args.workload == "decode" and args.path == "auto" and not args.no_prefill_leg:
        # The 4096-token Zipf prefill on the same resident experts (they
        # depend on H, E, I and the seed only).
        long_layer = Layer("long", device, table=layer.table)
        lf, lparity = measure(long_layer, args, rank, world, local, device, args.steps,
                              min(args.cpu_seconds, 5.0), 2)
        if lf is None:
            if rank == 0:
                line["prefill_long"] = {"value": None, "parity": lparity,
                                        "error": "parity against the oracle failed: nothing timed"}
                print(json.dumps(line), flush=True)
            raise SystemExit(1)
        line["prefill_long"] = lf
        del long_layer
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
