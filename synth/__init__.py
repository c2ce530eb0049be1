"""Seeded synthetic inputs for the routed MXFP4 MoE layer (input bytes only).

This package builds the activations, router weights and biases, the packed
MXFP4 expert weights and the bf16 shared expert for every workload, from the
counter-based definitions in ``synth.h``.  The CUDA library and the fp64 oracle
both consume what it makes; it contains none of the layer's arithmetic.

Workloads (shapes and structure follow the layer the pages describe: 896
experts, top-16 routing, MXFP4 experts [deltafin, "How it splits the model"];
wide verification of up to 64 positions per pass [Deltafin's custom compiled
runtime, "Complete target sequence tape"]):

* ``tiny``    T=4,  H=256,  E=8,   k=2,  I=128,  fp32 activations.
* ``decode``  T=1,  H=7168, E=896, k=16, I=1408, bf16 activations.
* ``wide``    T=8, same layer; routing planted so that 8 experts are shared
  by all tokens and 8 are private to each token (union of 72 experts).
* ``prefill`` T=512, same layer, uniform routing, plus one always-on bf16
  shared expert of the same shape.
* ``long``    T=4096, same layer, router bias tau*ln(p_e) with p_e a Zipf(1.1)
  popularity over a seeded permutation of the experts.
* ``decode_i1536`` T=1 with intermediate 1536 (17.55 MB experts).

Value distributions: activations z ~ N(0,1) (Irwin-Hall of twelve uniforms),
router weights 0.02*z in fp32, expert weights 0.02*z quantised to MX blocks,
shared-expert weights 0.02*z rounded to bf16.  Seed 0 throughout.
"""
from __future__ import annotations

import ctypes
import dataclasses
import json
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIBNAME = os.path.join(_HERE, "libmoe_synth.so")
_LOCK = threading.Lock()
_LIB = None

TAG_X = 1
TAG_ROUTER = 2
TAG_PLANT = 3
TAG_PERM = 4
TAG_SHARED = 0x100
TAG_EXPERT = 0x10000

SEED = 0


def _sources():
    return [os.path.join(_HERE, n) for n in ("synth.h", "synth_host.c", "synth_dev.cu")]


def build_command(out=_LIBNAME):
    return [
        "nvcc", "-shared", "-O2", "-std=c++17", "--fmad=false",
        "-gencode", "arch=compute_103a,code=sm_103a",
        "-Xcompiler", "-fPIC,-ffp-contract=off",
        os.path.join(_HERE, "synth_host.c"), os.path.join(_HERE, "synth_dev.cu"),
        "-o", out, "-lpthread",
    ]


def build(force: bool = False) -> str:
    """Compile libmoe_synth.so next to its sources (host fill + device fill)."""
    if not force and os.path.exists(_LIBNAME):
        newest = max(os.path.getmtime(p) for p in _sources())
        if os.path.getmtime(_LIBNAME) >= newest:
            return _LIBNAME
    tmp = _LIBNAME + f".tmp{os.getpid()}"
    subprocess.run(build_command(tmp), check=True)
    os.replace(tmp, _LIBNAME)
    return _LIBNAME


def lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            build()
            L = ctypes.CDLL(_LIBNAME)
            u64, i64, dbl, vp, i32 = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
            L.syn_key_c.restype = u64
            L.syn_key_c.argtypes = [u64, u64]
            L.syn_u64_c.restype = u64
            L.syn_u64_c.argtypes = [u64, u64]
            L.syn_normal_c.restype = dbl
            L.syn_normal_c.argtypes = [u64, u64]
            L.syn_bf16_c.restype = ctypes.c_uint16
            L.syn_bf16_c.argtypes = [ctypes.c_float]
            L.syn_fill_f32.argtypes = [u64, i64, dbl, vp, i32]
            L.syn_fill_bf16.argtypes = [u64, i64, dbl, vp, i32]
            L.syn_fill_mx.argtypes = [u64, i64, i64, vp, vp, i32]
            L.syn_quant_row.argtypes = [vp, i64, vp, vp]
            L.syn_dev_fill_mx.argtypes = [u64, i64, i64, vp, vp, vp]
            _LIB = L
    return _LIB


def _threads():
    return max(1, os.cpu_count() or 1)


def key(seed: int, tag: int) -> int:
    return int(lib().syn_key_c(seed, tag))


def normal(key_: int, n: int, scale: float = 1.0) -> np.ndarray:
    """fp32 array of (float)(scale * z_i), i < n."""
    out = np.empty(n, dtype=np.float32)
    lib().syn_fill_f32(key_, n, scale, out.ctypes.data, _threads())
    return out


def normal_bf16(key_: int, n: int, scale: float = 1.0) -> np.ndarray:
    out = np.empty(n, dtype=np.uint16)
    lib().syn_fill_bf16(key_, n, scale, out.ctypes.data, _threads())
    return out


def bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round fp32 values to bf16 bit patterns (nearest-even)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = ((u & 0x7F800000) == 0x7F800000) & ((u & 0x007FFFFF) != 0)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    r[nan] = ((u[nan] >> 16) | 0x40).astype(np.uint16)
    return r


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def mx_matrix(key_: int, rows: int, cols: int):
    """(q, s) of an MX-quantised rows x cols matrix: q [rows][cols/2], s [rows][cols/32]."""
    q = np.empty((rows, cols // 2), dtype=np.uint8)
    s = np.empty((rows, cols // 32), dtype=np.uint8)
    rc = lib().syn_fill_mx(key_, rows, cols, q.ctypes.data, s.ctypes.data, _threads())
    if rc != 0:
        raise ValueError("syn_fill_mx: cols must be a multiple of 32")
    return q, s


def quant_row(v: np.ndarray):
    """Quantise given reals (length multiple of 32) with the MX block quantiser."""
    v = np.ascontiguousarray(v, dtype=np.float64)
    q = np.empty(v.size // 2, dtype=np.uint8)
    s = np.empty(v.size // 32, dtype=np.uint8)
    if lib().syn_quant_row(v.ctypes.data, v.size, q.ctypes.data, s.ctypes.data) != 0:
        raise ValueError("length must be a multiple of 32")
    return q, s


def permutation(key_: int, n: int) -> np.ndarray:
    """Fisher-Yates shuffle of range(n) driven by the SplitMix64 stream of key_."""
    L = lib()
    p = np.arange(n, dtype=np.int64)
    for i in range(n - 1, 0, -1):
        j = int(L.syn_u64_c(key_, i) % (i + 1))
        p[i], p[j] = p[j], p[i]
    return p


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    x_dtype: str = "bf16"      # "bf16" or "f32"
    routing: str = "uniform"   # "uniform", "planted", "zipf"
    shared: bool = False

    @property
    def expert_bytes(self) -> int:
        """Bytes of one expert's six tensors (nibbles + E8M0 scales)."""
        return 3 * self.H * self.I // 2 + 3 * self.H * self.I // 32

    @property
    def flops_per_token(self) -> int:
        """Routed expert + router (+ shared) FLOPs per token (2 per multiply-add)."""
        f = self.k * 6 * self.H * self.I + 2 * self.H * self.E
        if self.shared:
            f += 6 * self.H * self.I
        return f


WORKLOADS = {
    "tiny": Workload("tiny_T4_H256_E8_k2_I128_f32", 4, 256, 8, 2, 128, x_dtype="f32"),
    "decode": Workload("decode_T1_H7168_E896_k16_I1408", 1, 7168, 896, 16, 1408),
    "wide": Workload("wide_decode_T8_H7168_E896_k16_I1408_planted50", 8, 7168, 896, 16, 1408, routing="planted"),
    "prefill": Workload("prefill_T512_H7168_E896_k16_I1408_shared", 512, 7168, 896, 16, 1408, shared=True),
    "long": Workload("long_prefill_T4096_H7168_E896_k16_I1408_zipf1.1", 4096, 7168, 896, 16, 1408, routing="zipf"),
    "decode_i1536": Workload("decode_T1_H7168_E896_k16_I1536", 1, 7168, 896, 16, 1536),
    # 1-token decode with fp32 activations (the pages keep activations in fp32).
    "decode_f32": Workload("decode_f32_T1_H7168_E896_k16_I1408", 1, 7168, 896, 16, 1408, x_dtype="f32"),
    # A 256-token batch of the full layer: the decode path's batched kernels.
    "batch256": Workload("batch_decode_T256_H7168_E896_k16_I1408", 256, 7168, 896, 16, 1408),
    # Small-footprint case of the decode kernels for profiler captures: 32
    # experts resident (515 MB, above the 129 MB L2), 16 of them routed.
    "decode_e32": Workload("decode_T1_H7168_E32_k16_I1408", 1, 7168, 32, 16, 1408),
    # Small-footprint case of the batched decode kernels for profiler
    # captures: 80 tokens over 256 experts resident (4.1 GB), ~5 routed pairs
    # per active expert, as in a 256-token batch of the full layer.
    "batch80_e256": Workload("batch_decode_T80_H7168_E256_k16_I1408", 80, 7168, 256, 16, 1408),
    # Small-footprint case of the prefill kernels for profiler captures: 64
    # experts resident (1.03 GB), 512 tokens, ~128 tokens per expert.
    "prefill_e64": Workload("prefill_T512_H7168_E64_k16_I1408", 512, 7168, 64, 16, 1408),
}

# Planted wide-decode routing: x_t = z_t + A*u + A*v_t; router rows of the 8
# shared experts get + C*u, the 8 private rows of token t get + C*v_t (u, v_t
# unit vectors).  Planted scores sit near C*A = 64, the rest near N(0, 1.7^2).
PLANT_SHARED = 8
PLANT_A = 16.0
PLANT_C = 4.0
ZIPF_ALPHA = 1.1
ZIPF_TAU_FILE = os.path.join(_HERE, "zipf_tau.json")


def zipf_tau() -> float:
    with open(ZIPF_TAU_FILE) as f:
        return float(json.load(f)["tau"])


def zipf_log_popularity(wl: Workload, seed: int = SEED) -> np.ndarray:
    """ln p_e with p_e proportional to rank(e)^-alpha over a seeded permutation."""
    perm = permutation(key(seed, TAG_PERM + 1), wl.E)
    rank = np.empty(wl.E, dtype=np.float64)
    rank[perm] = np.arange(1, wl.E + 1, dtype=np.float64)
    logw = -ZIPF_ALPHA * np.log(rank)
    return logw - math.log(float(np.sum(np.exp(logw))))


def zipf_bias(wl: Workload, tau: float, seed: int = SEED) -> np.ndarray:
    return (tau * zipf_log_popularity(wl, seed)).astype(np.float32)


def planted_sets(wl: Workload, seed: int = SEED):
    """(shared experts, private experts per token) of the planted routing."""
    perm = permutation(key(seed, TAG_PERM), wl.E)
    ns = PLANT_SHARED
    npriv = wl.k - ns
    shared = perm[:ns]
    private = [perm[ns + npriv * t: ns + npriv * (t + 1)] for t in range(wl.T)]
    return shared, private


def _unit(v: np.ndarray) -> np.ndarray:
    return v / np.sqrt(np.sum(v * v))


@dataclasses.dataclass
class LayerInputs:
    wl: Workload
    seed: int
    x: np.ndarray            # [T][H] uint16 (bf16 bits) or float32
    wr: np.ndarray           # [E][H] float32
    br: np.ndarray | None    # [E] float32
    shared: tuple | None     # (gate [I][H], up [I][H], down [H][I]) uint16 bf16 bits
    _experts: dict = dataclasses.field(default_factory=dict)

    @property
    def x_f32(self) -> np.ndarray:
        return self.x if self.wl.x_dtype == "f32" else bf16_to_f32(self.x)

    def expert_key(self, e: int, j: int) -> int:
        return key(self.seed, TAG_EXPERT + 4 * e + j)

    def expert(self, e: int) -> dict:
        """Host copy of expert e: gate_q/gate_s/up_q/up_s ([I][H] matrix) and
        down_q/down_s ([H][I] matrix), generated on demand."""
        if e not in self._experts:
            wl = self.wl
            gq, gs = mx_matrix(self.expert_key(e, 0), wl.I, wl.H)
            uq, us = mx_matrix(self.expert_key(e, 1), wl.I, wl.H)
            dq, ds = mx_matrix(self.expert_key(e, 2), wl.H, wl.I)
            self._experts[e] = dict(gate_q=gq, gate_s=gs, up_q=uq, up_s=us, down_q=dq, down_s=ds)
        return self._experts[e]


def make_inputs(wl: Workload, seed: int = SEED) -> LayerInputs:
    T, H, E, I = wl.T, wl.H, wl.E, wl.I
    z = normal(key(seed, TAG_X), T * H).reshape(T, H)
    wr = normal(key(seed, TAG_ROUTER), E * H, 0.02).reshape(E, H)
    br = None
    if wl.routing == "planted":
        shared, private = planted_sets(wl, seed)
        pz = normal(key(seed, TAG_PLANT), (T + 1) * H).astype(np.float64).reshape(T + 1, H)
        u = _unit(pz[0])
        xd = z.astype(np.float64)
        wrd = wr.astype(np.float64)
        for e in shared:
            wrd[e] += PLANT_C * u
        for t in range(T):
            v = _unit(pz[t + 1])
            xd[t] += PLANT_A * u + PLANT_A * v
            for e in private[t]:
                wrd[e] += PLANT_C * v
        z = xd.astype(np.float32)
        wr = wrd.astype(np.float32)
    elif wl.routing == "zipf":
        br = zipf_bias(wl, zipf_tau(), seed)
    x = z.astype(np.float32) if wl.x_dtype == "f32" else bf16_bits(z)
    shared_w = None
    if wl.shared:
        shared_w = (
            normal_bf16(key(seed, TAG_SHARED + 0), I * H, 0.02).reshape(I, H),
            normal_bf16(key(seed, TAG_SHARED + 1), I * H, 0.02).reshape(I, H),
            normal_bf16(key(seed, TAG_SHARED + 2), H * I, 0.02).reshape(H, I),
        )
    return LayerInputs(wl, seed, np.ascontiguousarray(x), np.ascontiguousarray(wr), br, shared_w)


# ---------------------------------------------------------------- device fill --

def expert_blob_layout(wl: Workload):
    """Byte offsets of the six tensors inside one expert's contiguous blob
    (gate_q, gate_s, up_q, up_s, down_q, down_s), each 256-byte aligned, and
    the blob stride."""
    def up256(n):
        return (n + 255) // 256 * 256
    sizes = [wl.I * wl.H // 2, wl.I * wl.H // 32, wl.I * wl.H // 2, wl.I * wl.H // 32,
             wl.H * wl.I // 2, wl.H * wl.I // 32]
    offs, o = [], 0
    for n in sizes:
        offs.append(o)
        o += up256(n)
    return offs, o


def fill_experts_device(inp: LayerInputs, blob_ptr: int, stream_ptr: int = 0) -> None:
    """Write all E experts into a device buffer of E * stride bytes (stride from
    expert_blob_layout), expert e at blob_ptr + e * stride."""
    wl = inp.wl
    offs, stride = expert_blob_layout(wl)
    L = lib()
    shapes = [(wl.I, wl.H), (wl.I, wl.H), (wl.H, wl.I)]
    for e in range(wl.E):
        base = blob_ptr + e * stride
        for j in range(3):
            rows, cols = shapes[j]
            rc = L.syn_dev_fill_mx(inp.expert_key(e, j), rows, cols,
                                   ctypes.c_void_p(base + offs[2 * j]), ctypes.c_void_p(base + offs[2 * j + 1]),
                                   ctypes.c_void_p(stream_ptr))
            if rc != 0:
                raise RuntimeError(f"syn_dev_fill_mx failed with CUDA error {rc}")
