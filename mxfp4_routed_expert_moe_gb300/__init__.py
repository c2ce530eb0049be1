"""Python binding of libmoe_mxfp4.so, the GB300 routed MXFP4 MoE layer.

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  Tensors are torch CUDA tensors (PyTorch provides device memory and
streams); the library's C ABI is declared in ``include/moe_mxfp4.h``.  There is
no fallback: if the library is missing or fails to load, importing the
binding's functions raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmoe_mxfp4.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_TIMEOUT = 5
MOE_ERR_DEVICE_CHECK = 6
MOE_ERR_RANGE = 7

DT_F32 = 0
DT_BF16 = 1

PATH_AUTO = 0
PATH_DECODE = 1
PATH_PREFILL = 2
PATH_DECODE_MX = 3  # the persistent block-scaled decode kernel (explicit choice only)
DECODE_MAX_T = 64                  # MOE_DECODE_MAX_T
DECODE_BATCH_MAX_T = 1024          # MOE_DECODE_BATCH_MAX_T
DECODE_AUTO_PAIRS_PER_EXPERT = 5  # MOE_DECODE_AUTO_PAIRS_PER_EXPERT

# Every symbol the header declares (checked by the tests against the .so).
EXPORTS = ("moe_abi_version", "moe_status_string", "moe_workspace_bytes", "moe_route", "moe_mxfp4_experts",
           "moe_forward", "moe_device_status", "moe_profile_events", "moe_forward_static_scratch",
           "moe_wait_selftest", "moe_select_path", "moe_set_wait_limit")
STATIC_SCRATCH_BYTES = 8 << 20

STAGE_ROUTE, STAGE_GATEUP, STAGE_DOWN, STAGE_COMBINE, STAGE_PF_GATEUP, STAGE_PF_DOWN = 1, 2, 3, 4, 5, 6


class MoeError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: status {status} ({status_string(status)})")
        self.status = status


class Shape(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("I", ctypes.c_int32),
                ("k", ctypes.c_int32)]


class DenseBf16(ctypes.Structure):
    _fields_ = [("gate", ctypes.c_void_p), ("up", ctypes.c_void_p), ("down", ctypes.c_void_p)]


_LOCK = threading.Lock()
_LIB = None


def lib():
    """The loaded library (raises if it is missing: there is no fallback)."""
    global _LIB
    with _LOCK:
        if _LIB is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m mxfp4_routed_expert_moe_gb300.build`")
            L = ctypes.CDLL(LIB_PATH)
            vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            P = ctypes.POINTER
            L.moe_abi_version.restype = ctypes.c_uint32
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_status_string.argtypes = [i32]
            L.moe_workspace_bytes.restype = sz
            L.moe_workspace_bytes.argtypes = [P(Shape)]
            L.moe_route.argtypes = [P(Shape), vp, i32, vp, vp, vp, vp, vp, vp, vp, sz, vp]
            L.moe_mxfp4_experts.argtypes = [P(Shape), vp, i32, vp, vp, vp, vp, vp, vp, i32, i32, vp, sz, vp]
            L.moe_forward.argtypes = [P(Shape), vp, i32, vp, vp, vp, P(DenseBf16), vp, i32, vp, vp, i32, vp, sz, vp]
            L.moe_device_status.argtypes = [vp, vp, P(ctypes.c_int)]
            L.moe_profile_events.argtypes = [i32, vp, vp]
            L.moe_wait_selftest.argtypes = [ctypes.c_longlong, vp, P(ctypes.c_int)]
            L.moe_set_wait_limit.argtypes = [ctypes.c_longlong]
            L.moe_select_path.argtypes = [P(Shape), i32, i32, i32, P(ctypes.c_int)]
            L.moe_forward_static_scratch.argtypes = [P(Shape), vp, i32, vp, vp, vp, P(DenseBf16), vp, i32, vp, vp,
                                                     i32, vp, vp]
            _LIB = L
    return _LIB


def abi_version() -> int:
    return int(lib().moe_abi_version())


def status_string(status: int) -> str:
    return lib().moe_status_string(status).decode()


def shape(T, H, E, I, k) -> Shape:
    return Shape(T, H, E, I, k)


def workspace_bytes(T, H, E, I, k) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(Shape(T, H, E, I, k))))


def select_path(T, H, E, I, k, x_dtype=DT_BF16, shared=False, path=PATH_AUTO) -> int:
    """moe_select_path: the path (PATH_DECODE or PATH_PREFILL) a call with
    this shape runs; raises MoeError where the call would fail before
    launching."""
    out = ctypes.c_int(-1)
    _check(lib().moe_select_path(ctypes.byref(Shape(T, H, E, I, k)), int(x_dtype), int(bool(shared)), int(path),
                                 ctypes.byref(out)), "moe_select_path")
    return int(out.value)


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_of(x) -> int:
    import torch
    if x.dtype == torch.float32:
        return DT_F32
    if x.dtype == torch.bfloat16:
        return DT_BF16
    raise TypeError("activations must be torch.float32 or torch.bfloat16")


def _check(rc, what):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def route(shp: Shape, x, w_router, b_router, ids, w, offsets, sorted_idx, ws, stream=None):
    """moe_route: fills ids [T][k] int32, w [T][k] fp32 and (optionally) the
    bucket layout offsets [E+1] / sorted_idx [T*k]."""
    rc = lib().moe_route(ctypes.byref(shp), _ptr(x), _dtype_of(x), _ptr(w_router), _ptr(b_router), _ptr(ids),
                         _ptr(w), _ptr(offsets), _ptr(sorted_idx), _ptr(ws), ws.numel() * ws.element_size(),
                         _stream(stream))
    _check(rc, "moe_route")


def mxfp4_experts(shp: Shape, x, experts, ids, w, offsets, sorted_idx, out, accumulate, ws, path=PATH_AUTO,
                  stream=None):
    """moe_mxfp4_experts: out [T][H] fp32 (+)= sum_j w[t][j] * expert_{ids[t][j]}(x_t)."""
    rc = lib().moe_mxfp4_experts(ctypes.byref(shp), _ptr(x), _dtype_of(x), _ptr(experts), _ptr(ids), _ptr(w),
                                 _ptr(offsets), _ptr(sorted_idx), _ptr(out), int(bool(accumulate)), int(path),
                                 _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_mxfp4_experts")


def forward(shp: Shape, x, w_router, b_router, experts, shared, out, accumulate, ws, ids_out=None, w_out=None,
            path=PATH_AUTO, stream=None):
    """moe_forward: the whole layer.  ``shared`` is None or (gate, up, down)
    bf16 tensors ([I][H], [I][H], [H][I])."""
    sh = None
    if shared is not None:
        sh = ctypes.byref(DenseBf16(_ptr(shared[0]), _ptr(shared[1]), _ptr(shared[2])))
    rc = lib().moe_forward(ctypes.byref(shp), _ptr(x), _dtype_of(x), _ptr(w_router), _ptr(b_router),
                           _ptr(experts), sh, _ptr(out), int(bool(accumulate)), _ptr(ids_out), _ptr(w_out),
                           int(path), _ptr(ws), ws.numel() * ws.element_size(), _stream(stream))
    _check(rc, "moe_forward")


def forward_static_scratch(shp: Shape, x, w_router, b_router, experts, shared, out, accumulate, ids_out=None,
                           w_out=None, path=PATH_AUTO, status_dev=None, stream=None):
    """moe_forward_static_scratch: the layer with the library's own static
    device scratch as workspace (no workspace argument; nothing allocated).
    For callers that cannot hand the library device memory; calls on one
    device must not overlap in time.  ``status_dev`` is None or a device int32
    tensor that receives the call's device status word."""
    sh = None
    if shared is not None:
        sh = ctypes.byref(DenseBf16(_ptr(shared[0]), _ptr(shared[1]), _ptr(shared[2])))
    rc = lib().moe_forward_static_scratch(ctypes.byref(shp), _ptr(x), _dtype_of(x), _ptr(w_router), _ptr(b_router),
                                          _ptr(experts), sh, _ptr(out), int(bool(accumulate)), _ptr(ids_out),
                                          _ptr(w_out), int(path), _ptr(status_dev), _stream(stream))
    _check(rc, "moe_forward_static_scratch")


def wait_selftest(max_cycles: int, stream=None) -> int:
    """moe_wait_selftest: run the device bounded-wait code on a barrier that
    never completes, with a limit of max_cycles; returns the device status
    (MOE_ERR_TIMEOUT when the wait gave up)."""
    st = ctypes.c_int(-1)
    _check(lib().moe_wait_selftest(int(max_cycles), _stream(stream), ctypes.byref(st)), "moe_wait_selftest")
    return st.value


def profile_events(stage: int, before=None, after=None) -> None:
    """Record torch.cuda.Event `before`/`after` around the kernel of `stage`
    in subsequent calls (None clears)."""
    b = None if before is None else before.cuda_event
    a = None if after is None else after.cuda_event
    _check(lib().moe_profile_events(int(stage), b, a), "moe_profile_events")


def set_wait_limit(cycles: int) -> None:
    """moe_set_wait_limit: SM clock cycles after which the kernels' bounded
    waits give up (diagnostic; 0 restores the default)."""
    _check(lib().moe_set_wait_limit(int(cycles)), "moe_set_wait_limit")


def device_status(ws, stream=None) -> int:
    st = ctypes.c_int(-1)
    rc = lib().moe_device_status(_ptr(ws), _stream(stream), ctypes.byref(st))
    _check(rc, "moe_device_status")
    return st.value


# --------------------------------------------------------------- model state --

class ExpertTable:
    """Device-resident MXFP4 experts: one contiguous blob per expert holding its
    six tensors (gate q/s, up q/s, down q/s), plus the device array of moe_expert
    descriptors (six pointers per expert) the library reads."""

    def __init__(self, E: int, H: int, I: int, device="cuda"):
        import torch
        self.E, self.H, self.I = E, H, I
        self.offsets, self.stride = self.blob_layout(H, I)
        self.blob = torch.empty(E * self.stride, dtype=torch.uint8, device=device)
        base = self.blob.data_ptr()
        desc = torch.empty((E, 6), dtype=torch.int64)
        for e in range(E):
            for j in range(6):
                desc[e, j] = base + e * self.stride + self.offsets[j]
        self.desc = desc.to(device)

    @staticmethod
    def blob_layout(H: int, I: int):
        """Byte offsets of gate_q, gate_s, up_q, up_s, down_q, down_s inside
        one expert blob (each 256-byte aligned) and the blob stride."""
        def up256(n):
            return (n + 255) // 256 * 256
        sizes = [I * H // 2, I * H // 32, I * H // 2, I * H // 32, H * I // 2, H * I // 32]
        offs, o = [], 0
        for n in sizes:
            offs.append(o)
            o += up256(n)
        return offs, o

    def tensor(self, e: int, j: int):
        """View of tensor j (0..5) of expert e as a 2-D uint8 tensor."""
        H, I = self.H, self.I
        shapes = [(I, H // 2), (I, H // 32), (I, H // 2), (I, H // 32), (H, I // 2), (H, I // 32)]
        r, c = shapes[j]
        o = e * self.stride + self.offsets[j]
        return self.blob[o:o + r * c].view(r, c)

    def load_host(self, e: int, ex: dict):
        import torch
        names = ("gate_q", "gate_s", "up_q", "up_s", "down_q", "down_s")
        for j, n in enumerate(names):
            self.tensor(e, j).copy_(torch.from_numpy(ex[n]))

    @property
    def ptr(self) -> int:
        return self.desc.data_ptr()
