"""The C-ABI library loads and exports every symbol its header declares; host
validation rejects bad arguments before any launch (no GPU needed: these
calls return before touching CUDA)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "moe_mxfp4.h")


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b(moe_\w+)\s*\(", src, flags=re.M)
    return sorted(set(names))


@pytest.fixture(scope="module")
def moe():
    import mxfp4_routed_expert_moe_gb300 as m
    import mxfp4_routed_expert_moe_gb300.build as b
    b.build()
    m.lib()
    return m


def test_header_declares_the_expected_entry_points(moe):
    assert _declared_functions() == sorted(moe.EXPORTS)


def test_library_exports_every_declared_symbol(moe):
    L = ctypes.CDLL(moe.LIB_PATH)
    for name in _declared_functions():
        assert hasattr(L, name), name


def test_version_and_status_strings(moe):
    assert moe.abi_version() == 1
    for st in range(8):
        assert moe.status_string(st) and moe.status_string(st) != "unknown status"
    assert moe.status_string(42) == "unknown status"


def test_workspace_bytes(moe):
    small = moe.workspace_bytes(4, 256, 8, 128, 2)
    big = moe.workspace_bytes(4096, 7168, 896, 1408, 16)
    assert 0 < small < big
    assert big % 256 == 0
    # Invalid shapes report 0.
    assert moe.workspace_bytes(0, 256, 8, 128, 2) == 0
    assert moe.workspace_bytes(4, 250, 8, 128, 2) == 0
    assert moe.workspace_bytes(4, 256, 8, 120, 2) == 0
    assert moe.workspace_bytes(4, 256, 8, 128, 9) == 0
    assert moe.workspace_bytes(4, 256, 64, 128, 33) == 0


def _call_route(moe, shp, x=16, wr=16, ids=16, w=16, ws=256, ws_bytes=None, dtype=1):
    L = moe.lib()
    if ws_bytes is None:
        ws_bytes = L.moe_workspace_bytes(ctypes.byref(shp))
    return L.moe_route(ctypes.byref(shp), x, dtype, wr, None, ids, w, None, None, ws, ws_bytes, None)


def test_route_rejects_bad_arguments_before_launch(moe):
    # Fake, never-dereferenced addresses: validation fails first.
    shp = moe.shape(4, 256, 8, 128, 2)
    A = 1 << 20
    assert _call_route(moe, shp, x=None, wr=A, ids=A, w=A, ws=A) == moe.MOE_ERR_INVALID_ARG
    assert _call_route(moe, shp, x=A + 8, wr=A, ids=A, w=A, ws=A) == moe.MOE_ERR_INVALID_ARG
    assert _call_route(moe, shp, x=A, wr=A, ids=A, w=A, ws=A + 16) == moe.MOE_ERR_INVALID_ARG
    assert _call_route(moe, shp, x=A, wr=A, ids=A, w=A, ws=A, ws_bytes=100) == moe.MOE_ERR_WORKSPACE
    assert _call_route(moe, shp, x=A, wr=A, ids=A, w=A, ws=A, dtype=5) == moe.MOE_ERR_INVALID_ARG
    bad = moe.shape(4, 256, 8, 128, 40)
    assert _call_route(moe, bad, x=A, wr=A, ids=A, w=A, ws=A, ws_bytes=1 << 30) == moe.MOE_ERR_INVALID_ARG
    big = moe.shape(4, 32768, 8, 128, 2)
    assert _call_route(moe, big, x=A, wr=A, ids=A, w=A, ws=A, ws_bytes=1 << 30) == moe.MOE_ERR_UNSUPPORTED


def test_degenerate_shapes_are_rejected_before_launch(moe):
    """An empty batch, k = 0, k > E and H off the 32-element MX block grid are
    invalid shapes (the header's limits): no workspace size, and every entry
    point returns MOE_ERR_INVALID_ARG without touching its (fake) pointers."""
    L = moe.lib()
    A = 1 << 20
    for T, H, E, I, k in [(0, 256, 8, 128, 2), (4, 256, 8, 128, 0), (4, 256, 8, 128, 9), (4, 240, 8, 128, 2),
                          (4, 256, 8, 112, 2), (4, 256, 0, 128, 1)]:
        shp = moe.shape(T, H, E, I, k)
        assert L.moe_workspace_bytes(ctypes.byref(shp)) == 0, (T, H, E, I, k)
        assert _call_route(moe, shp, x=A, wr=A, ids=A, w=A, ws=A, ws_bytes=1 << 30) == moe.MOE_ERR_INVALID_ARG
        rc = L.moe_forward(ctypes.byref(shp), A, 1, A, None, A, None, A, 0, None, None, 0, A, 1 << 30, None)
        assert rc == moe.MOE_ERR_INVALID_ARG
        rc = L.moe_mxfp4_experts(ctypes.byref(shp), A, 1, A, A, A, None, None, A, 0, 0, A, 1 << 30, None)
        assert rc == moe.MOE_ERR_INVALID_ARG


def test_forward_and_experts_reject_bad_arguments(moe):
    L = moe.lib()
    A = 1 << 20
    shp = moe.shape(4, 256, 8, 128, 2)
    wsb = L.moe_workspace_bytes(ctypes.byref(shp))
    # Null out.
    rc = L.moe_forward(ctypes.byref(shp), A, 1, A, None, A, None, None, 0, None, None, 0, A, wsb, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # Unknown path.
    rc = L.moe_forward(ctypes.byref(shp), A, 1, A, None, A, None, A, 0, None, None, 7, A, wsb, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # fp32 activations are not taken by the prefill path.
    rc = L.moe_forward(ctypes.byref(shp), A, 0, A, None, A, None, A, 0, None, None, 2, A, wsb, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    # Decode path: bf16 batches up to DECODE_BATCH_MAX_T tokens, fp32 up to 64.
    shp2 = moe.shape(moe.DECODE_BATCH_MAX_T + 1, 256, 8, 128, 2)
    wsb2 = L.moe_workspace_bytes(ctypes.byref(shp2))
    rc = L.moe_forward(ctypes.byref(shp2), A, 1, A, None, A, None, A, 0, None, None, 1, A, wsb2, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    shp3 = moe.shape(65, 256, 8, 128, 2)
    wsb3 = L.moe_workspace_bytes(ctypes.byref(shp3))
    rc = L.moe_forward(ctypes.byref(shp3), A, 0, A, None, A, None, A, 0, None, None, 1, A, wsb3, None)
    assert rc == moe.MOE_ERR_UNSUPPORTED
    # Experts-only: offsets without sorted_idx.
    rc = L.moe_mxfp4_experts(ctypes.byref(shp), A, 1, A, A, A, A, None, A, 0, 0, A, wsb, None)
    assert rc == moe.MOE_ERR_INVALID_ARG
    # Shared expert with a null tensor.
    sh = moe.DenseBf16(A, None, A)
    rc = L.moe_forward(ctypes.byref(shp), A, 1, A, None, A, ctypes.byref(sh), A, 0, None, None, 2, A, wsb, None)
    assert rc == moe.MOE_ERR_INVALID_ARG


def test_product_path_has_no_oracle_dependency():
    """The package and its CUDA sources never import or include the oracle."""
    pkg = os.path.join(ROOT, "mxfp4_routed_expert_moe_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "oracle.c" not in text and "from oracle" not in text, f
                assert "synth" not in text or f == "build.py" and "synth" not in text, f


def test_select_path_rules(moe):
    """The automatic path choice as the header states it: decode up to 64
    tokens or for fp32 activations; decode for larger bf16 batches while
    T*k <= DECODE_AUTO_PAIRS_PER_EXPERT * E and T <= DECODE_BATCH_MAX_T; else
    prefill.  Host only."""
    D, P = moe.PATH_DECODE, moe.PATH_PREFILL
    H, E, I, k = 7168, 896, 1408, 16
    sel = moe.select_path
    assert sel(1, H, E, I, k) == D
    assert sel(64, H, E, I, k) == D
    assert sel(64, H, E, I, k, x_dtype=moe.DT_F32) == D
    t_max = moe.DECODE_AUTO_PAIRS_PER_EXPERT * E // k  # largest T the rule sends to decode
    assert t_max <= moe.DECODE_BATCH_MAX_T
    assert sel(t_max, H, E, I, k) == D
    assert sel(t_max + 1, H, E, I, k) == P
    assert sel(4096, H, E, I, k) == P
    # Few experts: many pairs per expert, the tensor-core path.
    assert sel(512, H, 64, I, k) == P
    assert sel(65, H, 64, I, k) == P
    # A shared expert does not change the choice: the decode path runs it on
    # the prefill kernels after the routed experts (bf16, H and I % 128 == 0).
    assert sel(1, H, E, I, k, shared=True) == D
    assert sel(t_max, H, E, I, k, shared=True) == D
    assert sel(512, H, E, I, k, shared=True) == P
    assert sel(4096, H, E, I, k, shared=True) == P
    with pytest.raises(moe.MoeError) as ei:
        sel(1, 7168 + 32, E, I, k, shared=True)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    # A bf16 shape the decode kernels do not take (H > 8192) goes to the
    # prefill path when that path takes it (H, I % 128 == 0); fp32 cannot.
    assert sel(1, 12288, E, I, k) == P
    assert sel(64, 16384, E, I, k) == P
    with pytest.raises(moe.MoeError) as ei:
        sel(1, 12288, E, I, k, path=D)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        sel(1, 12288, E, I, k, x_dtype=moe.DT_F32)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    # Explicit paths.
    assert sel(512, H, 64, I, k, path=D) == D
    assert sel(1, H, E, I, k, path=P) == P
    with pytest.raises(moe.MoeError) as ei:
        sel(moe.DECODE_BATCH_MAX_T + 1, H, E, I, k, path=D)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        sel(65, H, E, I, k, x_dtype=moe.DT_F32)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        sel(1, H, E, I, k, x_dtype=moe.DT_F32, shared=True)
    assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
    with pytest.raises(moe.MoeError) as ei:
        sel(0, H, E, I, k)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
