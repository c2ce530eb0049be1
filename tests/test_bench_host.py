"""Host logic of bench.py that the reported rooflines rest on, checked on the
CPU: the algorithmic bytes and FLOPs against closed forms worked out by hand
for the pages' layer (H = 7168, I = 1408, k = 16, E = 896; MXFP4 = 4-bit codes
plus one 8-bit scale per 32 values [OCP Microscaling Formats v1.0, section
5]), the launches counted per step, and the lookup of recorded DRAM traffic,
which must drop a record once the kernel's sources change."""
import os

import pytest

import bench
import synth

H, I, K, E = 7168, 1408, 16, 896
MX_MATRIX = I * H // 2 + I * H // 32  # codes + scales of one I x H matrix: 5,361,664 bytes


def _layer(name, shared=False, path=None):
    """A bench.Layer with only the fields the host arithmetic reads (no GPU)."""
    import mxfp4_routed_expert_moe_gb300 as moe
    layer = object.__new__(bench.Layer)
    layer.moe = moe
    layer.wl = synth.WORKLOADS[name]
    layer.shared = object() if shared else None
    layer.path = moe.PATH_AUTO if path is None else path
    return layer


def test_mx_matrix_bytes():
    assert MX_MATRIX == 5_361_664


def test_decode_gateup_bytes_closed_form():
    """16 routed experts x (gate + up) + the bf16 token + fp32 h of its 16 pairs."""
    got = _layer("decode").algorithmic_bytes_gateup(16)
    assert got == 16 * 2 * MX_MATRIX + H * 2 + K * I * 4 == 171_677_696


def test_decode_step_bytes_closed_form():
    """Experts (3 matrices each), fp32 router weights, bf16 x in, fp32 out."""
    got = _layer("decode").algorithmic_bytes_step(16)
    assert got == 16 * 3 * MX_MATRIX + E * H * 4 + H * 2 + H * 4 == 283_092_992


def test_decode_f32_step_reads_fp32_activations():
    assert _layer("decode_f32").algorithmic_bytes_step(16) - _layer("decode").algorithmic_bytes_step(16) == H * 2


def test_long_prefill_flops_closed_form():
    """4096 tokens x 16 pairs: gate/up = 2 matrices x 2 H I per pair; the
    step adds down (2 H I per pair) and the router (2 E H per token)."""
    lay = _layer("long")
    T = lay.wl.T
    assert T == 4096
    assert lay.flops_gateup() == 2 * T * K * 2 * H * I == 2_645_699_854_336
    assert lay.flops_step() == T * (2 * K * 3 * H * I + 2 * E * H) == 4_021_163_130_880


def test_shared_expert_adds_its_rows_and_bytes():
    plain, sh = _layer("prefill"), _layer("prefill", shared=True)
    T = plain.wl.T
    assert sh.flops_gateup() - plain.flops_gateup() == 2 * T * 2 * H * I
    assert sh.algorithmic_bytes_step(10) - plain.algorithmic_bytes_step(10) == 3 * H * I * 2


@pytest.mark.parametrize("name,shared,launches", [
    ("decode", False, 3),   # router GEMV, gate/up (+ routing), down (+ combine)
    ("wide", False, 3),
    ("decode", True, 9),    # + the shared expert on the prefill kernels
    ("batch256", False, 9),  # screen router (3), bucket count/scatter, x->fp16, gate/up, down, combine
    ("long", False, 12),    # screen router (3) + 9 prefill launches
])
def test_launches_per_step(name, shared, launches):
    assert _layer(name, shared=shared).launches_per_step() == launches


def test_persistent_decode_counts_two_launches():
    import mxfp4_routed_expert_moe_gb300 as moe
    assert _layer("decode", path=moe.PATH_DECODE_MX).launches_per_step() == 2


def _fake_tree(root, kernel):
    for f in bench.KERNEL_SOURCES[kernel]:
        p = os.path.join(root, "mxfp4_routed_expert_moe_gb300", "csrc", f)
        os.makedirs(os.path.dirname(p), exist_ok=True)
        with open(p, "w") as fh:
            fh.write(f"// {f}\n")
    os.makedirs(os.path.join(root, "profiles"), exist_ok=True)


def test_traffic_record_follows_the_kernel_sources(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    kernel, wl = "dec_gateup", "decode_T1_H7168_E896_k16_I1408"
    _fake_tree(str(tmp_path), kernel)
    sha = bench.source_sha(kernel)
    (tmp_path / "profiles" / "k.md").write_text(
        f"notes\ntraffic[{kernel}:{wl}]: bytes_per_launch=175000000 source_sha={sha}\n")
    assert bench.traffic_from_profiles(kernel, wl) == (175000000, sha)
    # Another workload has no record.
    assert bench.traffic_from_profiles(kernel, "other")[0] is None
    # A changed source file makes the record stale.
    src = tmp_path / "mxfp4_routed_expert_moe_gb300" / "csrc" / bench.KERNEL_SOURCES[kernel][-1]
    src.write_text(src.read_text() + "// changed\n")
    got, new_sha = bench.traffic_from_profiles(kernel, wl)
    assert got is None and new_sha != sha
