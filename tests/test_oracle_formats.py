"""Pins of the oracle's MXFP4 decoding against the format definition.

The E2M1 table and the E8M0 scale come from the OCP Microscaling Formats (MX)
v1.0 specification; the scale-as-exponent view comes from [deltafin, "The
techniques that bought the 82x"] (the fused dequant+GEMV applies the E8M0
scale as integer arithmetic on the fp32 exponent).
"""
import math
import os
import struct

import numpy as np
import pytest

import oracle
from conftest import GOLDEN, parse_float


def _golden_table():
    table = {}
    with open(os.path.join(GOLDEN, "e2m1_table.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            c, v = line.split()
            table[int(c)] = parse_float(v)
    return table


def _same(a: float, b: float) -> bool:
    """Equal including the sign of zero and NaN-ness."""
    if math.isnan(a) or math.isnan(b):
        return math.isnan(a) and math.isnan(b)
    return a == b and math.copysign(1.0, a) == math.copysign(1.0, b)


def test_e2m1_matches_golden_table():
    table = _golden_table()
    assert sorted(table) == list(range(16))
    for c, v in table.items():
        assert _same(oracle.e2m1(c), v), (c, oracle.e2m1(c), v)


def test_e2m1_matches_bit_field_definition():
    # Independent closed form: sign s, exponent field E (bias 1), mantissa m;
    # E == 0 is subnormal: 0.m * 2^(1-1); else 1.m * 2^(E-1).
    for c in range(16):
        s, E, m = c >> 3, (c >> 1) & 3, c & 1
        mag = (m / 2.0) if E == 0 else (1.0 + m / 2.0) * 2.0 ** (E - 1)
        v = -mag if s else mag
        assert _same(oracle.e2m1(c), v), c


def test_e8m0_is_power_of_two_and_nan():
    for e in range(255):
        assert oracle.e8m0(e) == 2.0 ** (e - 127)
    assert math.isnan(oracle.e8m0(255))


def _golden_blocks():
    blocks, cur = [], None
    with open(os.path.join(GOLDEN, "mx_blocks.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line == "block":
                cur = {}
                blocks.append(cur)
                continue
            key, rest = line.split(None, 1)
            if key == "scale":
                cur["scale"] = int(rest)
            elif key == "bytes":
                cur["bytes"] = bytes(int(b, 16) for b in rest.split())
            elif key == "values":
                cur["values"] = [parse_float(t) for t in rest.split()]
    return blocks


def test_hand_worked_blocks():
    blocks = _golden_blocks()
    assert len(blocks) >= 5
    for b in blocks:
        q = np.frombuffer(b["bytes"], dtype=np.uint8).reshape(1, 16)
        s = np.array([[b["scale"]]], dtype=np.uint8)
        got = oracle.dequant(q, s, 1, 32)[0]
        assert len(b["values"]) == 32
        for i, v in enumerate(b["values"]):
            assert _same(float(got[i]), v), (b["scale"], i, got[i], v)


def test_multi_block_row_indexing():
    # Two rows, three blocks each, every block a different scale: element (r, c)
    # must use byte r*48 + c//2 and scale r*3 + c//32.
    rng = np.random.default_rng(7)
    q = rng.integers(0, 256, size=(2, 48), dtype=np.uint8)
    s = np.array([[120, 127, 130], [1, 200, 64]], dtype=np.uint8)
    got = oracle.dequant(q, s, 2, 96)
    for r in range(2):
        for c in range(96):
            byte = int(q[r, c // 2])
            code = byte & 0xF if c % 2 == 0 else byte >> 4
            expect = _golden_table()[code] * 2.0 ** (int(s[r, c // 32]) - 127)
            assert _same(float(got[r, c]), expect)


def _f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def _bits_f32(u: int) -> float:
    return struct.unpack("<f", struct.pack("<I", u & 0xFFFFFFFF))[0]


def test_scale_as_integer_exponent_add():
    # For every nonzero code and every scale whose result stays a normal fp32,
    # adding (e - 127) to the fp32 exponent field of the table value gives the
    # oracle's decoded element.
    for c in range(16):
        v = oracle.e2m1(c)
        if v == 0.0:
            continue
        bits = _f32_bits(v)
        exp = (bits >> 23) & 0xFF
        for e in range(255):
            ne = exp + (e - 127)
            if not (1 <= ne <= 254):
                continue
            shifted = (bits & ~(0xFF << 23)) | (ne << 23)
            q = np.array([[c | (c << 4)] + [0] * 15], dtype=np.uint8)
            s = np.array([[e]], dtype=np.uint8)
            assert oracle.dequant(q, s, 1, 32)[0, 0] == _bits_f32(shifted), (c, e)


def test_orc_mx_at_agrees_with_dequant():
    import synth
    q, s = synth.mx_matrix(synth.key(3, 9), 8, 128)
    d = oracle.dequant(q, s, 8, 128)
    L = oracle.lib()
    for r in (0, 3, 7):
        for c in (0, 1, 31, 32, 77, 127):
            assert L.orc_mx_at(q.ctypes.data, s.ctypes.data, 128, r, c) == d[r, c]


def test_dequant_rejects_bad_shape():
    with pytest.raises(ValueError):
        oracle.dequant(np.zeros((1, 10), np.uint8), np.zeros((1, 1), np.uint8), 1, 20)
