"""Checks of the seeded input generator (input bytes, not the layer)."""
import numpy as np
import pytest

import oracle
import synth
from test_oracle_mlp import decode_mx


def test_normal_moments_and_bounds():
    z = synth.normal(synth.key(0, 1), 400_000)
    assert abs(z.mean()) < 0.01
    assert abs(z.var() - 1.0) < 0.01
    assert z.min() >= -6.0 and z.max() <= 6.0
    # Values are multiples of 2^-16 (integer sum / 65536).
    assert np.all(np.mod(z.astype(np.float64) * 65536.0, 1.0) == 0.0)


def test_streams_are_deterministic_and_thread_count_free():
    L = synth.lib()
    k = synth.key(0, 2)
    a = np.empty(10_001, np.float32)
    b = np.empty(10_001, np.float32)
    L.syn_fill_f32(k, a.size, 0.02, a.ctypes.data, 1)
    L.syn_fill_f32(k, b.size, 0.02, b.ctypes.data, 7)
    np.testing.assert_array_equal(a, b)
    assert synth.key(0, 2) != synth.key(1, 2) != synth.key(0, 3)


def test_bf16_rounding_is_nearest_even():
    L = synth.lib()
    vals = np.array([1.0, 1.00390625, 1.01171875, -2.5, 3.0e38, 1e-40, 0.0, -0.0], dtype=np.float32)
    for v in vals:
        assert L.syn_bf16_c(float(v)) == synth.bf16_bits(np.array([v]))[0]
    # Ties: 1 + 2^-8 is halfway between bf16 1.0 and 1 + 2^-7 -> even (1.0).
    assert synth.bf16_bits(np.array([1.00390625], np.float32))[0] == 0x3F80
    # 1 + 3*2^-8 is halfway between 1+2^-7 (odd) and 1+2^-6 (even) -> 1+2^-6.
    assert synth.bf16_bits(np.array([1.01171875], np.float32))[0] == 0x3F82


def test_quantiser_error_within_half_step():
    rng = np.random.default_rng(0)
    v = 0.02 * rng.standard_normal(32 * 64)
    q, s = synth.quant_row(v)
    d = decode_mx(q, s, 1, v.size)[0]
    for b in range(64):
        blk = v[32 * b:32 * b + 32]
        X = int(np.floor(np.log2(np.abs(blk).max()))) - 2
        assert s[b] == X + 127
        step = 2.0 ** X
        err = np.abs(d[32 * b:32 * b + 32] - blk)
        # Within the grid (|v| <= 6 step) the largest gap is 2 step (4 -> 6);
        # above it, values up to amax < 8 step saturate to 6 step.
        inside = np.abs(blk) <= 6 * step
        assert np.all(err[inside] <= step + 1e-18)
        assert np.all(err[~inside] < 2 * step)
        # Below magnitude 2 the gaps are 0.5: error <= 0.25 step.
        small = np.abs(blk) / step < 1.75
        assert np.all(err[small] <= 0.25 * step + 1e-18)


def test_quantiser_special_blocks():
    q, s = synth.quant_row(np.zeros(32))
    assert s[0] == 0 and np.all(q == 0)
    # Exact grid values at scale 2^-1: amax = 3 -> X = floor(log2 3) - 2 = -1.
    v = np.array([0, .25, .5, .75, 1, 1.5, 2, 3] * 4, dtype=np.float64)
    q, s = synth.quant_row(v)
    assert s[0] == 126
    np.testing.assert_array_equal(decode_mx(q, s, 1, 32)[0], v)
    # Saturation: 7.5 * 2^X rounds to 6 (the grid's largest magnitude).
    v = np.zeros(32)
    v[0] = 7.9
    v[1] = -7.9
    q, s = synth.quant_row(v)
    d = decode_mx(q, s, 1, 32)[0]
    assert d[0] == 6.0 and d[1] == -6.0


def test_quantiser_ties_to_even_code():
    # Ties at 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5 (times the scale) go to the
    # code whose mantissa bit is 0.
    v = np.array([6.0, 0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0] + [0.0] * 24)
    q, s = synth.quant_row(v)
    assert s[0] == 127
    d = decode_mx(q, s, 1, 32)[0][:8]
    np.testing.assert_array_equal(d, [6.0, 0.0, 1.0, 1.0, 2.0, 2.0, 4.0, 4.0])


def test_mx_matrix_rows_are_independent_of_thread_split():
    L = synth.lib()
    k = synth.key(0, 0x10000)
    q1 = np.empty((40, 64), np.uint8)
    s1 = np.empty((40, 4), np.uint8)
    q2 = np.empty_like(q1)
    s2 = np.empty_like(s1)
    L.syn_fill_mx(k, 40, 128, q1.ctypes.data, s1.ctypes.data, 1)
    L.syn_fill_mx(k, 40, 128, q2.ctypes.data, s2.ctypes.data, 5)
    np.testing.assert_array_equal(q1, q2)
    np.testing.assert_array_equal(s1, s2)


def test_workload_shapes():
    wl = synth.WORKLOADS["decode"]
    assert wl.expert_bytes == 16_084_992
    assert synth.WORKLOADS["decode_i1536"].expert_bytes == 17_547_264
    assert wl.flops_per_token == 968_884_224 + 12_845_056


def test_planted_wide_routing_selects_the_planted_sets():
    wl = synth.WORKLOADS["wide"]
    inp = synth.make_inputs(wl)
    s = oracle.router_logits(inp.x, inp.wr)
    ids, w, margin = oracle.topk(s, wl.k)
    shared, private = synth.planted_sets(wl)
    union = set()
    for t in range(wl.T):
        assert set(ids[t]) == set(shared) | set(private[t])
        union |= set(ids[t])
    assert len(union) == 72
    # Planted margins are wide: no near-tie at the selection boundary.
    srt = np.sort(s, axis=1)[:, ::-1]
    assert np.all(srt[:, 15] - srt[:, 16] > 10.0)


def test_zipf_tau_record():
    import json
    with open(synth.ZIPF_TAU_FILE) as f:
        rec = json.load(f)
    assert 900 <= rec["max_load"] <= 1100
    assert rec["T"] == 4096 and rec["k"] == 16 and rec["E"] == 896
    b = synth.zipf_bias(synth.WORKLOADS["long"], rec["tau"])
    assert b.dtype == np.float32 and b.shape == (896,)
    # Popularity is a permutation of ranks: one expert per rank.
    lp = synth.zipf_log_popularity(synth.WORKLOADS["long"])
    assert np.isclose(np.exp(lp).sum(), 1.0)
    assert len(np.unique(lp)) == 896
