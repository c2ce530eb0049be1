"""Pins of the oracle's expert MLP and combine against independent numpy code.

A one-hot route reduces the layer to a dense SwiGLU MLP; the combine is the
slot-ordered weighted sum [Deltafin's custom compiled runtime, "The native
build": ordered reduction]; all selected experts run [Deltafin's custom
compiled runtime, "Weight fidelity"].  The numpy side decodes MXFP4 from the
bit fields (not from the oracle's table) and uses scipy's expit for silu.
"""
import numpy as np
import pytest
import scipy.special

import oracle
import synth


def decode_mx(q, s, rows, cols):
    """Independent MXFP4 decoder: sign / exponent (bias 1) / mantissa fields."""
    q = np.asarray(q, dtype=np.uint8).reshape(rows, cols // 2)
    codes = np.empty((rows, cols), dtype=np.int64)
    codes[:, 0::2] = q & 0xF
    codes[:, 1::2] = q >> 4
    sign, E, m = codes >> 3, (codes >> 1) & 3, codes & 1
    mag = np.where(E == 0, m * 0.5, (1.0 + m / 2.0) * np.exp2(E - 1.0))
    val = np.where(sign == 1, -mag, mag)
    se = np.asarray(s, dtype=np.int64).reshape(rows, cols // 32)
    scale = np.where(se == 255, np.nan, np.exp2(se - 127.0))
    return val * np.repeat(scale, 32, axis=1)


def dense_swiglu(x, wg, wu, wd):
    g = wg @ x
    u = wu @ x
    h = g * scipy.special.expit(g) * u
    return wd @ h


def _expert(seed, e, H, I):
    gq, gs = synth.mx_matrix(synth.key(seed, 100 + 3 * e), I, H)
    uq, us = synth.mx_matrix(synth.key(seed, 101 + 3 * e), I, H)
    dq, ds = synth.mx_matrix(synth.key(seed, 102 + 3 * e), H, I)
    return dict(gate_q=gq, gate_s=gs, up_q=uq, up_s=us, down_q=dq, down_s=ds)


def _dense_of(ex, H, I):
    return (decode_mx(ex["gate_q"], ex["gate_s"], I, H), decode_mx(ex["up_q"], ex["up_s"], I, H),
            decode_mx(ex["down_q"], ex["down_s"], H, I))


@pytest.mark.parametrize("H,I", [(64, 96), (96, 32), (256, 128)])
def test_expert_mlp_is_dense_swiglu(H, I):
    ex = _expert(1, 0, H, I)
    x = np.random.default_rng(H + I).standard_normal(H)
    y = oracle.expert_mlp(H, I, x, ex)
    ref = dense_swiglu(x, *_dense_of(ex, H, I))
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-13)


def test_one_hot_route_is_dense_mlp():
    # k = 1: out[t] = residual[t] + y_{e*}(x_t) with weight exactly 1.
    T, H, E, I = 5, 64, 3, 96
    rng = np.random.default_rng(0)
    x = rng.standard_normal((T, H)).astype(np.float32)
    wr = (0.02 * rng.standard_normal((E, H))).astype(np.float32)
    experts = {e: _expert(2, e, H, I) for e in range(E)}
    residual = rng.standard_normal((T, H)).astype(np.float32)
    out, ids, w = oracle.moe_tokens(x, wr, None, experts, E, I, 1, np.arange(T), residual=residual)
    assert np.all(w == 1.0)
    s = x.astype(np.float64) @ wr.astype(np.float64).T
    for t in range(T):
        e = int(np.argmax(s[t]))
        assert ids[t, 0] == e
        ref = residual[t].astype(np.float64) + dense_swiglu(x[t].astype(np.float64), *_dense_of(experts[e], H, I))
        np.testing.assert_allclose(out[t], ref, rtol=1e-11, atol=1e-12)


def test_single_expert_layer_is_textbook_mlp():
    H, I = 32, 64
    x = np.random.default_rng(1).standard_normal((2, H)).astype(np.float32)
    wr = np.ones((1, H), dtype=np.float32)
    ex = _expert(3, 0, H, I)
    out, ids, w = oracle.moe_tokens(x, wr, None, {0: ex}, 1, I, 1, np.arange(2))
    for t in range(2):
        np.testing.assert_allclose(out[t], dense_swiglu(x[t].astype(np.float64), *_dense_of(ex, H, I)),
                                   rtol=1e-11, atol=1e-12)


def test_topk_combine_is_weighted_sum():
    T, H, E, I, k = 4, 64, 6, 32, 3
    rng = np.random.default_rng(5)
    x = synth.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.05 * rng.standard_normal((E, H))).astype(np.float32)
    br = rng.standard_normal(E).astype(np.float32)
    experts = {e: _expert(4, e, H, I) for e in range(E)}
    out, ids, w = oracle.moe_tokens(x, wr, br, experts, E, I, k, np.arange(T))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    s = xf @ wr.astype(np.float64).T + br.astype(np.float64)
    for t in range(T):
        top = sorted(range(E), key=lambda e: (-s[t, e], e))[:k]
        assert list(ids[t]) == top
        wt = scipy.special.softmax(s[t, top])
        ref = sum(wt[j] * dense_swiglu(xf[t], *_dense_of(experts[top[j]], H, I)) for j in range(k))
        np.testing.assert_allclose(out[t], ref, rtol=1e-10, atol=1e-12)


def test_residual_linearity_and_token_subset():
    T, H, E, I, k = 6, 64, 5, 32, 2
    rng = np.random.default_rng(8)
    x = rng.standard_normal((T, H)).astype(np.float32)
    wr = (0.05 * rng.standard_normal((E, H))).astype(np.float32)
    experts = {e: _expert(5, e, H, I) for e in range(E)}
    res = rng.standard_normal((T, H)).astype(np.float32)
    sel = np.array([4, 1, 1], dtype=np.int32)
    o0, ids0, _ = oracle.moe_tokens(x, wr, None, experts, E, I, k, sel)
    o1, ids1, _ = oracle.moe_tokens(x, wr, None, experts, E, I, k, sel, residual=res)
    np.testing.assert_allclose(o1, o0 + res[sel].astype(np.float64), rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(o0[1], o0[2])
    full, _, _ = oracle.moe_tokens(x, wr, None, experts, E, I, k, np.arange(T))
    np.testing.assert_array_equal(full[4], o0[0])


def test_shared_expert_adds_dense_bf16_mlp():
    T, H, E, I, k = 3, 64, 4, 32, 2
    rng = np.random.default_rng(9)
    x = synth.bf16_bits(rng.standard_normal((T, H)).astype(np.float32))
    wr = (0.05 * rng.standard_normal((E, H))).astype(np.float32)
    experts = {e: _expert(6, e, H, I) for e in range(E)}
    sg = synth.bf16_bits((0.05 * rng.standard_normal((I, H))).astype(np.float32))
    su = synth.bf16_bits((0.05 * rng.standard_normal((I, H))).astype(np.float32))
    sd = synth.bf16_bits((0.05 * rng.standard_normal((H, I))).astype(np.float32))
    o0, _, _ = oracle.moe_tokens(x, wr, None, experts, E, I, k, np.arange(T))
    o1, _, _ = oracle.moe_tokens(x, wr, None, experts, E, I, k, np.arange(T), shared=(sg, su, sd))
    xf = synth.bf16_to_f32(x).astype(np.float64)
    dec = lambda a: synth.bf16_to_f32(a).astype(np.float64)
    for t in range(T):
        ref = dense_swiglu(xf[t], dec(sg), dec(su), dec(sd))
        np.testing.assert_allclose(o1[t] - o0[t], ref, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(oracle.dense_mlp_bf16(H, I, xf[t], sg, su, sd), ref, rtol=1e-12, atol=1e-14)


def test_missing_expert_is_an_error():
    H, I = 32, 32
    x = np.ones((1, H), dtype=np.float32)
    wr = np.ones((2, H), dtype=np.float32)
    with pytest.raises((KeyError, ValueError)):
        oracle.moe_tokens(x, wr, None, {1: _expert(7, 1, H, I)}, 2, I, 1, np.arange(1))
