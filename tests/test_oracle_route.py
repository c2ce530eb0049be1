"""Pins of the oracle's router, top-k and bucketing.

Routing: the k largest router scores per token with fp32 weights renormalised
over the k, in route order [Deltafin's custom compiled runtime, "Complete target
sequence tape"]; ties go to the lower expert index.  Bucketing: a counting sort
of the (token, slot) pairs by expert, ordered by route union [Deltafin's custom
compiled runtime, "Exact next-layer expert prefetch"].
"""
import itertools

import numpy as np
import pytest
import scipy.special

import oracle
import synth


def _rand_router(T, H, E, seed, dtype=np.float32):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((T, H)).astype(np.float32)
    wr = (0.02 * rng.standard_normal((E, H))).astype(np.float32)
    if dtype == np.uint16:
        x = synth.bf16_bits(x)
    return x, wr


def test_logits_match_library_matmul():
    x, wr = _rand_router(5, 96, 11, 0)
    b = np.linspace(-1, 1, 11).astype(np.float32)
    s = oracle.router_logits(x, wr, b)
    ref = x.astype(np.float64) @ wr.astype(np.float64).T + b.astype(np.float64)
    np.testing.assert_allclose(s, ref, rtol=1e-13, atol=1e-13)


def test_logits_bf16_activations_decode_exactly():
    x, wr = _rand_router(3, 64, 5, 1, np.uint16)
    s = oracle.router_logits(x, wr)
    ref = synth.bf16_to_f32(x).astype(np.float64) @ wr.astype(np.float64).T
    np.testing.assert_allclose(s, ref, rtol=1e-13, atol=1e-13)


def test_topk_invariants():
    x, wr = _rand_router(16, 128, 40, 2)
    s = oracle.router_logits(x, wr)
    ids, w, _ = oracle.topk(s, 7)
    for t in range(16):
        assert len(set(ids[t])) == 7
        sel = s[t, ids[t]]
        assert np.all(np.diff(sel) <= 0), "route order is descending score"
        assert abs(w[t].sum() - 1.0) < 1e-14
        assert np.all(np.diff(w[t]) <= 0)
        # Every unselected score is no larger than the smallest selected one.
        rest = np.setdiff1d(np.arange(40), ids[t])
        assert s[t, rest].max() <= sel.min()


def test_topk_weights_are_softmax_of_selected():
    x, wr = _rand_router(9, 64, 20, 3)
    s = oracle.router_logits(x, wr)
    ids, w, _ = oracle.topk(s, 5)
    for t in range(9):
        np.testing.assert_allclose(w[t], scipy.special.softmax(s[t, ids[t]]), rtol=1e-13)


def test_topk_k_equals_E_is_full_softmax():
    x, wr = _rand_router(4, 64, 12, 4)
    s = oracle.router_logits(x, wr)
    ids, w, _ = oracle.topk(s, 12)
    for t in range(4):
        full = scipy.special.softmax(s[t])
        np.testing.assert_allclose(w[t], full[ids[t]], rtol=1e-13)
        assert sorted(ids[t]) == list(range(12))


def test_topk_ties_go_to_lower_index():
    # Duplicate router rows give exactly equal fp64 scores.
    x, wr = _rand_router(6, 64, 10, 5)
    wr[7] = wr[2]
    wr[9] = wr[2]
    wr[4] = wr[1]
    s = oracle.router_logits(x, wr)
    assert np.all(s[:, 7] == s[:, 2]) and np.all(s[:, 9] == s[:, 2])
    ids, w, _ = oracle.topk(s, 10)
    for t in range(6):
        pos = {int(e): j for j, e in enumerate(ids[t])}
        assert pos[2] < pos[7] < pos[9]
        assert pos[1] < pos[4]
        assert w[t][pos[2]] == w[t][pos[7]] == w[t][pos[9]]
    # A k that cuts through a tie keeps the lower indices.
    s2 = np.zeros((1, 10))
    ids2, w2, _ = oracle.topk(s2, 3)
    assert list(ids2[0]) == [0, 1, 2]
    np.testing.assert_allclose(w2[0], [1 / 3] * 3, rtol=1e-15)


@pytest.mark.parametrize("E,k", [(8, 2), (6, 3), (5, 1), (7, 4)])
def test_topk_brute_force_subsets(E, k):
    # The selected set maximises the sum of scores over all k-subsets.
    x, wr = _rand_router(10, 32, E, 10 + E + k)
    s = oracle.router_logits(x, wr)
    ids, w, _ = oracle.topk(s, k)
    for t in range(10):
        best = max(itertools.combinations(range(E), k), key=lambda c: (sum(s[t, list(c)]), [-i for i in c]))
        assert sorted(ids[t]) == sorted(best)


def test_margin_is_smallest_adjacent_gap():
    s = np.array([[5.0, 1.0, 4.0, 4.5, 0.0]])
    ids, w, margin = oracle.topk(s, 2)
    assert list(ids[0]) == [0, 3]
    # sorted: 5, 4.5, 4, 1, 0 -> gaps within first k+1 = 3 entries: 0.5, 0.5
    assert margin[0] == 0.5


def _bucket_brute(ids, E):
    T, k = ids.shape
    pairs = sorted((int(ids[t, j]), t, j) for t in range(T) for j in range(k))
    sorted_idx = np.array([t * k + j for (_, t, j) in pairs], dtype=np.int32)
    counts = np.bincount(ids.ravel(), minlength=E)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, sorted_idx


def test_bucket_matches_sort():
    rng = np.random.default_rng(11)
    for T, E, k in [(1, 8, 2), (5, 8, 2), (33, 17, 4), (64, 50, 16)]:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
        off, srt = oracle.bucket(ids, E)
        off2, srt2 = _bucket_brute(ids, E)
        np.testing.assert_array_equal(off, off2)
        np.testing.assert_array_equal(srt, srt2)
        assert off[-1] == T * k
        for e in range(E):
            seg = srt[off[e]:off[e + 1]]
            assert np.all(np.diff(seg) > 0)
            assert np.all(ids.ravel()[seg] == e)


def test_bucket_zero_load_and_single_hot_expert():
    ids = np.array([[3, 0], [3, 1], [3, 2]], dtype=np.int32)
    off, srt = oracle.bucket(ids, 6)
    assert list(off) == [0, 1, 2, 3, 6, 6, 6]
    assert list(srt) == [1, 3, 5, 0, 2, 4]


def test_bucket_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.bucket(np.array([[0, 9]], dtype=np.int32), 4)
