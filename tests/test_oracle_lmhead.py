"""Pins of the oracle's LM head + softmax + argmax (CPU only).

[EAGLE] workflow paragraph: the frozen LM head turns each node's top-layer
feature into a next-token distribution.  Checked against a naive triple loop,
closed forms (uniform rows, one-hot limit) and invariants.
"""
import math

import numpy as np

import oracle as O


def test_logits_match_naive_triple_loop():
    g = np.random.default_rng(0)
    T, H, V = 3, 5, 7
    h = g.standard_normal((T, H)).astype(np.float32)
    w = g.standard_normal((V, H)).astype(np.float32)
    out = O.lmhead_softmax(h, w, 1.0)
    for t in range(T):
        for v in range(V):
            acc = 0.0
            for i in range(H):
                acc += float(h[t, i]) * float(w[v, i])
            assert abs(out["z"][t, v] - acc) < 1e-12


def test_vocab_blocking_does_not_change_logits():
    g = np.random.default_rng(1)
    h = g.standard_normal((4, 16)).astype(np.float32)
    w = g.standard_normal((37, 16)).astype(np.float32)
    a = O.lmhead_softmax(h, w, 1.0, vocab_chunk=5)
    b = O.lmhead_softmax(h, w, 1.0, vocab_chunk=1 << 20)
    np.testing.assert_allclose(a["z"], b["z"], rtol=1e-14, atol=1e-14)
    np.testing.assert_array_equal(a["q"], b["q"])


def test_softmax_sums_to_one_and_keeps_the_argmax():
    g = np.random.default_rng(2)
    h = g.standard_normal((6, 32)).astype(np.float32)
    w = (0.3 * g.standard_normal((101, 32))).astype(np.float32)
    for temp in (1.0, 0.7, 2.5):
        out = O.lmhead_softmax(h, w, temp)
        q64 = np.exp(out["z"] / temp - out["row_lse"][:, None])
        np.testing.assert_allclose(q64.sum(axis=1), 1.0, rtol=0, atol=1e-12)
        assert np.abs(out["q"].astype(np.float64).sum(axis=1) - 1).max() < 1e-5
        np.testing.assert_array_equal(np.argmax(out["q"], axis=1), out["argmax"])
        np.testing.assert_array_equal(np.argmax(out["z"], axis=1), out["argmax"])


def test_zero_features_give_the_uniform_distribution():
    V = 50
    out = O.lmhead_softmax(np.zeros((2, 8), np.float32),
                           np.ones((V, 8), np.float32), 0.9)
    np.testing.assert_allclose(out["row_lse"], math.log(V), rtol=1e-15)
    np.testing.assert_array_equal(out["q"], np.float32(1.0 / V))
    np.testing.assert_array_equal(out["argmax"], 0)       # all tied: lowest
    np.testing.assert_array_equal(out["top2_gap"], 0.0)


def test_small_temperature_tends_to_one_hot():
    g = np.random.default_rng(3)
    h = g.standard_normal((5, 12)).astype(np.float32)
    w = g.standard_normal((40, 12)).astype(np.float32)
    out = O.lmhead_softmax(h, w, 1e-4)
    for t in range(5):
        assert out["top2_gap"][t] > 1e-2
        assert out["q"][t, out["argmax"][t]] == np.float32(1.0)
        assert out["q"][t].sum() == np.float32(1.0)


def test_ties_take_the_lowest_index_and_gap_counts_duplicates():
    # one feature, weights chosen so that logits are [1, 3, 3, 2]
    w = np.array([[1.0], [3.0], [3.0], [2.0]], np.float32)
    out = O.lmhead_softmax(np.ones((1, 1), np.float32), w, 1.0)
    assert out["argmax"][0] == 1
    assert out["top2_gap"][0] == 0.0
    w[2, 0] = 2.5
    out = O.lmhead_softmax(np.ones((1, 1), np.float32), w, 1.0)
    assert out["argmax"][0] == 1 and abs(out["top2_gap"][0] - 0.5) < 1e-15
    assert abs(out["row_max"][0] - 3.0) < 1e-15
