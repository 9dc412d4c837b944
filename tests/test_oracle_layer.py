"""Pins of the oracle's decoder layer over the tree (CPU only).

The defining property ([EAGLE] workflow paragraph; [S4000] "EAGLE的创新点"
item 2): one forward pass over the tree gives every node the output it would
have as the last token of its own root-to-node path run as an ordinary
causal sequence after the cached context, at positions cache length + depth.
Checked against an independent causal layer, plus closed forms of the
rotary embedding, RMSNorm, SiLU and the bf16 rounding."""
import numpy as np
import pytest

import oracle as O
import synth


def _weights(seed, H, Hq, Hkv, D, I, std=0.05):
    g = np.random.default_rng(seed)
    bf = O.bf16_round
    return {"g_attn": bf(1 + 0.1 * g.standard_normal(H)),
            "wq": bf(std * g.standard_normal((Hq * D, H))),
            "wk": bf(std * g.standard_normal((Hkv * D, H))),
            "wv": bf(std * g.standard_normal((Hkv * D, H))),
            "wo": bf(std * g.standard_normal((H, Hq * D))),
            "g_mlp": bf(1 + 0.1 * g.standard_normal(H)),
            "wg": bf(std * g.standard_normal((I, H))),
            "wu": bf(std * g.standard_normal((I, H))),
            "wd": bf(std * g.standard_normal((H, I)))}


def test_tree_layer_equals_the_causal_layer_on_every_path():
    H, Hq, Hkv, D, I = 32, 4, 2, 8, 48
    theta, eps = 10000.0, 1e-5
    w = _weights(1, H, Hq, Hkv, D, I)
    g = np.random.default_rng(2)
    Ls = [5, 0, 3]
    parents = [synth.random_level_tree(10 + b, (1, 3, 3, 2), 9)[0] for b in range(3)]
    sizes = [len(p) for p in parents]
    tree_off = np.concatenate([[0], np.cumsum(sizes)])
    kv_off = np.concatenate([[0], np.cumsum(Ls)])
    parent = np.concatenate(parents)
    T = int(tree_off[-1])
    x = g.standard_normal((T, H))
    kc = O.bf16_round(g.standard_normal((int(kv_off[-1]), Hkv, D)))
    vc = O.bf16_round(g.standard_normal((int(kv_off[-1]), Hkv, D)))
    res = O.decoder_layer(x, w, kc, vc, kv_off, tree_off, parent, Hq, Hkv, theta, eps)
    for b in range(3):
        t0, t1 = int(tree_off[b]), int(tree_off[b + 1])
        c0, c1 = int(kv_off[b]), int(kv_off[b + 1])
        par = parent[t0:t1]
        for i in range(t1 - t0):
            path = [t0 + j for j in O.tree_path(par, i)]
            ref = O.decoder_layer_causal(x[path], w, kc[c0:c1], vc[c0:c1], c1 - c0, Hq, Hkv,
                                         theta, eps)
            np.testing.assert_allclose(res["out"][path], ref, rtol=1e-10, atol=1e-10)
            assert res["pos"][t0 + i] == (c1 - c0) + len(path) - 1


def test_rope_closed_forms():
    g = np.random.default_rng(3)
    D, theta = 8, 10000.0
    x = g.standard_normal((5, 3, D))
    pos = np.array([0, 1, 7, 100, 16383])
    r = O.rope(x, pos, theta)
    # position 0 is the identity; every (j, j + D/2) pair keeps its length
    np.testing.assert_allclose(r[0], x[0], rtol=0, atol=0)
    n_in = x[..., :D // 2] ** 2 + x[..., D // 2:] ** 2
    n_out = r[..., :D // 2] ** 2 + r[..., D // 2:] ** 2
    np.testing.assert_allclose(n_out, n_in, rtol=1e-12)
    # pair j turns by pos * theta^(-2j/D): pair 0 by pos radians exactly
    ang = np.arctan2(r[:, :, D // 2], r[:, :, 0]) - np.arctan2(x[:, :, D // 2], x[:, :, 0])
    np.testing.assert_allclose(np.cos(ang), np.broadcast_to(np.cos(pos)[:, None], ang.shape),
                               atol=1e-9)
    # scores depend only on the distance between positions
    q, k = g.standard_normal((1, 1, D)), g.standard_normal((1, 1, D))
    s1 = np.sum(O.rope(q, [9], theta) * O.rope(k, [4], theta))
    s2 = np.sum(O.rope(q, [109], theta) * O.rope(k, [104], theta))
    assert abs(s1 - s2) < 1e-12


def test_rmsnorm_and_silu_closed_forms():
    g = np.random.default_rng(4)
    x = g.standard_normal((3, 16))
    y = O.rmsnorm(x, np.ones(16), 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, axis=1)), 1.0, rtol=1e-12)
    np.testing.assert_allclose(O.rmsnorm(7.5 * x, np.ones(16), 0.0), y, rtol=1e-12)
    gain = g.standard_normal(16)
    np.testing.assert_allclose(O.rmsnorm(x, gain, 0.0), y * gain, rtol=1e-12)
    v = g.standard_normal(20)
    np.testing.assert_allclose(O.silu(v) - O.silu(-v), v, rtol=1e-12, atol=1e-15)
    assert O.silu(0.0) == 0.0


def test_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    g = np.random.default_rng(5)
    x = np.concatenate([g.standard_normal(10000) * 10.0 ** g.integers(-8, 8, 10000),
                        [0.0, -0.0, 1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8]]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(x), ref)


def test_zero_output_projections_leave_the_residual_stream():
    H, Hq, Hkv, D, I = 16, 2, 1, 8, 24
    w = _weights(6, H, Hq, Hkv, D, I)
    w["wo"] = np.zeros_like(w["wo"])
    w["wd"] = np.zeros_like(w["wd"])
    x = np.random.default_rng(7).standard_normal((4, H))
    res = O.decoder_layer(x, w, np.zeros((2, Hkv, D)), np.zeros((2, Hkv, D)), [0, 2],
                          [0, 4], [-1, 0, 1, 1], Hq, Hkv, 10000.0, 1e-5, with_abs=True)
    np.testing.assert_array_equal(res["out"], x)
    np.testing.assert_array_equal(res["out_abs"], np.abs(x))
    np.testing.assert_array_equal(res["pos"], [2, 3, 4, 4])
