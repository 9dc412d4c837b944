"""Pins of the oracle's draft loop pieces (CPU only): the draft head, the
draft distribution from the frozen LM head, and the level-by-level EAGLE-2
tree ([EAGLE] workflow paragraph; [EAGLE-2] §2 dynamic draft tree)."""
import numpy as np

import oracle as O
import synth


def test_draft_head_closed_form():
    H = 16
    g = np.random.default_rng(1)
    f, e = g.standard_normal(H), g.standard_normal(H)
    # Wd = [0 | I]: the next feature is the token's embedding (rounded)
    wd = np.concatenate([np.zeros((H, H)), np.eye(H)], axis=1)
    np.testing.assert_array_equal(O.draft_head(f, e, wd), O.bf16_round(e))
    wd2 = np.concatenate([np.eye(H), np.eye(H)], axis=1)
    np.testing.assert_array_equal(O.draft_head(f, e, wd2), O.bf16_round(f + e))


def test_draft_row_is_a_log_distribution():
    g = np.random.default_rng(2)
    w = g.standard_normal((50, 8))
    f = g.standard_normal(8)
    lp = O.draft_logp_row(f, w)
    assert lp.dtype == np.float32
    assert abs(np.exp(lp.astype(np.float64)).sum() - 1.0) < 1e-5
    assert int(np.argmax(lp)) == int(np.argmax(w @ f))


def test_level_by_level_tree_equals_the_tree_of_its_own_rows():
    # drafting with the head, then rebuilding the tree from the rows it
    # produced, gives the same tree; feeding those rows back gives them again
    H, V, B, k, depth = 16, 40, 2, 3, 4
    g = np.random.default_rng(3)
    emb = O.bf16_round(g.standard_normal((V, H)))
    wd = O.bf16_round(g.standard_normal((H, 2 * H)) * 0.2)
    wl = O.bf16_round(g.standard_normal((V, H)) * 0.5)
    f_ctx = O.bf16_round(g.standard_normal((B, H)))
    root = [5, 9]
    budget = [10, 7]
    tree, rows, scale = O.build_eagle2_tree_with_head(f_ctx, root, emb, wd, wl, B, k, depth,
                                                      budget)
    assert np.all(scale[:, 0] > 0)
    ref = O.build_eagle2_tree(rows, B=B, k=k, depth=depth, budget=budget, root_token=root)
    for key in ("tree_off", "parent", "tokens", "depth", "score", "p_row_of_node"):
        np.testing.assert_array_equal(tree[key], ref[key], err_msg=key)
    tree2, rows2, _ = O.build_eagle2_tree_with_head(f_ctx, root, emb, wd, wl, B, k, depth,
                                                    budget, rows=rows)
    np.testing.assert_array_equal(rows2, rows)
    np.testing.assert_array_equal(tree2["tokens"], tree["tokens"])
    # the root's row is the head applied to the context and the root token
    f_root = O.draft_head(f_ctx[0], emb[root[0]], wd)
    np.testing.assert_array_equal(rows[0, 0], O.draft_logp_row(f_root, wl))
