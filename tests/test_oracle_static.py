"""Pins of the oracle's EAGLE-1 static draft tree (CPU only).

[EAGLE-2] §2 (EAGLE-1's fixed top-k tree, which the dynamic tree replaces)
and [S4000] "EAGLE的创新点" item 1 (keep the top tokens at every draft step,
K^m candidate paths).  Checked against the pages' path count, a brute-force
definition of "the r-th most probable token", the greedy chain, the dynamic
tree where the two coincide, and the tree invariants."""
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if "=" in line:
                k, v = line.split("=")
                vals[k.strip()] = int(v)
    return vals


def test_full_tree_has_k_to_the_m_paths():
    g = _golden("static_tree_k3_m2.txt")
    parent, rank, row = O.static_template_full(g["K"], g["m"])
    assert len(parent) == g["nodes"]
    leaves = set(range(len(parent))) - set(parent[1:])
    assert len(leaves) == g["paths"]
    # every leaf's path has m drafted tokens
    assert all(len(O.tree_path(parent, i)) == g["m"] + 1 for i in leaves)
    # expanded nodes own distinct rows 0..(#expanded - 1), leaves none
    assert sorted(r for r in row if r >= 0) == list(range(len(parent) - len(leaves)))


def _brute_rank_token(row, r):
    # the token that exactly r others beat (larger value, or equal value and
    # a smaller token id)
    for t in range(len(row)):
        beat = sum(1 for u in range(len(row))
                   if row[u] > row[t] or (row[u] == row[t] and u < t))
        if beat == r:
            return t
    raise AssertionError


@pytest.mark.parametrize("K,m,V", [(3, 2, 7), (2, 3, 5), (4, 1, 4)])
def test_children_are_the_ranked_tokens_by_brute_force(K, m, V):
    parent, rank, row = O.static_template_full(K, m)
    R = max(row) + 1
    B = 2
    g = np.random.default_rng(K * 10 + m)
    # values on a coarse grid, so ties between tokens are common
    lp = (np.round(g.standard_normal((B, R, V)) * 2) / 2 - 5).astype(np.float32)
    tree = O.build_static_tree(lp, B, parent, rank, row, root_token=[11, 22])
    n = len(parent)
    for b in range(B):
        for i in range(1, n):
            p = parent[i]
            want = _brute_rank_token(lp[b, row[p]], rank[i])
            assert tree["tokens"][b * n + i] == want
            assert tree["score"][b * n + i] == np.float32(
                tree["score"][b * n + p] + lp[b, row[p], want])
            assert tree["p_row_of_node"][b * n + i] == b * R + row[p]
        assert tree["tokens"][b * n] == [11, 22][b]


def test_rank_zero_chain_is_greedy_drafting():
    V, m = 9, 4
    parent = [-1] + list(range(m))
    rank = [0] * (m + 1)
    row = list(range(m)) + [-1]
    lp = synth.draft_rows(3, "static-chain", m, V, 2.0)[0]
    tree = O.build_static_tree(lp, 1, parent, rank, row, root_token=[0])
    for d in range(m):
        assert tree["tokens"][d + 1] == int(np.argmax(lp[d]))


def test_one_level_full_tree_equals_the_dynamic_tree_with_budget_k():
    # depth 1, K children of the root: the static tree and the EAGLE-2 tree
    # of budget K both keep the root's top-K tokens, numbered by score
    V, K = 50, 6
    lp = synth.draft_rows(5, "static-vs-dynamic", 2, V, 3.0)[0]
    parent, rank, row = O.static_template_full(K, 1)
    st = O.build_static_tree(lp[:1], 1, parent, rank, row, root_token=[7])
    dy = O.build_eagle2_tree(lp[:1], B=1, k=K, depth=1, budget=[K], root_token=[7])
    for key in ("tree_off", "parent", "tokens", "depth", "score", "p_row_of_node"):
        np.testing.assert_array_equal(st[key], dy[key], err_msg=key)


def test_tree_invariants():
    K, m, V = 3, 3, 40
    parent, rank, row = O.static_template_full(K, m)
    R = max(row) + 1
    lp = synth.draft_rows(9, "static-inv", 2 * R, V, 3.0)[0].reshape(2, R, V)
    tree = O.build_static_tree(lp, 2, parent, rank, row, root_token=[1, 2])
    n = len(parent)
    for b in range(2):
        par = tree["parent"][b * n:(b + 1) * n]
        tok = tree["tokens"][b * n:(b + 1) * n]
        sc = tree["score"][b * n:(b + 1) * n]
        dep = tree["depth"][b * n:(b + 1) * n]
        for i in range(1, n):
            assert 0 <= par[i] < i
            assert sc[i] <= sc[par[i]]
            assert dep[i] == dep[par[i]] + 1
        for p in set(par[1:]):
            kids = [tok[i] for i in range(1, n) if par[i] == p]
            assert len(set(kids)) == len(kids)


def test_non_finite_draft_row_is_a_numeric_error():
    parent, rank, row = O.static_template_full(2, 1)
    lp = np.zeros((1, 1, 4), np.float32)
    lp[0, 0, 2] = np.nan
    with pytest.raises(O.OracleNumericError):
        O.build_static_tree(lp, 1, parent, rank, row, root_token=[0])
