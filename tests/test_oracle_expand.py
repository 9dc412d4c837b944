"""Pins of the oracle's EAGLE-2 expand + rerank (CPU only).

[EAGLE-2] §2 "EAGLE-2 的核心創新：動態草稿樹", items 1-3: each draft node gets a
confidence, expansion adapts to it, and a fixed draft-token budget is spent
greedily to maximise the expected acceptance length.  Pinned by a
hand-worked example, a library-sort special case, a full-vocabulary beam
search, brute-force optimality of the rerank and structural invariants.
"""
import itertools
import math
import os

import numpy as np
import pytest

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(seed, B, R, V, sigma=3.0):
    lp, _ = synth.draft_rows(seed, "expand-test", B * R, V, sigma)
    return lp


def test_hand_worked_example():
    # golden/expand_hand_worked.txt: V=4, k=2, depth=2, budget=4
    vals = {}
    with open(os.path.join(GOLDEN, "expand_hand_worked.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, rest = line.split("=", 1)
                vals[key.strip()] = rest.split()
    rows = np.array([float(x) for x in vals["logp"]], np.float32).reshape(3, 4)
    tree = O.build_eagle2_tree(rows, B=1, k=2, depth=2, budget=[int(vals["budget"][0])], root_token=[99])
    assert list(tree["parent"]) == [int(x) for x in vals["parent"]]
    assert list(tree["tokens"]) == [int(x) for x in vals["tokens"]]
    assert list(tree["depth"]) == [int(x) for x in vals["depth"]]
    assert list(tree["p_row_of_node"]) == [int(x) for x in vals["p_row_of_node"]]
    np.testing.assert_array_equal(tree["score"],
                                  np.array([float(x) for x in vals["score"]], np.float32))


def test_depth_one_tree_is_the_sorted_top_of_the_root_row():
    V, k = 50, 7
    row = _rows(1, 1, 1, V)
    row[0, 3] = row[0, 10] = row[0].max()        # a tie: lower token first
    for budget in (1, 4, 7, 20):
        tree = O.build_eagle2_tree(row, B=1, k=k, depth=1, budget=[budget], root_token=[0])
        order = np.argsort(-row[0], kind="stable")[:min(k, budget)]
        assert list(tree["tokens"][1:]) == list(order)
        assert list(tree["parent"]) == [-1] + [0] * len(order)
        np.testing.assert_array_equal(tree["score"][1:], row[0, order])


def _beam_full_vocab(rows, k, depth):
    """Beam search of width k over the FULL vocabulary: the frontier at each
    level is the k best of all (frontier node, token) extensions, ties by
    frontier rank then token.  Returns the frontier token paths per level."""
    V = rows.shape[1]
    frontier = [((), np.float32(0))]
    levels = []
    for d in range(depth):
        cand = []
        for f, (path, sc) in enumerate(frontier):
            row = rows[0] if d == 0 else rows[1 + (d - 1) * k + f]
            for t in range(V):
                cand.append((-float(np.float32(sc + row[t])), f, t, path + (t,),
                             np.float32(sc + row[t])))
        cand.sort(key=lambda c: (c[0], c[1], c[2]))
        frontier = [(c[3], c[4]) for c in cand[:k]]
        levels.append([c[3] for c in cand[:k]])
    return levels


def test_frontier_equals_full_vocabulary_beam_search():
    for seed in range(5):
        V, k, depth = 9, 3, 4
        R = 1 + (depth - 1) * k
        rows = _rows(10 + seed, 1, R, V, sigma=1.0)
        pools = [O.eagle_oracle._Pool()]
        beam = _beam_full_vocab(rows, k, depth)
        for lev in range(depth):
            O.expand_level(pools, rows, lev, k, R)
            pool = pools[0]

            def path_of(j):
                toks = []
                while j >= 0:
                    toks.append(pool.token[j])
                    j = pool.parent[j]
                return tuple(toks[::-1])
            assert [path_of(j) for j in pool.frontier] == beam[lev]


def test_rerank_maximises_total_path_value_by_brute_force():
    V, k, depth = 4, 2, 3
    R = 1 + (depth - 1) * k
    for seed in range(6):
        rows = _rows(20 + seed, 1, R, V, sigma=1.5)
        pools = [O.eagle_oracle._Pool()]
        for lev in range(depth):
            O.expand_level(pools, rows, lev, k, R)
        pool = pools[0]
        n = len(pool.token)
        assert n == k + (depth - 1) * k * k
        for budget in (1, 3, 5):
            best, best_sets = -1.0, []
            for sub in itertools.combinations(range(n), budget):
                s = set(sub)
                if any(pool.parent[j] >= 0 and pool.parent[j] not in s for j in sub):
                    continue
                val = sum(math.exp(float(pool.score[j])) for j in sub)
                if val > best + 1e-12:
                    best, best_sets = val, [s]
                elif abs(val - best) <= 1e-12:
                    best_sets.append(s)
            tree = O.expand_finalize([pool], [budget], [0], R)
            got = sum(math.exp(float(x)) for x in tree["score"][1:])
            assert abs(got - best) < 1e-9


@pytest.mark.parametrize("B,V,k,depth,budgets", [
    (1, 64, 4, 3, [10]),
    (3, 100, 5, 4, [1, 17, 200]),
    (2, 33, 8, 5, [64, 40]),
])
def test_tree_invariants(B, V, k, depth, budgets):
    R = 1 + (depth - 1) * k
    rows = _rows(B * 100 + V, B, R, V)
    tree = O.build_eagle2_tree(rows, B=B, k=k, depth=depth, budget=budgets,
                               root_token=list(range(B)))
    pool_n = k + (depth - 1) * k * k
    off = tree["tree_off"]
    for b in range(B):
        t0, t1 = off[b], off[b + 1]
        assert t1 - t0 == min(budgets[b], pool_n) + 1
        par = tree["parent"][t0:t1]
        assert par[0] == -1
        for i in range(1, t1 - t0):
            p = par[i]
            assert 0 <= p < i
            assert tree["depth"][t0 + i] == tree["depth"][t0 + p] + 1
            assert tree["score"][t0 + i] <= tree["score"][t0 + p]
            row = tree["p_row_of_node"][t0 + i]
            assert row // R == b
            want = np.float32(tree["score"][t0 + p] + rows[row, tree["tokens"][t0 + i]])
            assert tree["score"][t0 + i] == want
        for i in range(t1 - t0):
            kids = [j for j in range(t1 - t0) if par[j] == i]
            toks = [tree["tokens"][t0 + j] for j in kids]
            assert len(set(toks)) == len(toks)
            # siblings share the row they were drafted from
            assert len({int(tree["p_row_of_node"][t0 + j]) for j in kids}) <= 1
        # depth ordering then score descending within a depth
        d = tree["depth"][t0:t1]
        assert np.all(np.diff(d) >= 0)


def test_unlimited_budget_keeps_the_whole_pool():
    V, k, depth = 20, 3, 3
    R = 1 + (depth - 1) * k
    rows = _rows(5, 1, R, V)
    tree = O.build_eagle2_tree(rows, B=1, k=k, depth=depth, budget=[10 ** 6], root_token=[1])
    assert len(tree["parent"]) == 1 + k + (depth - 1) * k * k
    # each frontier node of each level has exactly k children
    par = list(tree["parent"])
    counts = np.bincount(np.array(par[1:]), minlength=len(par))
    assert counts[0] == k
    assert sorted(set(counts[1:]) - {0}) == [k]
