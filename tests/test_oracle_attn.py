"""Pins of the oracle's tree attention (CPU only).

The defining property ([S4000] "EAGLE的创新点" item 2; [EAGLE] workflow
paragraph): one forward pass over the tree mask scores every root-to-node
path exactly as if that path were run as an ordinary causal sequence after the
cached context.  The oracle's tree routine is checked against an independent
causal-attention routine, plus closed forms.
"""
import numpy as np
import pytest

import oracle as O
import synth


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(B, Ls, level_sizes, Hq, Hkv, D, seed):
    parents, Ts = [], []
    for b in range(B):
        par, _ = synth.random_level_tree(seed + b, level_sizes, 7)
        parents.append(par)
        Ts.append(len(par))
    T = sum(Ts)
    tree_off = np.concatenate([[0], np.cumsum(Ts)]).astype(np.int32)
    kv_off = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    q = _rand((T, Hq, D), seed + 11)
    kt = _rand((T, Hkv, D), seed + 12)
    vt = _rand((T, Hkv, D), seed + 13)
    kc = _rand((int(kv_off[-1]), Hkv, D), seed + 14)
    vc = _rand((int(kv_off[-1]), Hkv, D), seed + 15)
    return q, kt, vt, kc, vc, kv_off, tree_off, np.concatenate(parents)


@pytest.mark.parametrize("B,Ls,levels,Hq,Hkv", [
    (1, [9], (1, 3, 4, 2), 4, 4),
    (2, [5, 0], (1, 2, 3, 3), 4, 2),
    (3, [1, 17, 4], (1, 4, 6, 6, 6, 3), 8, 2),
])
def test_tree_attention_equals_causal_attention_on_every_path(B, Ls, levels, Hq, Hkv):
    D = 8
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(B, Ls, levels, Hq, Hkv, D, 3)
    out = O.tree_attn(q, kt, vt, kc, vc, kv_off, tree_off, parent)
    for b in range(B):
        t0, t1 = tree_off[b], tree_off[b + 1]
        c0, c1 = kv_off[b], kv_off[b + 1]
        par = parent[t0:t1]
        for i in range(t1 - t0):
            path = [t0 + j for j in O.tree_path(par, i)]
            kseq = np.concatenate([kc[c0:c1], kt[path]])
            vseq = np.concatenate([vc[c0:c1], vt[path]])
            ref = O.causal_attn(q[path], kseq, vseq, n_prefix=c1 - c0)
            # every prefix of the path is the path of an ancestor
            np.testing.assert_allclose(out[path], ref, rtol=1e-12, atol=1e-12)


def test_chain_tree_is_plain_causal_attention():
    D, Hq, Hkv, L, N = 16, 4, 2, 13, 7
    g = np.random.default_rng(0)
    q = g.standard_normal((N, Hq, D))
    kt, vt = g.standard_normal((N, Hkv, D)), g.standard_normal((N, Hkv, D))
    kc, vc = g.standard_normal((L, Hkv, D)), g.standard_normal((L, Hkv, D))
    parent = np.arange(-1, N - 1, dtype=np.int32)
    out = O.tree_attn(q, kt, vt, kc, vc, [0, L], [0, N], parent)
    ref = O.causal_attn(q, np.concatenate([kc, kt]), np.concatenate([vc, vt]), L)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12)


def test_single_node_without_cache_returns_its_own_value():
    # softmax over one key is 1: the output is that key's value row
    g = np.random.default_rng(1)
    Hq, Hkv, D = 4, 2, 8
    q = g.standard_normal((1, Hq, D))
    kt, vt = g.standard_normal((1, Hkv, D)), g.standard_normal((1, Hkv, D))
    empty = np.zeros((0, Hkv, D))
    out = O.tree_attn(q, kt, vt, empty, empty, [0, 0], [0, 1], [-1])
    for h in range(Hq):
        np.testing.assert_array_equal(out[0, h], vt[0, h // 2])


def test_equal_keys_give_the_mean_of_the_visible_values():
    # all scores equal -> uniform weights over cache + path: closed form
    g = np.random.default_rng(2)
    Hq = Hkv = 2
    D, L = 4, 5
    parent = np.array([-1, 0, 0, 1, 3], dtype=np.int32)
    N = len(parent)
    q = g.standard_normal((N, Hq, D))
    kt = np.zeros((N, Hkv, D))
    kc = np.zeros((L, Hkv, D))
    vt, vc = g.standard_normal((N, Hkv, D)), g.standard_normal((L, Hkv, D))
    out = O.tree_attn(q, kt, vt, kc, vc, [0, L], [0, N], parent)
    for i in range(N):
        path = O.tree_path(parent, i)
        ref = np.concatenate([vc, vt[path]]).mean(axis=0)
        np.testing.assert_allclose(out[i], ref, rtol=1e-13, atol=1e-14)


def test_star_tree_node_sees_cache_root_and_itself():
    g = np.random.default_rng(3)
    Hq = Hkv = 1
    D, L, N = 8, 3, 6
    parent = np.array([-1] + [0] * (N - 1), dtype=np.int32)
    q = g.standard_normal((N, Hq, D))
    kt, vt = g.standard_normal((N, Hkv, D)), g.standard_normal((N, Hkv, D))
    kc, vc = g.standard_normal((L, Hkv, D)), g.standard_normal((L, Hkv, D))
    out = O.tree_attn(q, kt, vt, kc, vc, [0, L], [0, N], parent)
    for i in range(1, N):
        keys = np.concatenate([kc[:, 0], kt[[0, i], 0]])
        vals = np.concatenate([vc[:, 0], vt[[0, i], 0]])
        s = keys @ q[i, 0] / np.sqrt(D)
        w = np.exp(s - s.max())
        np.testing.assert_allclose(out[i, 0], w @ vals / w.sum(), rtol=1e-12)


def test_gqa_equals_mha_with_repeated_kv_heads():
    # query head h reads kv head h // (Hq/Hkv): repeating each kv head
    # (Hq/Hkv) times and running MHA must give the same result
    Hq, Hkv, D = 8, 2, 8
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(2, [6, 3], (1, 3, 3), Hq, Hkv, D, 9)
    G = Hq // Hkv
    gqa = O.tree_attn(q, kt, vt, kc, vc, kv_off, tree_off, parent)
    rep = lambda a: np.repeat(a, G, axis=1)
    mha = O.tree_attn(q, rep(kt), rep(vt), rep(kc), rep(vc), kv_off, tree_off, parent)
    np.testing.assert_allclose(gqa, mha, rtol=1e-13, atol=1e-14)


def test_sibling_subtrees_do_not_see_each_other():
    # changing the K/V of one branch must leave every node outside that
    # branch's subtree unchanged (the mask hides non-ancestors)
    Hq = Hkv = 2
    D = 8
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(1, [4], (1, 3, 4, 4), Hq, Hkv, D, 21)
    base = O.tree_attn(q, kt, vt, kc, vc, kv_off, tree_off, parent)
    victim = 2
    kt2, vt2 = kt.copy(), vt.copy()
    kt2[victim] += 5.0
    vt2[victim] -= 3.0
    out = O.tree_attn(q, kt2, vt2, kc, vc, kv_off, tree_off, parent)
    for i in range(len(parent)):
        in_subtree = victim in O.tree_path(parent, i)
        same = np.allclose(out[i], base[i], rtol=0, atol=0)
        assert same != in_subtree


def test_abs_scale_is_the_weighted_mean_of_absolute_values():
    # the error scale of an output element, sum_j p_j |v_j|: the same
    # softmax weights applied to |v| (closed form on a star tree), never
    # below |out| (triangle inequality), and equal to out where every v >= 0
    g = np.random.default_rng(5)
    Hq = Hkv = 1
    D, L, N = 8, 4, 5
    parent = np.array([-1] + [0] * (N - 1), dtype=np.int32)
    q = g.standard_normal((N, Hq, D))
    kt, vt = g.standard_normal((N, Hkv, D)), g.standard_normal((N, Hkv, D))
    kc, vc = g.standard_normal((L, Hkv, D)), g.standard_normal((L, Hkv, D))
    out, ab = O.tree_attn(q, kt, vt, kc, vc, [0, L], [0, N], parent, with_abs=True)
    for i in range(1, N):
        keys = np.concatenate([kc[:, 0], kt[[0, i], 0]])
        vals = np.concatenate([vc[:, 0], vt[[0, i], 0]])
        s = keys @ q[i, 0] / np.sqrt(D)
        w = np.exp(s - s.max())
        np.testing.assert_allclose(ab[i, 0], w @ np.abs(vals) / w.sum(), rtol=1e-12)
    assert np.all(ab >= np.abs(out) - 1e-15)
    pos_out, pos_ab = O.tree_attn(q, kt, np.abs(vt), kc, np.abs(vc), [0, L], [0, N], parent,
                                  with_abs=True)
    np.testing.assert_allclose(pos_ab, pos_out, rtol=1e-14)
    # the plain output is unchanged by asking for the scale
    np.testing.assert_array_equal(out, O.tree_attn(q, kt, vt, kc, vc, [0, L], [0, N], parent))


def test_paged_cache_reads_the_same_keys_as_the_packed_cache():
    # scatter each sequence's packed cache over shuffled pages of a pool
    # (page size 4, partial last pages, an empty sequence, unused pool
    # pages): attention over the paged cache equals attention over the packed
    # one exactly, and gathering the pages gives back the packed rows
    g = np.random.default_rng(12)
    Hq, Hkv, D, P = 4, 2, 8, 4
    Ls = [9, 0, 4, 13]
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(4, Ls, (1, 3, 2), Hq, Hkv, D, 31)
    n_pages = sum((L + P - 1) // P for L in Ls) + 3
    perm = g.permutation(n_pages)
    kp = g.standard_normal((n_pages, P, Hkv, D))
    vp = g.standard_normal((n_pages, P, Hkv, D))
    max_pages = max((L + P - 1) // P for L in Ls)
    table = np.full((4, max_pages), -1)
    nxt = 0
    for b, L in enumerate(Ls):
        for j in range((L + P - 1) // P):
            page = perm[nxt]
            nxt += 1
            table[b, j] = page
            for r in range(P):
                pos = j * P + r
                if pos < L:
                    kp[page, r] = kc[kv_off[b] + pos]
                    vp[page, r] = vc[kv_off[b] + pos]
    packed, off = O.gather_pages(kp, table, Ls)
    np.testing.assert_array_equal(packed, kc)
    np.testing.assert_array_equal(off, kv_off)
    ref = O.tree_attn(q, kt, vt, kc, vc, kv_off, tree_off, parent)
    got = O.tree_attn_paged(q, kt, vt, kp, vp, table, Ls, tree_off, parent)
    np.testing.assert_array_equal(got, ref)
    # a table entry outside the pool is an error
    bad = table.copy()
    bad[0, 0] = n_pages
    with pytest.raises(ValueError):
        O.gather_pages(kp, bad, Ls)


def test_commit_appends_the_accepted_path_and_preserves_its_attention():
    # after committing the root and the accepted nodes, the cache is the old
    # cache followed by their K/V rows, and the deepest accepted node's query
    # sees exactly the keys its tree attention saw: the same output
    g = np.random.default_rng(21)
    Hq, Hkv, D, P = 4, 2, 8, 4
    Ls = [5, 0]
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(2, Ls, (1, 3, 3, 3), Hq, Hkv, D, 41)
    n_pages = 12
    kp = g.standard_normal((n_pages, P, Hkv, D))
    vp = g.standard_normal((n_pages, P, Hkv, D))
    table = np.array([[3, 7, 1, 9], [0, 5, 11, 2]])
    for b, L in enumerate(Ls):
        for pos in range(L):
            kp[table[b, pos // P], pos % P] = kc[kv_off[b] + pos]
            vp[table[b, pos // P], pos % P] = vc[kv_off[b] + pos]
    before = O.tree_attn_paged(q, kt, vt, kp, vp, table, Ls, tree_off, parent)
    # an accepted path in each tree: root, then the first child chain
    accept_len, nodes = [], np.full((2, 4), -1)
    for b in range(2):
        par = parent[tree_off[b]:tree_off[b + 1]]
        path, cur = [0], 0
        while True:
            kids = O.tree_children(par, cur)
            if not kids or len(path) == 3:
                break
            cur = kids[-1]
            path.append(cur)
        nodes[b, :len(path)] = path
        accept_len.append(len(path) - 1)
    kp2, vp2, L2 = O.kv_commit_paged(kp, vp, table, Ls, tree_off, kt, vt, accept_len, nodes)
    for b in range(2):
        packed, _ = O.gather_pages(kp2, table[b:b + 1], [L2[b]])
        path = [tree_off[b] + n for n in nodes[b, :accept_len[b] + 1]]
        np.testing.assert_array_equal(packed, np.concatenate([kc[kv_off[b]:kv_off[b + 1]],
                                                              kt[path]]))
        last = path[-1]
        keys, vals = packed, O.gather_pages(vp2, table[b:b + 1], [L2[b]])[0]
        for h in range(Hq):
            s = keys[:, h // (Hq // Hkv)] @ q[last, h] / np.sqrt(D)
            w = np.exp(s - s.max())
            np.testing.assert_allclose(w @ vals[:, h // (Hq // Hkv)] / w.sum(), before[last, h],
                                       rtol=1e-12, atol=1e-13)
    # pages not named by the table are untouched
    used = set(table.reshape(-1).tolist())
    for page in range(n_pages):
        if page not in used:
            np.testing.assert_array_equal(kp2[page], kp[page])
