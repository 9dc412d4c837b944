"""Pins of the oracle's greedy tree walk (CPU only).

[S4000] greedy-decoding paragraph and its figure: the drafted candidates are
matched against the target's most probable token from the first one on, and
the sequence is cut at the first mismatch (4 candidates, the first 3 kept).
[EAGLE] speculative-sampling paragraph: alpha accepted drafts give alpha + 1
tokens from one verify pass.
"""
import os

import numpy as np

import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_kv(path):
    vals = {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rest = line.split("=", 1)
            vals[key.strip()] = [int(x) for x in rest.split()]
    return vals


def test_four_candidates_three_accepted_example():
    # chain tree: root then 4 drafted candidates; the target agrees with the
    # first three and disagrees at the fourth
    g = _read_kv(os.path.join(GOLDEN, "greedy_chain_4_draft_3_accept.txt"))
    parent, tokens, argmax = g["parent"], g["tokens"], g["argmax"]
    n = len(parent)
    acc, nodes, out = O.accept_greedy([0, n], parent, tokens, argmax, max_depth=n - 1)
    assert acc[0] == g["alpha"][0] == 3
    assert list(out[0, :acc[0] + 1]) == g["out_tokens"]
    assert list(nodes[0, :acc[0] + 1]) == [0, 1, 2, 3]


def _textbook_chain(drafts, target_next):
    """Plain speculative greedy check on a linear draft: target_next[j] is
    the target's argmax after j accepted drafts."""
    out = []
    for j, d in enumerate(drafts):
        if d != target_next[j]:
            break
        out.append(d)
    out.append(target_next[len(out)])
    return out


def test_chain_tree_matches_the_textbook_rule():
    g = np.random.default_rng(0)
    for trial in range(300):
        n = int(g.integers(1, 9))
        V = int(g.integers(2, 5))
        tokens = g.integers(0, V, size=n)
        argmax = g.integers(0, V, size=n)
        parent = np.arange(-1, n - 1)
        acc, nodes, out = O.accept_greedy([0, n], parent, tokens, argmax, n - 1)
        ref = _textbook_chain(list(tokens[1:]), list(argmax))
        assert list(out[0, :acc[0] + 1]) == ref
        assert acc[0] + 1 == len(ref)
        assert np.all(out[0, acc[0] + 1:] == -1)


def test_alpha_plus_one_tokens_and_valid_path_on_random_trees():
    g = np.random.default_rng(1)
    for trial in range(200):
        par, tok = synth.random_level_tree(trial, (1, 3, 4, 4, 2), 3)
        n = len(par)
        argmax = g.integers(0, 3, size=n)
        acc, nodes, out = O.accept_greedy([0, n], par, tok, argmax, 4)
        a = acc[0]
        assert np.count_nonzero(out[0] >= 0) == a + 1
        path = list(nodes[0, :a + 1])
        assert path[0] == 0
        for d in range(1, a + 1):
            assert par[path[d]] == path[d - 1]
            assert tok[path[d]] == argmax[path[d - 1]] == out[0, d - 1]
        # the walk stopped: no child of the last node carries its argmax
        last = path[-1]
        assert all(tok[c] != argmax[last] for c in O.tree_children(par, last))
        assert out[0, a] == argmax[last]


class _ToyTarget:
    """A one-layer toy target: token embeddings give q/k/v, attention over
    [cache | sequence], logits = W_lm @ concat(heads).  Used to compare the
    tree walk with serial argmax decoding."""

    def __init__(self, seed, V=11, Hq=2, Hkv=1, D=6, L=4):
        g = np.random.default_rng(seed)
        self.V, self.Hq, self.Hkv, self.D = V, Hq, Hkv, D
        self.Eq = g.standard_normal((V, Hq, D))
        self.Ek = g.standard_normal((V, Hkv, D))
        self.Ev = g.standard_normal((V, Hkv, D))
        self.W = g.standard_normal((V, Hq * D))
        self.kc = g.standard_normal((L, Hkv, D))
        self.vc = g.standard_normal((L, Hkv, D))
        self.L = L

    def serial(self, root, steps):
        seq = [root]
        for _ in range(steps):
            toks = np.array(seq)
            o = O.causal_attn(self.Eq[toks], np.concatenate([self.kc, self.Ek[toks]]),
                              np.concatenate([self.vc, self.Ev[toks]]), self.L)
            logits = self.W @ o[-1].reshape(-1)
            seq.append(int(np.argmax(logits)))
        return seq[1:]

    def tree_argmax(self, tokens, parent):
        tokens = np.asarray(tokens)
        n = len(tokens)
        o = O.tree_attn(self.Eq[tokens], self.Ek[tokens], self.Ev[tokens],
                        self.kc, self.vc, [0, self.L], [0, n], parent)
        return O.lmhead_softmax(o.reshape(n, -1), self.W, 1.0, want_q=False)["argmax"]


def test_tree_walk_equals_serial_argmax_decoding():
    hits = 0
    for seed in range(40):
        m = _ToyTarget(seed)
        g = np.random.default_rng(100 + seed)
        root = int(g.integers(0, m.V))
        depth = 4
        serial = m.serial(root, depth + 1)
        par, tok = synth.random_level_tree(seed, (1, 3, 3, 3, 2), m.V)
        tok = tok.copy()
        tok[0] = root
        planted = set()
        if seed % 2 == 0:
            # plant the serial continuation along one random root-to-leaf path
            leaf = int(g.integers(len(par) - 2, len(par)))
            path = O.tree_path(par, leaf)
            for d, node in enumerate(path[1:]):
                tok[node] = serial[d]
                planted.add(node)
        # sibling tokens distinct (as in an EAGLE-2 tree): re-label the
        # non-planted duplicates
        for i in range(len(par)):
            kids = O.tree_children(par, i)
            for c in kids:
                if c in planted:
                    continue
                used = {int(tok[j]) for j in kids if j != c}
                if int(tok[c]) in used:
                    tok[c] = min(set(range(m.V)) - used)
        argmax = m.tree_argmax(tok, par)
        acc, nodes, out = O.accept_greedy([0, len(par)], par, tok, argmax, depth)
        a = int(acc[0])
        # the emitted tokens are the serial decode's first alpha+1 tokens
        assert list(out[0, :a + 1]) == serial[:a + 1]
        # alpha is the longest prefix of the serial decode present as a path
        best = 0
        for i in range(len(par)):
            p = O.tree_path(par, i)[1:]
            if [int(tok[j]) for j in p] == serial[:len(p)]:
                best = max(best, len(p))
        assert a == best
        if seed % 2 == 0:
            assert a == len(O.tree_path(par, leaf)) - 1
            hits += 1
    assert hits == 20


def test_duplicate_sibling_tokens_take_the_lowest_index():
    par = [-1, 0, 0, 1, 2]
    tok = [9, 5, 5, 7, 7]
    argmax = [5, 7, 7, 1, 1]
    acc, nodes, out = O.accept_greedy([0, 5], par, tok, argmax, 2)
    assert list(nodes[0, :3]) == [0, 1, 3]
    assert list(out[0, :3]) == [5, 7, 1]


def test_batched_sequences_are_independent():
    par = [-1, 0, 0, -1, 0, 1]
    tok = [0, 1, 2, 0, 2, 1]
    argmax = [2, 0, 0, 2, 1, 3]
    acc, nodes, out = O.accept_greedy([0, 3, 6], par, tok, argmax, 2)
    assert list(acc) == [1, 2]
    assert list(out[0, :2]) == [2, 0] and list(out[1, :3]) == [2, 1, 3]
