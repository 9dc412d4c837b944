"""GPU parity of the acceptance walks against the oracle (bit-exact).

Both sides get identical trees, argmax rows, probability rows and uniforms;
accept lengths, accepted node ids and emitted tokens must be equal."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _dev(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _forest(seed, B, V, levels_choices, distinct=False):
    g = np.random.default_rng(seed)
    parents, toks = [], []
    for b in range(B):
        levels = levels_choices[int(g.integers(0, len(levels_choices)))]
        par, tok = synth.random_level_tree(seed * 1000 + b, levels, V)
        tok = tok.copy()
        if distinct:
            for i in range(len(par)):
                kids = O.tree_children(par, i)
                used = set()
                for c in kids:
                    while int(tok[c]) in used:
                        tok[c] = (int(tok[c]) + 1) % V
                    used.add(int(tok[c]))
        parents.append(par)
        toks.append(tok)
    sizes = [len(p) for p in parents]
    tree_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    return tree_off, np.concatenate(parents).astype(np.int32), np.concatenate(toks).astype(np.int32)


def _run_greedy(E, tree_off, parent, tokens, argmax, max_depth):
    import torch
    B = len(tree_off) - 1
    W = max_depth + 1
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_nodes = int(np.max(np.diff(tree_off)))
    E.eagle_accept_greedy(_dev(tree_off), _dev(parent), _dev(tokens), _dev(argmax), acc, nodes,
                          out, st, max_nodes=max_nodes, max_depth=max_depth)
    torch.cuda.synchronize()
    return to_np(acc), to_np(nodes), to_np(out), int(st.item())


@pytest.mark.parametrize("seed,B,V", [(0, 1, 3), (1, 7, 2), (2, 37, 5), (3, 16, 4)])
def test_greedy_walk_matches_oracle(seed, B, V):
    E = cuda_ready()
    levels = [(1,), (1, 1), (1, 4, 6, 6, 6, 3), (1, 3, 9, 20, 40, 60, 80, 30, 7),
              (1,) * 12, (1, 10, 10, 10)]
    tree_off, parent, tokens = _forest(seed, B, V, levels)
    g = np.random.default_rng(seed)
    argmax = g.integers(0, V, size=len(parent)).astype(np.int32)
    # plant matches along random paths so deep walks happen
    for b in range(B):
        t0, t1 = tree_off[b], tree_off[b + 1]
        leaf = int(g.integers(0, t1 - t0))
        path = O.tree_path(parent[t0:t1], leaf)
        for a, c in zip(path[:-1], path[1:]):
            argmax[t0 + a] = tokens[t0 + c]
    depth = max(max(O.tree_depths(parent[tree_off[b]:tree_off[b + 1]])) for b in range(B))
    ref = O.accept_greedy(tree_off, parent, tokens, argmax, depth)
    got = _run_greedy(E, tree_off, parent, tokens, argmax, depth)
    assert got[3] == 0
    for r, x in zip(ref, got[:3]):
        np.testing.assert_array_equal(x, r)
    assert got[0].max() >= 1


def test_greedy_node_limit_and_chain():
    E = cuda_ready()
    n = 256                                   # EAGLE_MAX_TREE_NODES
    parent = np.arange(-1, n - 1, dtype=np.int32)
    tokens = np.arange(n, dtype=np.int32) % 7
    argmax = np.roll(tokens, -1).astype(np.int32)
    argmax[200] = 99                          # mismatch after 200 accepts
    tree_off = np.array([0, n], np.int32)
    ref = O.accept_greedy(tree_off, parent, tokens, argmax, n - 1)
    got = _run_greedy(E, tree_off, parent, tokens, argmax, n - 1)
    assert got[3] == 0 and got[0][0] == 200
    for r, x in zip(ref, got[:3]):
        np.testing.assert_array_equal(x, r)


def _run_stoch(E, tree_off, parent, tokens, q, p_rows, prow, ua, us, max_depth, mode):
    import torch
    B = len(tree_off) - 1
    W = max_depth + 1
    acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    nodes = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    out = torch.full((B, W), -7, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    max_nodes = int(np.max(np.diff(tree_off)))
    E.eagle_accept_stochastic(_dev(tree_off), _dev(parent), _dev(tokens), _dev(q), _dev(p_rows),
                              _dev(prow), _dev(ua), _dev(us), acc, nodes, out, st,
                              max_nodes=max_nodes, max_depth=max_depth, mode=mode)
    torch.cuda.synchronize()
    return to_np(acc), to_np(nodes), to_np(out), int(st.item())


def _stoch_case(seed, B, V, levels, plant_frac=0.5):
    tree_off, parent, tokens = _forest(seed, B, V, levels, distinct=True)
    T = len(parent)
    g = np.random.default_rng(seed + 99)
    # node i's children are drafted from row i
    p_rows = synth.random_probs(seed, "p", T, V, sigma=2.0)
    prow = np.full(T, -1, np.int32)
    for b in range(B):
        t0, t1 = tree_off[b], tree_off[b + 1]
        for i in range(1, t1 - t0):
            prow[t0 + i] = t0 + parent[t0 + i]
    q = synth.random_probs(seed, "q", T, V, sigma=2.0)
    # make some entries exactly zero on both sides
    zero = g.random((T, V)) < 0.02
    q[zero] = 0
    p_rows[np.roll(zero, 1, axis=1)] = 0
    # plant: for some nodes the target row equals the draft row (accepts)
    for t in range(T):
        if g.random() < plant_frac:
            q[t] = p_rows[t]
    ua = synth.uniforms24(seed, "ua", T)
    us = synth.uniforms24(seed, "us", T)
    return tree_off, parent, tokens, q, p_rows, prow, ua, us


@pytest.mark.parametrize("mode", [O.MODE_NO_REPLACE, O.MODE_REPLACE])
@pytest.mark.parametrize("seed,B,V", [(0, 1, 7), (1, 3, 1023), (2, 5, 1024), (3, 2, 32000),
                                      (4, 1, 128256), (5, 16, 4099)])
def test_stochastic_walk_matches_oracle(mode, seed, B, V):
    E = cuda_ready()
    levels = [(1,), (1, 4, 6, 6, 6, 3), (1, 8, 8, 8, 8), (1, 2, 3, 4, 5, 6, 7)]
    case = _stoch_case(seed, B, V, levels)
    tree_off, parent = case[0], case[1]
    depth = max(max(O.tree_depths(parent[tree_off[b]:tree_off[b + 1]])) for b in range(B))
    ref = O.accept_stochastic(*case, max_depth=depth, mode=mode)
    got = _run_stoch(E, *case, depth, mode)
    assert got[3] == 0
    for r, x in zip(ref, got[:3]):
        np.testing.assert_array_equal(x, r)


@pytest.mark.parametrize("B", [4, 12, 16])
def test_stochastic_many_rejections_then_sample_at_full_vocab(B):
    # random target vs random draft: almost every child is rejected, so every
    # sequence runs up to k residual rounds and then the inverse-CDF sampler.
    # The walk's launch shape follows B: 4 sequences fit at once as 16 CTAs
    # of 1024 threads; 12 do not, and run as 16 CTAs of 512 threads, two per
    # SM; 16 do not fit either way and run in smaller clusters of 512-thread
    # CTAs (13 of them, 20 entries per thread, when all 16 clusters fit).
    E = cuda_ready()
    V = 128256
    case = _stoch_case(11, B, V, [(1, 8, 8)], plant_frac=0.0)
    for mode in (O.MODE_NO_REPLACE, O.MODE_REPLACE):
        ref = O.accept_stochastic(*case, max_depth=2, mode=mode)
        got = _run_stoch(E, *case, 2, mode)
        assert got[3] == 0
        for r, x in zip(ref, got[:3]):
            np.testing.assert_array_equal(x, r)


def _lmhead(E, h, w, temperature, logits):
    import torch
    T, V = h.shape[0], w.shape[0]
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    rm, lse, gap = (torch.empty(T, dtype=torch.float32, device="cuda") for _ in range(3))
    out = torch.full((T, V), -7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(E.eagle_lmhead_workspace_bytes(T, V), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.eagle_lmhead_softmax(h, w, am, rm, lse, gap, out, ws, st, temperature=temperature,
                           logits=logits)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, lse


@pytest.mark.parametrize("dtype,V,H,temp", [("f32", 1024, 256, 0.7), ("bf16", 32000, 256, 1.0),
                                            ("bf16", 4099, 512, 0.7), ("bf16", 128256, 128, 1.0)])
def test_walk_on_logits_equals_walk_on_probabilities(dtype, V, H, temp):
    # The logits walk normalises each visited row itself; fed the LM head's
    # logits and row log-sum-exp it must take exactly the decisions of the
    # walk fed the LM head's probability-mode q, and both the oracle's.
    import torch
    E = cuda_ready()
    B = 3
    tree_off, parent, tokens = _forest(V + H, B, V, [(1, 4, 6, 6, 3), (1, 8, 8, 8)],
                                       distinct=True)
    T = len(parent)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    h = torch.from_numpy(synth.normal(V, "h", (T, H))).to(tdt).cuda()
    w = torch.from_numpy(synth.normal(V, "w", (V, H), std=0.5 / np.sqrt(H) * 8)).to(tdt).cuda()
    q, _ = _lmhead(E, h, w, temp, logits=False)
    z, lse = _lmhead(E, h, w, temp, logits=True)
    qn = to_np(q)
    g = np.random.default_rng(V)
    # draft rows: node i's children drafted from row i; some rows equal the
    # target's (accepts), the rest random (rejections, residual rounds)
    p_rows = synth.random_probs(V, "p", T, V, sigma=2.0)
    for t in range(T):
        if g.random() < 0.6:
            p_rows[t] = qn[t]
    prow = np.full(T, -1, np.int32)
    for b in range(B):
        t0, t1 = tree_off[b], tree_off[b + 1]
        for i in range(1, t1 - t0):
            prow[t0 + i] = t0 + parent[t0 + i]
    ua = synth.uniforms24(V, "ua", T)
    us = synth.uniforms24(V, "us", T)
    depth = max(max(O.tree_depths(parent[tree_off[b]:tree_off[b + 1]])) for b in range(B))
    for mode in (O.MODE_NO_REPLACE, O.MODE_REPLACE):
        ref = O.accept_stochastic(tree_off, parent, tokens, qn, p_rows, prow, ua, us,
                                  max_depth=depth, mode=mode)
        got_q = _run_stoch(E, tree_off, parent, tokens, qn, p_rows, prow, ua, us, depth, mode)
        Wd = depth + 1
        acc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
        nodes = torch.full((B, Wd), -7, dtype=torch.int32, device="cuda")
        out = torch.full((B, Wd), -7, dtype=torch.int32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        E.eagle_accept_stochastic_logits(_dev(tree_off), _dev(parent), _dev(tokens), z, lse,
                                         _dev(p_rows), _dev(prow), _dev(ua), _dev(us), acc,
                                         nodes, out, st, temperature=temp,
                                         max_nodes=int(np.max(np.diff(tree_off))),
                                         max_depth=depth, mode=mode)
        torch.cuda.synchronize()
        assert got_q[3] == 0 and int(st.item()) == 0
        got_z = (to_np(acc), to_np(nodes), to_np(out))
        for r, a, b_ in zip(ref, got_q[:3], got_z):
            np.testing.assert_array_equal(a, r)
            np.testing.assert_array_equal(b_, r)
        assert ref[0].max() >= 1
