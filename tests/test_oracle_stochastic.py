"""Pins of the oracle's multi-round stochastic acceptance (CPU only).

[S4000] random-decoding paragraph: accept a draft with min(1, q/p), else
resample from the corrected distribution, which keeps the target
distribution.  [EAGLE] "多轮投机采样": the rule is applied recursively over a
tree.  [EAGLE-2] §2 basic principle: the output distribution equals the
target's.  The pins below check that property exactly (by enumerating every
uniform on the 2^-24 grid through bisection over the oracle itself) and by
Monte-Carlo chi-square, plus closed forms.
"""
import itertools

import numpy as np
import pytest

import oracle as O

GRID = 1 << 24
U_MAX = np.float32((GRID - 1) / GRID)


def _one_level(q_root, p, toks, u_acc, u_samp, mode):
    k = len(toks)
    parent = np.array([-1] + [0] * k, dtype=np.int32)
    tokens = np.array([0] + list(toks), dtype=np.int32)
    V = len(q_root)
    q = np.tile(np.asarray(q_root, np.float32), (k + 1, 1))
    prow = np.zeros(k + 1, dtype=np.int32)
    ua = np.array([0.0] + list(u_acc), dtype=np.float32)
    us = np.array([u_samp] * (k + 1), dtype=np.float32)
    acc, nodes, out = O.accept_stochastic([0, k + 1], parent, tokens, q,
                                          np.asarray(p, np.float32)[None, :],
                                          prow, ua, us, max_depth=1, mode=mode)
    return int(acc[0]), int(nodes[0, 1]), int(out[0, 0])


def _count_true_prefix(pred):
    """Number of U in [0, 2^24) with pred(U) true, for pred true on a prefix."""
    lo, hi = 0, GRID           # pred(lo-1) true (or lo == 0), pred(hi) false
    while lo < hi:
        mid = (lo + hi) // 2
        if pred(mid):
            lo = mid + 1
        else:
            hi = mid
    return lo


def _exact_first_token_distribution(q_root, p, toks, mode):
    """Exact law of the first emitted token for fixed child tokens, over
    independent uniforms on the 2^-24 grid."""
    V, k = len(q_root), len(toks)
    dist = np.zeros(V)
    u = [U_MAX] * k                      # children before j: forced rejects
    reach = 1.0
    for j in range(k):
        def accepts(U, j=j):
            uu = list(u)
            uu[j] = np.float32(U / GRID)
            acc, node, _ = _one_level(q_root, p, toks, uu, 0.0, mode)
            return acc == 1 and node == j + 1
        A = _count_true_prefix(accepts)
        dist[toks[j]] += reach * A / GRID
        reach *= (GRID - A) / GRID
        if A == GRID:
            return dist
    # every child rejected: inverse-CDF sample over u_sample
    lo_of = []
    for x in range(V + 1):
        if x == 0:
            lo_of.append(0)
            continue
        def below(U, x=x):
            _, _, tok = _one_level(q_root, p, toks, u, np.float32(U / GRID), mode)
            return tok < x
        lo_of.append(_count_true_prefix(below))
    lo_of[V] = GRID
    for x in range(V):
        dist[x] += reach * (lo_of[x + 1] - lo_of[x]) / GRID
    return dist


def _draws(p, k, mode):
    V = len(p)
    if mode == O.MODE_REPLACE:
        for toks in itertools.product(range(V), repeat=k):
            yield toks, float(np.prod([p[t] for t in toks]))
    else:
        for toks in itertools.permutations(range(V), k):
            pr, left = 1.0, 1.0
            for t in toks:
                pr *= p[t] / left
                left -= p[t]
            yield toks, pr


@pytest.mark.parametrize("mode,V,k,seed", [
    (O.MODE_NO_REPLACE, 4, 1, 0),
    (O.MODE_NO_REPLACE, 5, 2, 1),
    (O.MODE_NO_REPLACE, 4, 3, 2),
    (O.MODE_REPLACE, 4, 2, 3),
    (O.MODE_REPLACE, 3, 3, 4),
])
def test_exact_enumeration_reproduces_the_target_distribution(mode, V, k, seed):
    g = np.random.default_rng(seed)
    q = g.dirichlet(np.ones(V)).astype(np.float32)
    p = g.dirichlet(np.ones(V) * 0.7).astype(np.float32)
    p64 = p.astype(np.float64)
    p64 /= p64.sum()
    total = np.zeros(V)
    mass = 0.0
    for toks, pr in _draws(p64, k, mode):
        total += pr * _exact_first_token_distribution(q, p, list(toks), mode)
        mass += pr
    assert abs(mass - 1) < 1e-12
    np.testing.assert_allclose(total, q.astype(np.float64), rtol=0, atol=2e-6)


def test_single_child_accept_probability_is_sum_of_min():
    g = np.random.default_rng(7)
    V = 6
    q = g.dirichlet(np.ones(V)).astype(np.float32)
    p = g.dirichlet(np.ones(V)).astype(np.float32)
    acc_prob = 0.0
    for t in range(V):
        def accepts(U, t=t):
            a, _, _ = _one_level(q, p, [t], [np.float32(U / GRID)], 0.0,
                                 O.MODE_NO_REPLACE)
            return a == 1
        acc_prob += float(p[t]) * _count_true_prefix(accepts) / GRID
    ref = float(np.minimum(p.astype(np.float64), q.astype(np.float64)).sum())
    assert abs(acc_prob - ref) < 2e-7


def test_identical_draft_and_target_accepts_every_first_child():
    g = np.random.default_rng(8)
    parent = [-1, 0, 0, 1, 1, 3, 2]
    n = len(parent)
    V = 9
    rows = g.dirichlet(np.ones(V), size=n).astype(np.float32)
    tokens = g.integers(0, V, size=n).astype(np.int32)
    rows[:, :] = np.maximum(rows, 1e-3)
    rows /= rows.sum(axis=1, keepdims=True)
    # node i's children are drafted from row i; the target's row i is equal
    prow = np.array([-1] + parent[1:], dtype=np.int32)
    ua = g.integers(0, GRID, size=n).astype(np.float64) / GRID
    us = g.integers(0, GRID, size=n).astype(np.float64) / GRID
    acc, nodes, out = O.accept_stochastic([0, n], parent, tokens, rows, rows, prow,
                                          ua.astype(np.float32), us.astype(np.float32), 3)
    assert list(nodes[0, :acc[0] + 1]) == [0, 1, 3, 5]


def test_acceptance_boundary_is_exact():
    # u*p == q exactly must reject; one grid step lower must accept
    q = np.array([0.25, 0.75], np.float32)
    p = np.array([0.5, 0.5], np.float32)
    a, _, _ = _one_level(q, p, [0], [np.float32(0.5)], 0.0, O.MODE_NO_REPLACE)
    assert a == 0
    a, _, _ = _one_level(q, p, [0], [np.float32(0.5 - 2 ** -24)], 0.0, O.MODE_NO_REPLACE)
    assert a == 1


def test_rejection_resamples_from_the_residual():
    # q = [.5,.5], p = [1,0], child token 0: accept iff u < 1/2, and the
    # residual max(0, q - p) = [0, .5] puts all mass on token 1
    q = np.array([0.5, 0.5], np.float32)
    p = np.array([1.0, 0.0], np.float32)
    for U in (0, GRID // 2 - 1):
        a, _, tok = _one_level(q, p, [0], [np.float32(U / GRID)], 0.3, O.MODE_NO_REPLACE)
        assert (a, tok) == (1, 0)
    for U in (GRID // 2, GRID - 1):
        for us in (0.0, 0.5, float(U_MAX)):
            a, _, tok = _one_level(q, p, [0], [np.float32(U / GRID)], us,
                                   O.MODE_NO_REPLACE)
            assert (a, tok) == (0, 1)


def test_inverse_cdf_sampler_boundaries():
    # q = [1/4, 1/2, 1/4]: W = [2^38, 2^39, 2^38], Z = 2^40, target = U * 2^16
    q = np.array([0.25, 0.5, 0.25], np.float32)
    p = np.array([1.0, 0.0, 0.0], np.float32)
    cases = [(0, 0), ((1 << 22) - 1, 0), (1 << 22, 1), (3 << 22, 2), (GRID - 1, 2),
             ((3 << 22) - 1, 1)]
    for U, want in cases:
        # the root is a leaf, so the walk samples the bonus token from q[0]
        acc, nodes, out = O.accept_stochastic([0, 1], [-1], [0], q[None, :], p[None, :],
                                              [-1], [0.0], [np.float32(U / GRID)], 0)
        assert acc[0] == 0 and out[0, 0] == want


def test_no_replace_zeroes_the_rejected_token():
    # q puts no mass on token 0; p = [.5,.25,.25]. After rejecting child
    # token 0 the next draft distribution is [0, .5, .5]; a second child with
    # token 0 now has p = 0 and q_1(0) = 0, so it must be rejected for any u.
    q = np.array([0.0, 0.5, 0.5], np.float32)
    p = np.array([0.5, 0.25, 0.25], np.float32)
    trace = []
    parent = [-1, 0, 0]
    O.accept_stochastic([0, 3], parent, [0, 0, 0], np.tile(q, (3, 1)), p[None, :],
                        [-1, 0, 0], np.float32([0, 0, 0]), np.float32([0.1] * 3), 1,
                        mode=O.MODE_NO_REPLACE, trace=trace)
    trace = [t for t in trace if t[2] != "sample"]
    assert [t[6] for t in trace] == [False, False]
    assert trace[1][5] == 0.0         # p_1(0)
    trace = []
    O.accept_stochastic([0, 3], parent, [0, 0, 1], np.tile(q, (3, 1)), p[None, :],
                        [-1, 0, 0], np.float32([0, 0.99, 0.99]), np.float32([0.1] * 3), 1,
                        mode=O.MODE_NO_REPLACE, trace=trace)
    trace = [t for t in trace if t[2] != "sample"]
    # second child token 1: p_1(1) = .5, q_1(1) = .5 -> u = .99 accepts
    assert trace[1][4:7] == (0.5, 0.5, True)


def test_f32_of_int_rounds_to_nearest_even():
    assert O.f32_of_int(2 ** 24 + 1) == np.float32(2 ** 24)
    assert O.f32_of_int(2 ** 24 + 3) == np.float32(2 ** 24 + 4)
    assert O.f32_of_int(2 ** 24 + 2) == np.float32(2 ** 24 + 2)
    g = np.random.default_rng(0)
    for _ in range(2000):
        n = int(g.integers(0, 2 ** 62)) >> int(g.integers(0, 60))
        ref = np.float32(np.float64(n)) if n < 2 ** 53 else None
        if ref is not None:
            assert O.f32_of_int(n) == ref


def _mc_first_tokens(mode, V, k, n_trials, seed, depth2=False):
    g = np.random.default_rng(seed)
    q_root = g.dirichlet(np.ones(V)).astype(np.float32)
    p_root = g.dirichlet(np.ones(V)).astype(np.float32)
    q_tok = g.dirichlet(np.ones(V), size=V).astype(np.float32)   # target after token x
    p_tok = g.dirichlet(np.ones(V), size=V).astype(np.float32)   # draft after token x
    firsts, seconds = [], []
    for _ in range(n_trials):
        def draw(p, m):
            p64 = p.astype(np.float64)
            p64 /= p64.sum()
            return list(g.choice(V, size=m, replace=(mode == O.MODE_REPLACE), p=p64))
        kids = draw(p_root, k)
        parent, tokens, qrows, prow = [-1], [0], [q_root], [-1]
        for t in kids:
            parent.append(0); tokens.append(t); qrows.append(q_tok[t]); prow.append(0)
        rows = [p_root]
        if depth2:
            for ci, t in enumerate(kids):
                rows.append(p_tok[t])
                for t2 in draw(p_tok[t], 2):
                    parent.append(ci + 1); tokens.append(t2)
                    qrows.append(q_root); prow.append(len(rows) - 1)
        n = len(parent)
        ua = (g.integers(0, GRID, size=n) / GRID).astype(np.float32)
        us = (g.integers(0, GRID, size=n) / GRID).astype(np.float32)
        acc, nodes, out = O.accept_stochastic([0, n], parent, tokens, np.array(qrows),
                                              np.array(rows), prow, ua, us, 2, mode=mode)
        firsts.append(out[0, 0])
        if acc[0] >= 1:
            seconds.append((out[0, 0], out[0, 1]))
    return q_root, q_tok, np.array(firsts), seconds


@pytest.mark.parametrize("mode", [O.MODE_NO_REPLACE, O.MODE_REPLACE])
def test_monte_carlo_chi_square_on_a_tiny_vocabulary(mode):
    from scipy.stats import chisquare
    V, k, n = 8, 3, 40000
    q_root, q_tok, firsts, seconds = _mc_first_tokens(mode, V, k, n, 11 + mode, depth2=True)
    obs = np.bincount(firsts, minlength=V)
    qr = q_root.astype(np.float64)
    exp = qr / qr.sum() * n
    assert chisquare(obs, exp).pvalue > 1e-3
    # second token given an accepted first token x: follows the target row of x
    xs = np.array([s[0] for s in seconds])
    x = int(np.bincount(xs, minlength=V).argmax())
    sec = np.array([s[1] for s in seconds if s[0] == x])
    obs2 = np.bincount(sec, minlength=V)
    qx = q_tok[x].astype(np.float64)
    exp2 = qx / qx.sum() * len(sec)
    assert len(sec) > 2000
    assert chisquare(obs2, exp2).pvalue > 1e-3
