"""GPU parity of the EAGLE-1 static draft tree (eagle_draft_static) against
the oracle: tokens, parents, depths, scores and draft rows bit-exact on
identical log-prob rows, for full K-ary templates, a sparse template, rows
full of ties, and the device-side error reports."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _run(E, lp, parent, rank, row, root, max_rank=None):
    import torch
    B, R, V = lp.shape
    N = len(parent)
    i32 = torch.int32
    dev = lambda a, t=i32: torch.tensor(np.asarray(a), dtype=t, device="cuda")
    outs = dict(tree_off=torch.full((B + 1,), -9, dtype=i32, device="cuda"),
                parent=torch.full((B * N,), -9, dtype=i32, device="cuda"),
                tokens=torch.full((B * N,), -9, dtype=i32, device="cuda"),
                depth=torch.full((B * N,), -9, dtype=i32, device="cuda"),
                score=torch.full((B * N,), 9.0, dtype=torch.float32, device="cuda"),
                p_row_of_node=torch.full((B * N,), -9, dtype=i32, device="cuda"))
    st = torch.zeros(1, dtype=i32, device="cuda")
    mr = max_rank if max_rank is not None else int(max(rank[1:] or [0])) + 1
    E.eagle_draft_static(dev(parent), dev(rank), dev(row), dev(lp, torch.float32), dev(root),
                         outs["tree_off"], outs["parent"], outs["tokens"], outs["depth"],
                         outs["score"], outs["p_row_of_node"], st, max_rank=mr)
    torch.cuda.synchronize()
    return {k: to_np(v) for k, v in outs.items()}, int(st.item())


def _check(got, ref):
    for k in ("tree_off", "parent", "tokens", "depth", "score", "p_row_of_node"):
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)


@pytest.mark.parametrize("K,m,V,B,ties", [
    (3, 2, 7, 2, True),          # the pages' K = 3, m = 2 example, tied rows
    (4, 3, 32000, 1, False),     # Vicuna-7B vocabulary, 85 nodes
    (8, 2, 128256, 3, False),    # LLaMA-3 vocabulary, top-8, three sequences
    (2, 7, 1000, 2, True),       # deep binary template (255 nodes)
    (32, 1, 40, 1, True),        # the widest rank set, V barely above it
])
def test_full_template_matches_oracle(K, m, V, B, ties):
    E = cuda_ready()
    parent, rank, row = O.static_template_full(K, m)
    R = max(row) + 1
    if ties:
        g = np.random.default_rng(K + m)
        lp = (np.round(g.standard_normal((B, R, V)) * 2) / 2 - 6).astype(np.float32)
    else:
        lp = synth.draft_rows(K * 7 + m, "static-gpu", B * R, V, 3.0)[0].reshape(B, R, V)
    root = list(range(5, 5 + B))
    got, st = _run(E, lp, parent, rank, row, root)
    assert st == 0
    _check(got, O.build_static_tree(lp, B, parent, rank, row, root))


def test_sparse_template_matches_oracle():
    # a hand-made sparse tree: the root's ranks 0..2, then only the first
    # child grows a chain of its top tokens, the second child one rank-3 child
    E = cuda_ready()
    parent = [-1, 0, 0, 0, 1, 4, 5, 2]
    rank = [0, 0, 1, 2, 0, 0, 0, 3]
    row = [0, 1, 2, -1, 3, 4, -1, -1]
    V = 5000
    lp = synth.draft_rows(77, "static-sparse", 2 * 5, V, 3.0)[0].reshape(2, 5, V)
    got, st = _run(E, lp, parent, rank, row, [1, 2])
    assert st == 0
    _check(got, O.build_static_tree(lp, 2, parent, rank, row, [1, 2]))


def test_device_errors():
    E = cuda_ready()
    parent, rank, row = O.static_template_full(2, 2)
    lp = synth.draft_rows(3, "static-err", 3, 64, 3.0)[0].reshape(1, 3, 64)
    # a rank at or past max_rank
    _, st = _run(E, lp, parent, rank, row, [0], max_rank=1)
    assert st == 1                                   # EAGLE_ERR_INVALID_ARG
    # a parent that does not precede its child
    bad = list(parent)
    bad[3] = 5
    _, st = _run(E, lp, bad, rank, row, [0])
    assert st == 2                                   # EAGLE_ERR_INVALID_TREE
    # a non-finite log-prob in a row that is read
    lp2 = lp.copy()
    lp2[0, 1, 17] = np.inf
    _, st = _run(E, lp2, parent, rank, row, [0])
    assert st == 4                                   # EAGLE_ERR_NUMERIC
