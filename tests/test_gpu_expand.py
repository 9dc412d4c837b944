"""GPU parity of the EAGLE-2 expand + rerank against the oracle (bit-exact):
identical draft log-prob rows must give identical trees (parent, tokens,
depth, scores, draft-row ids)."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _gpu_tree(E, lp, B, V, k, depth, budget, root_token, fused=False, all_levels=False):
    import torch
    R = 1 + (depth - 1) * k
    pool = torch.zeros(E.eagle_draft_pool_bytes(B, k, depth, V), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    d_lp = torch.from_numpy(lp.reshape(B, R, V)).cuda()
    n_pool = k + (depth - 1) * k * k
    T = sum(min(b, n_pool) + 1 for b in budget)
    out = {n: torch.full((T,), -7, dtype=torch.int32, device="cuda")
           for n in ("parent", "tokens", "node_depth", "p_row_of_node")}
    out["score"] = torch.full((T,), -7.0, dtype=torch.float32, device="cuda")
    out["tree_off"] = torch.full((B + 1,), -7, dtype=torch.int32, device="cuda")
    fin = dict(budget=torch.tensor(budget, dtype=torch.int32, device="cuda"),
               root_token=torch.tensor(root_token, dtype=torch.int32, device="cuda"), **out)
    if all_levels:
        E.eagle_draft_expand_all(pool, st, B=B, V=V, k=k, depth=depth, draft_logp=d_lp, **fin)
        torch.cuda.synchronize()
        return {n: to_np(t) for n, t in out.items()}, int(st.item())
    for lev in range(depth - 1 if fused else depth):
        E.eagle_draft_expand(pool, st, B=B, V=V, k=k, depth=depth, level=lev, draft_logp=d_lp)
    if fused:
        E.eagle_draft_expand(pool, st, B=B, V=V, k=k, depth=depth, level=depth - 1, finalize=2,
                             draft_logp=d_lp, **fin)
    else:
        E.eagle_draft_expand(pool, st, B=B, V=V, k=k, depth=depth, finalize=1, **fin)
    torch.cuda.synchronize()
    return {n: to_np(t) for n, t in out.items()}, int(st.item())


@pytest.mark.parametrize("B,V,k,depth,budgets,sigma", [
    (1, 4, 2, 2, [4], 1.0),
    (1, 1000, 4, 3, [12], 3.0),
    (3, 777, 5, 4, [1, 17, 200], 3.0),
    (1, 32000, 10, 6, [60], 3.0),             # Vicuna-7B shaped tree
    (1, 128256, 8, 7, [64], 3.0),             # LLaMA-3-8B shaped tree
    (2, 128256, 8, 8, [64, 33], 3.0),         # LLaMA-3-70B / batched shape
    (2, 5000, 32, 3, [500, 0], 0.5),          # k at its limit, an empty budget
    # levels larger than one wave of CTAs: persistent streaming through
    # shared memory, ragged last chunks
    (8, 40000, 8, 3, [20, 64, 0, 5, 64, 64, 33, 1], 3.0),
    (8, 70004, 6, 3, [30, 12, 64, 7, 1, 0, 9, 40], 3.0),
])
@pytest.mark.parametrize("mode", ["levels", "fused", "all"])
def test_expand_matches_oracle(B, V, k, depth, budgets, sigma, mode):
    # fused: the last level and the finalize in one launch; all: every level
    # in one call (all levels' chunks ranked in one launch, then the merges)
    E = cuda_ready()
    R = 1 + (depth - 1) * k
    lp, _ = synth.draft_rows(B * 7 + V, "expand", B * R, V, sigma)
    ref = O.build_eagle2_tree(lp, B=B, k=k, depth=depth, budget=budgets,
                              root_token=list(range(B)))
    got, st = _gpu_tree(E, lp, B, V, k, depth, budgets, list(range(B)), fused=(mode == "fused"),
                        all_levels=(mode == "all"))
    assert st == 0
    for name in ("tree_off", "parent", "tokens", "p_row_of_node", "score"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    np.testing.assert_array_equal(got["node_depth"], ref["depth"])


def test_expand_ties_are_broken_by_token_then_creation_order():
    # quantised log-probs produce many exact ties in values and in scores
    E = cuda_ready()
    B, V, k, depth = 2, 3000, 6, 4
    R = 1 + (depth - 1) * k
    g = np.random.default_rng(5)
    lp = (-np.round(g.random((B * R, V)) * 8) / 4).astype(np.float32)
    budgets = [40, 90]
    ref = O.build_eagle2_tree(lp, B=B, k=k, depth=depth, budget=budgets, root_token=[3, 4])
    got, st = _gpu_tree(E, lp, B, V, k, depth, budgets, [3, 4])
    assert st == 0
    for name in ("tree_off", "parent", "tokens", "p_row_of_node", "score"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)


def test_expand_reports_non_finite_log_probs():
    import torch
    E = cuda_ready()
    B, V, k, depth = 1, 2048, 4, 2
    R = 1 + (depth - 1) * k
    lp, _ = synth.draft_rows(1, "nan", B * R, V, 3.0)
    lp[0, 17] = np.nan
    _, st = _gpu_tree(E, lp, B, V, k, depth, [5], [0])
    assert st == 4                            # EAGLE_ERR_NUMERIC


@pytest.mark.parametrize("B,V,k,depth,budgets,order", [
    (1, 40000, 32, 3, [300], "random"),       # many chunk-list keys above the first bound
    (1, 32000, 10, 3, [40], "descending"),    # one chunk holds every top key
    (2, 9000, 7, 3, [30, 50], "ascending"),   # top keys at the row's ragged end
])
def test_expand_concentrated_top_keys(B, V, k, depth, budgets, order):
    # Rows whose top keys crowd into one chunk (sorted rows) or into many
    # chunk lists at once (k = 32): the selection bounds must be raised
    # several times before the exact rank count; the tree must not change.
    E = cuda_ready()
    R = 1 + (depth - 1) * k
    lp, _ = synth.draft_rows(V + k, "concentrated", B * R, V, 3.0)
    if order != "random":
        lp = np.sort(lp, axis=1)
        if order == "descending":
            lp = lp[:, ::-1].copy()
    ref = O.build_eagle2_tree(lp, B=B, k=k, depth=depth, budget=budgets,
                              root_token=list(range(B)))
    got, st = _gpu_tree(E, lp, B, V, k, depth, budgets, list(range(B)))
    assert st == 0
    for name in ("tree_off", "parent", "tokens", "p_row_of_node", "score"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
    np.testing.assert_array_equal(got["node_depth"], ref["depth"])


def test_expand_all_equal_rows():
    # every log-prob equal: the order is decided by token index alone
    E = cuda_ready()
    B, V, k, depth = 1, 20000, 12, 3
    R = 1 + (depth - 1) * k
    lp = np.full((B * R, V), -np.log(V), dtype=np.float32)
    ref = O.build_eagle2_tree(lp, B=B, k=k, depth=depth, budget=[100], root_token=[0])
    got, st = _gpu_tree(E, lp, B, V, k, depth, [100], [0])
    assert st == 0
    for name in ("tree_off", "parent", "tokens", "p_row_of_node", "score"):
        np.testing.assert_array_equal(got[name], ref[name], err_msg=name)
