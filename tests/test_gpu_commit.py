"""GPU parity of the KV commit (eagle_kv_commit_paged) against the oracle:
the accepted path's K/V rows land bit for bit at the sequence's next cache
positions, across page boundaries, and the length advances; then the paged
attention of the next step reads them."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _setup(seed, Ls, P, Hkv, D, levels, max_depth):
    import torch
    B = len(Ls)
    parents = [synth.random_level_tree(seed + b, levels, 5)[0] for b in range(B)]
    sizes = [len(p) for p in parents]
    tree_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    parent = np.concatenate(parents).astype(np.int32)
    T = int(tree_off[-1])
    kt = synth.to_bf16_values(synth.normal(seed, "ck", (T, Hkv, D)))
    vt = synth.to_bf16_values(synth.normal(seed, "cv", (T, Hkv, D)))
    cap = [(L + max_depth + 1 + P - 1) // P for L in Ls]
    n_pages = sum(cap) + 3
    perm = np.random.default_rng(seed).permutation(n_pages)
    table = np.full((B, max(cap)), -1, np.int32)
    nxt = 0
    for b in range(B):
        for j in range(cap[b]):
            table[b, j] = perm[nxt]
            nxt += 1
    kp = synth.to_bf16_values(synth.normal(seed, "ckp", (n_pages, P, Hkv, D)))
    vp = synth.to_bf16_values(synth.normal(seed, "cvp", (n_pages, P, Hkv, D)))
    # the accepted path: greedy walk with the argmax planted along a random
    # root-to-leaf path, cut at a random depth
    g = np.random.default_rng(seed + 1)
    argmax = g.integers(0, 5, T).astype(np.int32)
    tokens = g.integers(0, 5, T).astype(np.int32)
    alen, anodes, _ = O.accept_greedy(tree_off, parent, tokens, argmax, max_depth)
    return dict(tree_off=tree_off, parent=parent, kt=kt, vt=vt, kp=kp, vp=vp, table=table,
                kv_len=np.array(Ls, np.int32), alen=alen, anodes=anodes)


@pytest.mark.parametrize("Ls,P,levels", [([5, 0, 127, 300], 128, (1, 3, 3, 3, 3)),
                                         ([15, 16, 1], 16, (1, 2, 2, 2, 2, 2, 2))])
def test_commit_matches_oracle(Ls, P, levels):
    import torch
    E = cuda_ready()
    Hkv, D = 8, 128
    md = len(levels) - 1
    c = _setup(len(Ls) + P, Ls, P, Hkv, D, levels, md)
    dev = lambda a, t: torch.from_numpy(np.ascontiguousarray(a)).to(t).cuda()
    bf, i32 = torch.bfloat16, torch.int32
    kp, vp = dev(c["kp"], bf), dev(c["vp"], bf)
    kv_len = dev(c["kv_len"], i32)
    st = torch.zeros(1, dtype=i32, device="cuda")
    E.eagle_kv_commit_paged(dev(c["tree_off"], i32), dev(c["alen"], i32), dev(c["anodes"], i32),
                            dev(c["kt"], bf), dev(c["vt"], bf), kp, vp, dev(c["table"], i32),
                            kv_len, st, max_depth=md)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rk, rv, rlen = O.kv_commit_paged(c["kp"], c["vp"], c["table"], c["kv_len"], c["tree_off"],
                                     c["kt"], c["vt"], c["alen"], c["anodes"])
    np.testing.assert_array_equal(to_np(kv_len), rlen)
    np.testing.assert_array_equal(to_np(kp.float()), rk)
    np.testing.assert_array_equal(to_np(vp.float()), rv)


def test_commit_rejects_a_position_without_a_page():
    import torch
    E = cuda_ready()
    c = _setup(3, [126], 128, 8, 128, (1, 2, 2, 2), 3)
    c["table"][:, 1:] = -1                 # the second page is missing
    c["alen"][:] = 3
    c["anodes"][0, :4] = 0                  # in range: only the page is missing
    dev = lambda a, t: torch.from_numpy(np.ascontiguousarray(a)).to(t).cuda()
    bf, i32 = torch.bfloat16, torch.int32
    kp = dev(c["kp"], bf)
    kv_len = dev(c["kv_len"], i32)
    st = torch.zeros(1, dtype=i32, device="cuda")
    E.eagle_kv_commit_paged(dev(c["tree_off"], i32), dev(c["alen"], i32), dev(c["anodes"], i32),
                            dev(c["kt"], bf), dev(c["vt"], bf), kp, dev(c["vp"], bf),
                            dev(c["table"], i32), kv_len, st, max_depth=3)
    torch.cuda.synchronize()
    assert int(st.item()) == 1                      # EAGLE_ERR_INVALID_ARG
    assert int(kv_len.item()) == 126                # the sequence is left unchanged
    np.testing.assert_array_equal(to_np(kp.float()), c["kp"])
