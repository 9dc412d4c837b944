"""GPU parity of tree attention against the oracle.

Error metric per element: |g - r| / max(|r|, sum_j p_j |v_j|) with the
oracle's own fp64 softmax weights p, bounded by 2e-3 for bf16 inputs and
1e-5 for fp32 (the stricter |g - r| / max(|r|, 1e-3 rms) is printed beside
it for the record).  The mask itself is checked by an
invariant that holds at any size: changing the keys/values of one node must
leave every node outside its subtree bit-for-bit unchanged."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, report_attn_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _case(seed, dtype, Ls, levels_list, Hq, Hkv, D):
    B = len(Ls)
    parents = []
    for b in range(B):
        par, _ = synth.random_level_tree(seed + b, levels_list[b % len(levels_list)], 5)
        parents.append(par)
    sizes = [len(p) for p in parents]
    T = sum(sizes)
    tree_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    kv_off = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    cast = synth.to_bf16_values if dtype == "bf16" else (lambda a: a)
    q = cast(synth.normal(seed, "q", (T, Hq, D)))
    kt = cast(synth.normal(seed, "kt", (T, Hkv, D)))
    vt = cast(synth.normal(seed, "vt", (T, Hkv, D)))
    kc = cast(synth.normal(seed, "kc", (int(kv_off[-1]), Hkv, D)))
    vc = cast(synth.normal(seed, "vc", (int(kv_off[-1]), Hkv, D)))
    return q, kt, vt, kc, vc, kv_off, tree_off, np.concatenate(parents).astype(np.int32)


def _run(E, dtype, q, kt, vt, kc, vc, kv_off, tree_off, parent):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    dev = lambda a, t=tdt: torch.from_numpy(np.ascontiguousarray(a)).to(t).cuda()
    T, Hq, D = q.shape
    Hkv = kt.shape[1]
    B = len(tree_off) - 1
    max_nodes = int(np.max(np.diff(tree_off)))
    max_kv = int(np.max(np.diff(kv_off)))
    if kc.shape[0] == 0:
        kc = np.zeros((1, Hkv, D), np.float32)
        vc = kc
    out = torch.full((T, Hq, D), -7.0, dtype=torch.float32, device="cuda")
    ws_n = E.eagle_tree_attn_workspace_bytes(B, T, Hq, Hkv, D, max_nodes, max_kv)
    ws = torch.empty(max(ws_n, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    i32 = torch.int32
    E.eagle_tree_attn(dev(q), dev(kt), dev(vt), dev(kc), dev(vc), dev(kv_off, i32),
                      dev(tree_off, i32), dev(parent, i32), out, st, max_nodes=max_nodes,
                      max_kv=max_kv, ws=ws)
    torch.cuda.synchronize()
    return to_np(out), int(st.item())


@pytest.mark.parametrize("dtype,Ls,levels,Hq,Hkv,D", [
    ("f32", [128], [(1, 4, 6, 6, 6, 3)], 4, 4, 64),                   # tiny fp32 layer
    ("f32", [0, 1, 127, 129], [(1,), (1, 3, 3), (1, 5, 9, 2)], 8, 2, 128),
    ("bf16", [300], [(1, 10, 20, 20, 10)], 32, 8, 128),              # GQA 32/8
    ("bf16", [64, 0, 1000], [(1, 8, 8, 8, 8, 8, 8, 8, 8)], 64, 8, 128),  # GQA 64/8, 65 nodes
    ("bf16", [2048], [(1, 10, 10, 10, 10, 10, 10)], 32, 32, 128),   # Vicuna-7B shaped (MHA)
])
def test_tree_attention_matches_oracle(dtype, Ls, levels, Hq, Hkv, D):
    E = cuda_ready()
    case = _case(len(Ls) * 31 + Hq, dtype, Ls, levels, Hq, Hkv, D)
    got, st = _run(E, dtype, *case)
    assert st == 0
    ref, ab = O.tree_attn(*case, with_abs=True)
    assert report_attn_err(f"{dtype} L={Ls} {Hq}/{Hkv}", got, ref, ab) <= tol_for(dtype)


def test_tree_attention_long_cache_sampled_nodes():
    # LLaMA-3-8B shaped: GQA 32/8, L = 8192, 65 nodes; the oracle checks a
    # sample of nodes (including the root and the deepest leaf)
    E = cuda_ready()
    case = _case(3, "bf16", [8192], [(1, 8, 8, 8, 8, 8, 8, 8, 8)], 32, 8, 128)
    got, st = _run(E, "bf16", *case)
    assert st == 0
    nodes = [0, 1, 17, 40, 64]
    ref, ab = O.tree_attn(*case, nodes=nodes, with_abs=True)
    assert report_attn_err("L=8192 32/8", got[nodes], ref[nodes], ab[nodes]) <= 2e-3


def test_malformed_parent_is_reported_on_the_device():
    E = cuda_ready()
    case = list(_case(9, "f32", [16], [(1, 3, 3)], 4, 4, 64))
    case[-1] = case[-1].copy()
    case[-1][4] = 5                         # parent not smaller than the child
    _, st = _run(E, "f32", *case)
    assert st == 2                          # EAGLE_ERR_INVALID_TREE


@pytest.mark.parametrize("dtype,L,Hq,Hkv", [("bf16", 8192, 32, 8), ("f32", 129, 8, 2)])
def test_changing_one_branch_leaves_the_rest_of_the_tree_unchanged(dtype, L, Hq, Hkv):
    # node i must see exactly the cache and its own root-to-i path: perturb
    # the K/V of one node and compare every other node's output bit for bit
    E = cuda_ready()
    case = list(_case(17, dtype, [L], [(1, 8, 8, 8, 8, 8, 8, 8, 8)], Hq, Hkv, 128))
    base, st = _run(E, dtype, *case)
    assert st == 0
    parent = case[-1]
    victim = 9                                   # a depth-2 node
    for which in (1, 2):                         # keys, then values
        c2 = [a.copy() if i in (1, 2) else a for i, a in enumerate(case)]
        c2[which][victim] = -c2[which][victim] + 0.5
        out, st = _run(E, dtype, *c2)
        assert st == 0
        for i in range(len(parent)):
            inside = victim in O.tree_path(parent, i)
            same = np.array_equal(out[i], base[i])
            assert same != inside, (which, i)


def test_rising_scores_force_output_rescaling():
    # Scores climb ~20 nats across every cache chunk, so the running row max
    # grows by more than 2^8 (log2 units) several times inside one CTA: the
    # kernel's deferred rescaling of O must keep the result exact.  Eight
    # heads and L = 8192 also give the largest split of one row tile (8
    # chunks, one cluster of 8).
    E = cuda_ready()
    q, kt, vt, kc, vc, kv_off, tree_off, parent = _case(23, "bf16", [8192], [(1, 10, 10)], 8, 8,
                                                        128)
    q = synth.to_bf16_values(q + 1.0)
    ramp = (np.arange(8192, dtype=np.float64) / 8192.0 * 2000.0 / 128.0)[:, None, None]
    kc = synth.to_bf16_values(0.1 * kc + ramp)
    case = (q, kt, vt, kc, vc, kv_off, tree_off, parent)
    got, st = _run(E, "bf16", *case)
    assert st == 0
    nodes = list(range(0, 21, 4))
    ref, ab = O.tree_attn(*case, nodes=nodes, with_abs=True)
    assert report_attn_err("rising scores", got[nodes], ref[nodes], ab[nodes]) <= 2e-3
