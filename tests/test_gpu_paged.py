"""GPU parity of tree attention over a paged KV cache (eagle_tree_attn_paged).

Each sequence's cache is scattered over shuffled pages of a pool.  Checked
against the oracle (per-element bound as in test_gpu_attn) and, where the
same kernel runs, bit for bit against eagle_tree_attn on the packed cache:
paging moves the keys, not the arithmetic."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, report_attn_err, to_np, tol_for

pytestmark = pytest.mark.gpu


def _case(seed, dtype, Ls, levels, Hq, Hkv, D, page_size, spare=5):
    B = len(Ls)
    parents = [synth.random_level_tree(seed + b, levels, 5)[0] for b in range(B)]
    sizes = [len(p) for p in parents]
    T = sum(sizes)
    tree_off = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    cast = synth.to_bf16_values if dtype == "bf16" else (lambda a: a)
    q = cast(synth.normal(seed, "q", (T, Hq, D)))
    kt = cast(synth.normal(seed, "kt", (T, Hkv, D)))
    vt = cast(synth.normal(seed, "vt", (T, Hkv, D)))
    need = [(L + page_size - 1) // page_size for L in Ls]
    n_pages = sum(need) + spare
    perm = np.random.default_rng(seed).permutation(n_pages)
    kp = cast(synth.normal(seed, "kp", (n_pages, page_size, Hkv, D)))
    vp = cast(synth.normal(seed, "vp", (n_pages, page_size, Hkv, D)))
    max_pages = max(max(need), 1)
    table = np.full((B, max_pages), -1, np.int32)
    nxt = 0
    for b in range(B):
        for j in range(need[b]):
            table[b, j] = perm[nxt]
            nxt += 1
    kv_len = np.array(Ls, np.int32)
    return (q, kt, vt, kp, vp, table, kv_len, tree_off,
            np.concatenate(parents).astype(np.int32))


def _dev(a, t):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(t).cuda()


def _run_paged(E, dtype, q, kt, vt, kp, vp, table, kv_len, tree_off, parent):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    i32 = torch.int32
    T, Hq, D = q.shape
    out = torch.full((T, Hq, D), -7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=i32, device="cuda")
    E.eagle_tree_attn_paged(_dev(q, tdt), _dev(kt, tdt), _dev(vt, tdt), _dev(kp, tdt),
                            _dev(vp, tdt), _dev(table, i32), _dev(kv_len, i32),
                            _dev(tree_off, i32), _dev(parent, i32), out, st,
                            max_nodes=int(np.max(np.diff(tree_off))),
                            max_kv=int(np.max(kv_len)))
    torch.cuda.synchronize()
    return to_np(out), int(st.item())


def _run_packed(E, dtype, q, kt, vt, kc, vc, kv_off, tree_off, parent):
    import torch
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    i32 = torch.int32
    T, Hq, D = q.shape
    Hkv = kt.shape[1]
    if kc.shape[0] == 0:
        kc = np.zeros((1, Hkv, D), np.float32)
        vc = kc
    out = torch.full((T, Hq, D), -7.0, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=i32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    E.eagle_tree_attn(_dev(q, tdt), _dev(kt, tdt), _dev(vt, tdt), _dev(kc, tdt), _dev(vc, tdt),
                      _dev(kv_off, i32), _dev(tree_off, i32), _dev(parent, i32), out, st,
                      max_nodes=int(np.max(np.diff(tree_off))),
                      max_kv=int(np.max(np.diff(kv_off))), ws=ws)
    torch.cuda.synchronize()
    return to_np(out), int(st.item())


@pytest.mark.parametrize("dtype,Ls,levels,Hq,Hkv,page", [
    ("bf16", [1000, 0, 1, 300], (1, 8, 8, 8, 8, 8, 8, 8, 8), 32, 8, 128),   # tensor cores
    ("bf16", [2048, 700], (1, 10, 10, 10, 10, 10, 10), 32, 32, 256),      # MHA, 256-key pages
    ("bf16", [333, 64], (1, 4, 4, 4), 8, 2, 16),                           # 16-key pages
    ("f32", [129, 0, 40], (1, 3, 5, 2), 8, 2, 32),                         # fp32
])
def test_paged_attention_matches_oracle_and_packed(dtype, Ls, levels, Hq, Hkv, page):
    E = cuda_ready()
    case = _case(len(Ls) * 13 + page, dtype, Ls, levels, Hq, Hkv, 128, page)
    got, st = _run_paged(E, dtype, *case)
    assert st == 0
    q, kt, vt, kp, vp, table, kv_len, tree_off, parent = case
    ref, ab = O.tree_attn_paged(*case, with_abs=True)
    assert report_attn_err(f"paged {dtype} page={page}", got, ref, ab) <= tol_for(dtype)
    if dtype == "bf16" and page % 128:
        return        # this page size runs the CUDA-core kernel, the packed cache does not
    kc, kv_off = O.gather_pages(kp, table, kv_len)
    vc, _ = O.gather_pages(vp, table, kv_len)
    packed, st = _run_packed(E, dtype, q, kt, vt, kc, vc, kv_off.astype(np.int32), tree_off,
                             parent)
    assert st == 0
    np.testing.assert_array_equal(got, packed)


def test_page_outside_the_pool_is_reported():
    E = cuda_ready()
    case = list(_case(5, "bf16", [400], (1, 4, 4), 32, 8, 128, 128))
    table = case[5].copy()
    table[0, 1] = 10_000
    case[5] = table
    _, st = _run_paged(E, "bf16", *case)
    assert st == 1                                  # EAGLE_ERR_INVALID_ARG
