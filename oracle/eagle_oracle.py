"""Plain CPU oracle of the EAGLE / EAGLE-2 tree-verify step.

TEST INFRASTRUCTURE ONLY.  This file is imported by the tests, by the smoke
check and by the benchmark's CPU-baseline leg, never by the product path.  It
shares no code with the CUDA library: it is written from the method's
description alone, in numpy, with fp64 arithmetic wherever the method is
floating point, and favours the obvious formulation over speed.

Sources (page title, then section):
  [S4000]   大模型推理效率突破：EAGLE推测解码算法在摩尔线程GPU的实践与优化
            - "greedy decoding" paragraph of the verification-strategy part
            - "random decoding" paragraph (accept with min(1, q/p), else
              resample from the corrected distribution)
            - "EAGLE的创新点" list, item 2 (tree attention turns every path
              into one attention mask, one target forward pass)
  [EAGLE]   大模型推理效率无损提升3倍，滑铁卢大学、北京大学等机构发布EAGLE
            - speculative-sampling paragraph (alpha accepted -> alpha+1 tokens)
            - workflow paragraph (frozen LM head gives the next-token
              distribution of every node)
            - "树状生成结构" (sparse draft tree)
            - "多轮投机采样" (multi-round speculative sampling over a tree;
              the draft probability of every sampled token is recorded)
  [EAGLE-2] EAGLE-2：動態草稿樹讓 LLM 推論加速 4 倍而不失精度
            - §2 "推測解碼的基礎原理" (rejection sampling keeps the output
              distribution equal to the target's)
            - §2 "EAGLE-2 的核心創新：動態草稿樹", items 1-3 (confidence,
              adaptive expansion, greedy selection under a draft-token budget)

Readings taken where the pages leave a step open (each is also listed, with
its reason, in the design notes):
  * tree attention: no positional encoding inside the step; scale 1/sqrt(d);
    GQA kv head of query head h is h // (Hq/Hkv).
  * LM head: q = softmax(z / temperature); argmax takes the lowest index on
    ties; the "top-2 gap" is top1 - second largest logit (duplicates count).
  * greedy walk: children scanned in ascending node index; the lowest index
    wins among equal tokens.
  * multi-round stochastic walk: the pseudocode the EAGLE release page refers
    to is missing, so the algorithm below is the recursive rejection-sampling
    rule written to be lossless and reproducible bit for bit:
      - test:    accept child c (token t) iff u_accept[c] * p_k[t] < q_k[t],
                 evaluated exactly (fp32 x fp32 is exact in fp64);
      - reject:  r = max(0, q_k - p_k) (fp32), W = trunc(r * 2^40) (integer),
                 Z = sum W (exact), q_{k+1} = fp32(W) / fp32(Z), the plain fp32
                 quotient; Z == 0 keeps q_{k+1} = q_k;
      - p update, NO_REPLACE (siblings drawn without replacement): P =
                 trunc(p_k * 2^40) with the rejected token's entry zeroed,
                 p_{k+1} = fp32(P) / fp32(sum P)  (all zero if the sum is 0);
                 REPLACE (siblings drawn i.i.d.): p_{k+1} = p_k;
      - stop:    sample from q_final by inverse CDF over W = trunc(q*2^40):
                 U = trunc(u_sample*2^24), target = (U*Z) >> 24, token =
                 smallest j whose inclusive prefix sum exceeds target.
    Mass below 2^-40 per token is dropped (at most V*2^-40 in total).  Every
    operation rounds to nearest once (IEEE), so the result is reproducible
    bit for bit on any IEEE machine.
  * EAGLE-2 expand/rerank: a node's value is its cumulative draft log-prob
    (the log of the product of draft confidences along its path).  Level d:
    every frontier node takes the top-k tokens of its draft row (value
    descending, token ascending); child score = fp32(parent score + logp);
    the next frontier is the top-k children by (score desc, creation order).
    Finalize: keep the top-`budget` pool nodes by (score desc, creation
    order), then number them by (depth, score desc, creation order).

Every function here is pinned by CPU tests to closed forms, invariants,
brute force or special cases that reduce to textbook routines; none is
"parity unpinned".
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

import numpy as np

FRAC_BITS = 40            # fixed-point fraction bits of resampling weights
U_BITS = 24               # uniforms are multiples of 2^-24
_SCALE40 = np.float32(2.0 ** FRAC_BITS)

MODE_REPLACE = 0
MODE_NO_REPLACE = 1

__all__ = [
    "FRAC_BITS", "MODE_REPLACE", "MODE_NO_REPLACE", "OracleNumericError",
    "tree_path", "tree_children", "tree_depths", "tree_attn", "causal_attn",
    "gather_pages", "tree_attn_paged", "kv_commit_paged",
    "lmhead_softmax", "accept_greedy", "accept_stochastic",
    "expand_level", "expand_finalize", "build_eagle2_tree", "f32_of_int",
    "static_template_full", "build_static_tree",
    "draft_head", "draft_logp_row", "build_eagle2_tree_with_head",
    "bf16_round", "rmsnorm", "rope", "silu", "tree_positions", "decoder_layer",
    "decoder_layer_causal",
]


class OracleNumericError(ValueError):
    """Raised where the CUDA path reports a numeric status (NaN/Inf, an
    out-of-range probability or a distribution with no mass)."""


# --------------------------------------------------------------------------
# tree helpers
# --------------------------------------------------------------------------
def tree_path(parent_local: Sequence[int], i: int) -> List[int]:
    """Nodes on the root -> i path (inclusive), by following parent[]."""
    path = []
    j = int(i)
    while j >= 0:
        path.append(j)
        j = int(parent_local[j])
    return path[::-1]


def tree_children(parent_local: Sequence[int], i: int) -> List[int]:
    """Children of node i, ascending node index."""
    return [j for j in range(len(parent_local)) if int(parent_local[j]) == i]


def tree_depths(parent_local: Sequence[int]) -> List[int]:
    return [len(tree_path(parent_local, i)) - 1 for i in range(len(parent_local))]


def _check_tree(parent_local):
    if len(parent_local) == 0 or int(parent_local[0]) != -1:
        raise ValueError("tree root must be node 0 with parent -1")
    for i in range(1, len(parent_local)):
        if not (0 <= int(parent_local[i]) < i):
            raise ValueError(f"parent[{i}]={parent_local[i]} is not in [0,{i})")


# --------------------------------------------------------------------------
# a1: tree attention
# --------------------------------------------------------------------------
def tree_attn(q, k_tree, v_tree, k_cache, v_cache, kv_off, tree_off, parent,
              scale: Optional[float] = None, nodes: Optional[Sequence[int]] = None,
              with_abs: bool = False):
    """Tree-masked attention of every draft-tree node over [KV cache | its
    ancestors and itself].

    [S4000] "EAGLE的创新点" item 2 and [EAGLE] workflow paragraph: all tree
    paths are verified in one target forward pass by an attention mask in
    which node i sees the cached context and exactly the nodes on its own
    root-to-i path.

    q [T,Hq,D], k_tree/v_tree [T,Hkv,D], k_cache/v_cache [sum L,Hkv,D],
    kv_off/tree_off [B+1], parent [T] (local per sequence, -1 at the root).
    Returns O [T,Hq,D] float64 (rows outside `nodes`, if given, stay zero).
    With `with_abs`, also returns A [T,Hq,D] = sum_j p_j |v_j| with the same
    softmax weights p: the magnitude of the terms each output element sums,
    which is the scale its rounding error is measured against.
    """
    q = np.asarray(q, dtype=np.float64)
    kt = np.asarray(k_tree, dtype=np.float64)
    vt = np.asarray(v_tree, dtype=np.float64)
    kc = np.asarray(k_cache, dtype=np.float64)
    vc = np.asarray(v_cache, dtype=np.float64)
    T, Hq, D = q.shape
    Hkv = kt.shape[1]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = Hq // Hkv
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    out = np.zeros((T, Hq, D), dtype=np.float64)
    absout = np.zeros((T, Hq, D), dtype=np.float64) if with_abs else None
    B = len(tree_off) - 1
    want = None if nodes is None else set(int(n) for n in nodes)
    for b in range(B):
        t0, t1 = int(tree_off[b]), int(tree_off[b + 1])
        c0, c1 = int(kv_off[b]), int(kv_off[b + 1])
        par = [int(x) for x in parent[t0:t1]]
        _check_tree(par)
        for i in range(t1 - t0):
            if want is not None and (t0 + i) not in want:
                continue
            path = [t0 + j for j in tree_path(par, i)]
            keys = np.concatenate([kc[c0:c1], kt[path]], axis=0)   # [n,Hkv,D]
            vals = np.concatenate([vc[c0:c1], vt[path]], axis=0)
            qi = q[t0 + i].reshape(Hkv, G, D)
            sc = np.einsum("nkd,kgd->kgn", keys, qi) * s            # [Hkv,G,n]
            sc -= sc.max(axis=2, keepdims=True)
            w = np.exp(sc)
            o = np.einsum("kgn,nkd->kgd", w, vals) / w.sum(axis=2)[..., None]
            out[t0 + i] = o.reshape(Hq, D)
            if with_abs:
                a = np.einsum("kgn,nkd->kgd", w, np.abs(vals)) / w.sum(axis=2)[..., None]
                absout[t0 + i] = a.reshape(Hq, D)
    return (out, absout) if with_abs else out


def gather_pages(pages, block_table, kv_len):
    """A paged KV cache read back as the packed cache of tree_attn: sequence
    b's keys are its first kv_len[b] positions, position p sitting at row
    p % page_size of page block_table[b][p // page_size] of the pool
    pages [n_pages, page_size, Hkv, D].  Returns (packed [sum L, Hkv, D],
    kv_off [B+1])."""
    pages = np.asarray(pages)
    P = pages.shape[1]
    rows, off = [], [0]
    for b, L in enumerate(kv_len):
        L = int(L)
        for p in range(L):
            page = int(block_table[b][p // P])
            if not (0 <= page < pages.shape[0]):
                raise ValueError("block table names a page outside the pool")
            rows.append(pages[page, p % P])
        off.append(off[-1] + L)
    packed = (np.stack(rows) if rows
              else np.zeros((0,) + pages.shape[2:], dtype=pages.dtype))
    return packed, np.asarray(off, dtype=np.int64)


def tree_attn_paged(q, k_tree, v_tree, k_pages, v_pages, block_table, kv_len, tree_off,
                    parent, scale: Optional[float] = None,
                    nodes: Optional[Sequence[int]] = None, with_abs: bool = False):
    """tree_attn over a paged KV cache: the same attention, with each
    sequence's cached keys and values read through its block table
    (gather_pages).  Paging changes where the cache is stored, not what is
    computed."""
    kc, kv_off = gather_pages(k_pages, block_table, kv_len)
    vc, _ = gather_pages(v_pages, block_table, kv_len)
    return tree_attn(q, k_tree, v_tree, kc, vc, kv_off, tree_off, parent, scale=scale,
                     nodes=nodes, with_abs=with_abs)


def kv_commit_paged(k_pages, v_pages, block_table, kv_len, tree_off, k_tree, v_tree,
                    accept_len, accepted_nodes):
    """Commit a verify step's accepted tokens to a paged KV cache.

    [EAGLE] speculative-sampling paragraph: alpha accepted drafts turn into
    alpha + 1 tokens; the root of the tree (the last token of the previous
    step) and the alpha accepted nodes now belong to the context, so their
    keys and values (computed by the verify pass, rotated to their
    positions) are appended to the sequence's cache: path entry i goes to
    cache position kv_len[b] + i.  Returns (k_pages, v_pages, kv_len), new
    arrays; the block table must already hold pages for the new length."""
    kp = np.array(k_pages, copy=True)
    vp = np.array(v_pages, copy=True)
    P = kp.shape[1]
    new_len = np.array(kv_len, dtype=np.int64, copy=True)
    for b in range(len(kv_len)):
        t0 = int(tree_off[b])
        for i in range(int(accept_len[b]) + 1):
            node = int(accepted_nodes[b][i])
            pos = int(kv_len[b]) + i
            page = int(block_table[b][pos // P])
            if not (0 <= page < kp.shape[0]):
                raise ValueError("no page for the committed position")
            kp[page, pos % P] = k_tree[t0 + node]
            vp[page, pos % P] = v_tree[t0 + node]
        new_len[b] = int(kv_len[b]) + int(accept_len[b]) + 1
    return kp, vp, new_len


def causal_attn(q_seq, k_seq, v_seq, n_prefix: int, scale: Optional[float] = None):
    """Ordinary causal attention of a query sequence over keys
    [prefix (n_prefix) | the sequence itself]: query p sees keys
    0 .. n_prefix + p.  An independent routine used to pin tree_attn.
    q_seq [S,Hq,D], k_seq/v_seq [n_prefix+S,Hkv,D] -> [S,Hq,D] float64."""
    q_seq = np.asarray(q_seq, dtype=np.float64)
    k_seq = np.asarray(k_seq, dtype=np.float64)
    v_seq = np.asarray(v_seq, dtype=np.float64)
    S, Hq, D = q_seq.shape
    n = k_seq.shape[0]
    Hkv = k_seq.shape[1]
    G = Hq // Hkv
    s = (1.0 / np.sqrt(D)) if scale is None else float(scale)
    out = np.empty((S, Hq, D), dtype=np.float64)
    mask = np.arange(n)[None, :] <= (n_prefix + np.arange(S))[:, None]   # [S,n]
    for h in range(Hq):
        g = h // G
        sc = (q_seq[:, h, :] @ k_seq[:, g, :].T) * s                    # [S,n]
        sc = np.where(mask, sc, -np.inf)
        sc = sc - sc.max(axis=1, keepdims=True)
        e = np.exp(sc)
        out[:, h, :] = (e / e.sum(axis=1, keepdims=True)) @ v_seq[:, g, :]
    return out


# --------------------------------------------------------------------------
# f1: one decoder layer of the target model over the tree
# --------------------------------------------------------------------------
# [EAGLE] workflow paragraph and [S4000] "EAGLE的创新点" item 2: the verify
# pass is one forward pass of the target model over all tree tokens, whose
# attention sees the cache and each node's ancestors.  The pages name the
# target models (Vicuna, LLaMA-2/3, Mixtral) but not their layer, so the
# layer here is the plain reading of "a LLaMA-shaped layer": pre-norm
# RMSNorm, Q/K/V projections, rotary position embedding on q and k, tree
# attention, output projection plus residual, RMSNorm, SwiGLU MLP plus
# residual.  A tree node's position is its sequence's cache length plus its
# depth (the position it would have on its own root-to-node path).

def bf16_round(x) -> np.ndarray:
    """Round to the nearest bf16 value (ties to even), returned as float64:
    the storage format of the layer's matrix-multiply operands."""
    x32 = np.ascontiguousarray(np.asarray(x, dtype=np.float64)).astype(np.float32)
    u = x32.view(np.uint32)
    lsb = (u >> 16) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)).view(np.float32)
    return r.astype(np.float64)


def rmsnorm(x, g, eps: float):
    """x / sqrt(mean(x^2) + eps) * g over the last axis, in fp64."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(g, np.float64)


def rope(x, pos, theta: float):
    """Rotary position embedding of x [T, heads, D] at positions pos [T]:
    the pair (x_j, x_{j+D/2}) is rotated by pos * theta^(-2j/D), in fp64."""
    x = np.asarray(x, dtype=np.float64)
    D = x.shape[-1]
    j = np.arange(D // 2, dtype=np.float64)
    ang = np.asarray(pos, np.float64)[:, None] * theta ** (-2.0 * j / D)     # [T, D/2]
    c, s_ = np.cos(ang)[:, None, :], np.sin(ang)[:, None, :]
    a, b = x[..., :D // 2], x[..., D // 2:]
    return np.concatenate([a * c - b * s_, a * s_ + b * c], axis=-1)


def silu(x):
    x = np.asarray(x, dtype=np.float64)
    return x / (1.0 + np.exp(-x))


def tree_positions(kv_len, tree_off, parent):
    """Position of every tree node: its sequence's cache length plus its
    depth in the tree."""
    pos = np.zeros(int(tree_off[-1]), dtype=np.int64)
    for b in range(len(tree_off) - 1):
        t0, t1 = int(tree_off[b]), int(tree_off[b + 1])
        dep = tree_depths([int(x) for x in parent[t0:t1]])
        pos[t0:t1] = int(kv_len[b]) + np.asarray(dep)
    return pos


def decoder_layer(x, wts: Dict[str, np.ndarray], k_cache, v_cache, kv_off, tree_off, parent,
                  Hq: int, Hkv: int, theta: float, eps: float, with_abs: bool = False):
    """One pre-norm decoder layer over every tree node.

    x [T, H] residual stream in; wts: g_attn [H], wq [Hq*D, H], wk, wv
    [Hkv*D, H], wo [H, Hq*D], g_mlp [H], wg, wu [I, H], wd [H, I] (rows are
    output features).  k_cache / v_cache hold the cached keys (already
    rotated at their positions) and values of each sequence.

    Every value that the layer feeds to a matrix multiply or to the
    attention is stored in bf16 (the tensor-core operand format): the normed
    activations, q / k / v after the rotation, the attention output and the
    gated MLP activation.  All arithmetic is fp64.  Returns a dict with the
    output residual stream "out" [T, H] and the intermediates; with
    `with_abs`, "out_abs" is the elementwise sum of the magnitudes of the
    terms that make up each output (|x| + |o|·|wo| + |m|·|wd|), the scale
    its rounding error is measured against."""
    x = np.asarray(x, dtype=np.float64)
    T, H = x.shape
    D = wts["wq"].shape[0] // Hq
    f = {k: np.asarray(v, dtype=np.float64) for k, v in wts.items()}
    kv_len = np.diff(np.asarray(kv_off, dtype=np.int64))
    pos = tree_positions(kv_len, tree_off, parent)
    a = bf16_round(rmsnorm(x, f["g_attn"], eps))
    q = bf16_round(rope((a @ f["wq"].T).reshape(T, Hq, D), pos, theta))
    k = bf16_round(rope((a @ f["wk"].T).reshape(T, Hkv, D), pos, theta))
    v = bf16_round((a @ f["wv"].T).reshape(T, Hkv, D))
    o = tree_attn(q, k, v, k_cache, v_cache, kv_off, tree_off, parent)
    ob = bf16_round(o.reshape(T, Hq * D))
    h1 = x + ob @ f["wo"].T
    bn = bf16_round(rmsnorm(h1, f["g_mlp"], eps))
    gt = bn @ f["wg"].T
    up = bn @ f["wu"].T
    m = bf16_round(silu(gt) * up)
    out = h1 + m @ f["wd"].T
    res = {"out": out, "h1": h1, "q": q, "k": k, "v": v, "attn": o, "pos": pos}
    if with_abs:
        res["out_abs"] = np.abs(x) + np.abs(ob) @ np.abs(f["wo"]).T + np.abs(m) @ np.abs(f["wd"]).T
    return res


def decoder_layer_causal(x_seq, wts: Dict[str, np.ndarray], k_prefix, v_prefix, pos0: int,
                         Hq: int, Hkv: int, theta: float, eps: float):
    """The same layer run as an ordinary causal sequence: tokens x_seq
    [S, H] at positions pos0 .. pos0+S-1 after a cached prefix (k_prefix,
    v_prefix [pos0, Hkv, D]); token p attends to the prefix and tokens
    0..p.  Independent of the tree routines (causal_attn); used to pin
    decoder_layer.  Same bf16 storage points.  Returns out [S, H]."""
    x = np.asarray(x_seq, dtype=np.float64)
    S, H = x.shape
    D = wts["wq"].shape[0] // Hq
    f = {k: np.asarray(v, dtype=np.float64) for k, v in wts.items()}
    pos = pos0 + np.arange(S)
    a = bf16_round(rmsnorm(x, f["g_attn"], eps))
    q = bf16_round(rope((a @ f["wq"].T).reshape(S, Hq, D), pos, theta))
    k = bf16_round(rope((a @ f["wk"].T).reshape(S, Hkv, D), pos, theta))
    v = bf16_round((a @ f["wv"].T).reshape(S, Hkv, D))
    kk = np.concatenate([np.asarray(k_prefix, np.float64), k], axis=0)
    vv = np.concatenate([np.asarray(v_prefix, np.float64), v], axis=0)
    o = causal_attn(q, kk, vv, n_prefix=pos0)
    h1 = x + bf16_round(o.reshape(S, Hq * D)) @ f["wo"].T
    bn = bf16_round(rmsnorm(h1, f["g_mlp"], eps))
    m = bf16_round(silu(bn @ f["wg"].T) * (bn @ f["wu"].T))
    return h1 + m @ f["wd"].T


# --------------------------------------------------------------------------
# a2: LM head, softmax, argmax
# --------------------------------------------------------------------------
def lmhead_softmax(h, w_lm, temperature: float = 1.0, want_q: bool = True,
                   rows: Optional[Sequence[int]] = None, vocab_chunk: int = 8192
                   ) -> Dict[str, np.ndarray]:
    """Frozen LM head over every tree node and its next-token distribution.

    [EAGLE] workflow paragraph: the frozen classification head maps each
    node's top-layer feature to a next-token distribution; with temperature
    the distribution is softmax(z / temperature).

    z = h @ w_lm^T in fp64 (inputs up-converted exactly).  Returns argmax
    (lowest index on ties), row_max = max z, row_lse = log sum exp(z/T),
    top2_gap = top1 - second largest z, and q = softmax(z/T) rounded to fp32
    (only if want_q).  `rows` restricts the computation to some rows.
    The vocabulary is processed in column blocks only to bound memory; each
    logit is one complete fp64 dot product."""
    h = np.asarray(h)
    if rows is not None:
        h = h[np.asarray(rows, dtype=np.int64)]
    h64 = h.astype(np.float64)
    V = w_lm.shape[0]
    z = np.empty((h64.shape[0], V), dtype=np.float64)
    for v0 in range(0, V, vocab_chunk):
        v1 = min(V, v0 + vocab_chunk)
        z[:, v0:v1] = h64 @ np.asarray(w_lm[v0:v1], dtype=np.float64).T
    if not np.all(np.isfinite(z)):
        raise OracleNumericError("non-finite logit")
    out = {}
    out["argmax"] = np.argmax(z, axis=1).astype(np.int32)
    out["row_max"] = z.max(axis=1)
    if V >= 2:
        top2 = -np.partition(-z, 1, axis=1)[:, :2]
        out["top2_gap"] = top2[:, 0] - top2[:, 1]
    else:
        out["top2_gap"] = np.full(z.shape[0], np.inf)
    zt = z / float(temperature)
    mt = zt.max(axis=1, keepdims=True)
    lse = mt[:, 0] + np.log(np.exp(zt - mt).sum(axis=1))
    out["row_lse"] = lse
    if want_q:
        out["q"] = np.exp(zt - lse[:, None]).astype(np.float32)
    out["z"] = z
    return out


# --------------------------------------------------------------------------
# a3: greedy acceptance
# --------------------------------------------------------------------------
def accept_greedy(tree_off, parent, tokens, argmax, max_depth: int):
    """Greedy tree walk.

    [S4000] greedy-decoding paragraph: feed the drafted tokens to the target
    and match its most probable token from the first position, stopping at
    the first mismatch.  On a tree: at node `cur` accept the child whose token
    equals argmax[cur] (lowest node index if several), move there and repeat;
    the bonus token is argmax of the last accepted node.
    [EAGLE] speculative-sampling paragraph: alpha accepted drafts give
    alpha + 1 tokens from one verify pass.

    Returns accept_len [B], accepted_nodes [B, max_depth+1] (local indices of
    the root and the accepted nodes, -1 padded) and out_tokens
    [B, max_depth+1] (accepted tokens then the bonus token, -1 padded)."""
    B = len(tree_off) - 1
    W = max_depth + 1
    acc_len = np.zeros(B, dtype=np.int32)
    acc_nodes = np.full((B, W), -1, dtype=np.int32)
    out_tok = np.full((B, W), -1, dtype=np.int32)
    for b in range(B):
        t0, t1 = int(tree_off[b]), int(tree_off[b + 1])
        par = [int(x) for x in parent[t0:t1]]
        _check_tree(par)
        cur, alpha = 0, 0
        acc_nodes[b, 0] = 0
        while True:
            want = int(argmax[t0 + cur])
            nxt = -1
            for c in tree_children(par, cur):
                if int(tokens[t0 + c]) == want:
                    nxt = c
                    break
            if nxt < 0:
                break
            if alpha + 1 > max_depth:
                raise ValueError("tree deeper than max_depth")
            out_tok[b, alpha] = int(tokens[t0 + nxt])
            alpha += 1
            acc_nodes[b, alpha] = nxt
            cur = nxt
        out_tok[b, alpha] = int(argmax[t0 + cur])
        acc_len[b] = alpha
    return acc_len, acc_nodes, out_tok


# --------------------------------------------------------------------------
# a4: multi-round stochastic acceptance
# --------------------------------------------------------------------------
def f32_of_int(n: int) -> np.float32:
    """Round a non-negative integer to the nearest float32 (ties to even)."""
    n = int(n)
    if n < 0:
        raise ValueError("negative")
    e = n.bit_length()
    if e <= 24:
        return np.float32(n)
    shift = e - 24
    m = n >> shift
    rem = n - (m << shift)
    half = 1 << (shift - 1)
    if rem > half or (rem == half and (m & 1)):
        m += 1
    return np.float32(float(m) * float(2 ** shift))


def _fixed40(x: np.ndarray) -> np.ndarray:
    """trunc(x * 2^40) for fp32 x in [0, 1]: the scaling is exact."""
    return (x.astype(np.float32) * _SCALE40).astype(np.uint64)


def _normalise(Wint: np.ndarray, Z: int) -> np.ndarray:
    """The renormalised weights W / Z as the plain fp32 quotient
    fp32(W) / fp32(Z): each operand rounded to nearest once, then one IEEE
    division (round to nearest).  W <= 2^40 < 2^53, so W -> fp64 is exact
    and fp64 -> fp32 rounds once."""
    wf = Wint.astype(np.float64).astype(np.float32)
    zf = f32_of_int(Z)
    return (wf / zf).astype(np.float32)


def _check_row(x: np.ndarray, what: str):
    if not np.all(np.isfinite(x)) or np.any(x < 0) or np.any(x > 1):
        raise OracleNumericError(f"{what} row has a value outside [0,1]")


def _sample_fixed(qrow: np.ndarray, u: np.float32, info: Optional[dict] = None) -> int:
    """Inverse-CDF sample from an fp32 distribution over integer weights.
    If `info` is given it receives the target and the chosen token's CDF
    interval [lo, hi) (integers), for diagnosing near-ties."""
    Wq = _fixed40(qrow)
    Z = int(Wq.sum(dtype=np.uint64))
    if Z == 0:
        raise OracleNumericError("distribution with no mass above 2^-40")
    U = int(np.float32(u) * np.float32(2.0 ** U_BITS))
    if not (0 <= U < (1 << U_BITS)):
        raise ValueError("u_sample outside [0,1)")
    target = (U * Z) >> U_BITS
    csum = np.cumsum(Wq, dtype=np.uint64)
    tok = int(np.searchsorted(csum, np.uint64(target), side="right"))
    if info is not None:
        info.update(target=target, Z=Z, lo=int(csum[tok]) - int(Wq[tok]), hi=int(csum[tok]))
    return tok


def accept_stochastic(tree_off, parent, tokens, q, p_rows, p_row_of_node,
                      u_accept, u_sample, max_depth: int,
                      mode: int = MODE_NO_REPLACE, trace: Optional[list] = None):
    """Multi-round speculative sampling over the draft tree.

    [S4000] random-decoding paragraph: accept a drafted token with
    probability min(1, q/p) (accept when the uniform falls below the ratio),
    otherwise resample from the corrected distribution.  [EAGLE]
    "多轮投机采样": the rule is applied recursively, child after child, using
    the recorded draft probability of every sampled token.  [EAGLE-2] §2
    basic principle: the result follows the target distribution exactly.

    Walk: at `cur`, q_0 = q[cur], p_0 = p_rows[p_row_of_node[first child]].
    For each child c in ascending node index (token t): accept iff
    u_accept[c] * p_k[t] < q_k[t] (exact in fp64); on accept move to c and
    restart; on reject form q_{k+1}, p_{k+1} as in the module docstring.
    When every child is rejected, or cur is a leaf, sample the bonus token
    from the current q with u_sample[cur].

    q [T,V] fp32, p_rows [R,V] fp32, p_row_of_node [T] (global row index),
    u_accept/u_sample [T] fp32 on [0,1).  Returns accept_len [B],
    accepted_nodes [B,max_depth+1], out_tokens [B,max_depth+1]."""
    B = len(tree_off) - 1
    Wd = max_depth + 1
    acc_len = np.zeros(B, dtype=np.int32)
    acc_nodes = np.full((B, Wd), -1, dtype=np.int32)
    out_tok = np.full((B, Wd), -1, dtype=np.int32)
    for b in range(B):
        t0, t1 = int(tree_off[b]), int(tree_off[b + 1])
        par = [int(x) for x in parent[t0:t1]]
        _check_tree(par)
        cur, alpha = 0, 0
        acc_nodes[b, 0] = 0
        while True:
            qk = np.array(q[t0 + cur], dtype=np.float32, copy=True)
            _check_row(qk, "q")
            kids = tree_children(par, cur)
            moved = False
            if kids:
                pk = np.array(p_rows[int(p_row_of_node[t0 + kids[0]])],
                              dtype=np.float32, copy=True)
                _check_row(pk, "p")
                for c in kids:
                    t = int(tokens[t0 + c])
                    ua = np.float32(u_accept[t0 + c])
                    if not (0.0 <= ua < 1.0):
                        raise ValueError("u_accept outside [0,1)")
                    accept = float(ua) * float(pk[t]) < float(qk[t])
                    if trace is not None:
                        trace.append((b, cur, c, t, float(qk[t]), float(pk[t]),
                                      bool(accept)))
                    if accept:
                        if alpha + 1 > max_depth:
                            raise ValueError("tree deeper than max_depth")
                        out_tok[b, alpha] = t
                        alpha += 1
                        acc_nodes[b, alpha] = c
                        cur = c
                        moved = True
                        break
                    # reject: residual of the target, renormalised
                    r = np.maximum(np.float32(0), qk - pk)
                    Wr = _fixed40(r)
                    Z = int(Wr.sum(dtype=np.uint64))
                    if Z > 0:
                        qk = _normalise(Wr, Z)
                    if mode == MODE_NO_REPLACE:
                        P = _fixed40(pk)
                        P[t] = 0
                        SP = int(P.sum(dtype=np.uint64))
                        pk = _normalise(P, SP) if SP > 0 else np.zeros_like(pk)
            if moved:
                continue
            info = {} if trace is not None else None
            out_tok[b, alpha] = _sample_fixed(qk, np.float32(u_sample[t0 + cur]), info)
            if trace is not None:
                trace.append((b, cur, "sample", info))
            break
        acc_len[b] = alpha
    return acc_len, acc_nodes, out_tok


# --------------------------------------------------------------------------
# a5: EAGLE-2 dynamic draft tree, expand and rerank
# --------------------------------------------------------------------------
def _topk_tokens(row: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest values, value descending then index
    ascending."""
    row = np.asarray(row, dtype=np.float32)
    if not np.all(np.isfinite(row)):
        raise OracleNumericError("non-finite draft log-prob")
    order = np.lexsort((np.arange(row.shape[0]), -row))
    return order[:k]


class _Pool:
    """Candidate pool of one sequence: parallel lists in creation order."""

    def __init__(self):
        self.token: List[int] = []
        self.parent: List[int] = []     # pool index, -1 = the root
        self.score: List[np.float32] = []
        self.depth: List[int] = []
        self.p_row: List[int] = []      # local draft row the token came from
        self.frontier: List[int] = []   # pool indices, frontier rank order


def expand_level(pools: List[_Pool], draft_logp, level: int, k: int,
                 rows_per_seq: int):
    """One EAGLE-2 expansion level for every sequence.

    [EAGLE-2] §2 dynamic draft tree, items 1-2: every frontier node is
    expanded by its draft distribution; a child's value is the product of
    the draft confidences on its path, kept here as a cumulative log-prob.
    Row layout of draft_logp: [B, rows_per_seq, V]; level 0 uses row 0 (the
    root), level d >= 1 uses rows 1 + (d-1)*k + f for frontier rank f."""
    B = len(pools)
    V = draft_logp.shape[-1]
    kk = min(k, V)
    lp = np.asarray(draft_logp, dtype=np.float32).reshape(B, rows_per_seq, V)
    for b in range(B):
        pool = pools[b]
        if level == 0:
            front = [(-1, np.float32(0.0), 0, 0)]   # (pool idx, score, depth, row)
        else:
            front = [(f, pool.score[f], pool.depth[f], 1 + (level - 1) * k + r)
                     for r, f in enumerate(pool.frontier)]
        children = []                                # creation order
        for (fidx, fscore, fdepth, row) in front:
            for t in _topk_tokens(lp[b, row], kk):
                sc = np.float32(np.float32(fscore) + lp[b, row, t])
                children.append((int(t), fidx, sc, fdepth + 1, row))
        base = len(pool.token)
        for (t, fidx, sc, dep, row) in children:
            pool.token.append(t)
            pool.parent.append(fidx)
            pool.score.append(sc)
            pool.depth.append(dep)
            pool.p_row.append(row)
        # next frontier: top-k children by score, ties by creation order
        order = sorted(range(len(children)), key=lambda j: (-float(children[j][2]), j))
        pool.frontier = [base + j for j in order[:kk]]
    return pools


def expand_finalize(pools: List[_Pool], budget: Sequence[int],
                    root_token: Sequence[int], rows_per_seq: int):
    """EAGLE-2 rerank: keep the global top-`budget` pool nodes.

    [EAGLE-2] §2 dynamic draft tree, item 3: under a fixed draft-token budget,
    choose nodes greedily to maximise the expected acceptance length.  A
    node's value (product of confidences on its path) never exceeds its
    parent's, so the top-`budget` values form a parent-closed set whose total
    value is the largest of any parent-closed set of that size.

    Returns dict of tree_off [B+1], parent [T] (local), tokens [T], depth [T],
    score [T] (fp32; root 0), p_row_of_node [T] (global row, root -1)."""
    B = len(pools)
    trees = []
    for b in range(B):
        pool = pools[b]
        n = len(pool.token)
        keep_n = min(int(budget[b]), n)
        sel = sorted(range(n), key=lambda j: (-float(pool.score[j]), j))[:keep_n]
        sel_set = set(sel)
        for j in sel:
            if pool.parent[j] >= 0 and pool.parent[j] not in sel_set:
                raise AssertionError("selection is not parent-closed")
        order = sorted(sel, key=lambda j: (pool.depth[j], -float(pool.score[j]), j))
        node_of = {j: i + 1 for i, j in enumerate(order)}
        par = [-1] + [0 if pool.parent[j] < 0 else node_of[pool.parent[j]] for j in order]
        tok = [int(root_token[b])] + [pool.token[j] for j in order]
        dep = [0] + [pool.depth[j] for j in order]
        sc = [np.float32(0)] + [pool.score[j] for j in order]
        prow = [-1] + [b * rows_per_seq + pool.p_row[j] for j in order]
        trees.append((par, tok, dep, sc, prow))
    tree_off = np.zeros(B + 1, dtype=np.int32)
    tree_off[1:] = np.cumsum([len(t[0]) for t in trees])
    cat = lambda i, dt: np.concatenate([np.asarray(t[i], dtype=dt) for t in trees])
    return {"tree_off": tree_off, "parent": cat(0, np.int32), "tokens": cat(1, np.int32),
            "depth": cat(2, np.int32), "score": cat(3, np.float32),
            "p_row_of_node": cat(4, np.int32)}


def static_template_full(K: int, m: int):
    """The full static top-K tree of m draft steps: every node of depth < m
    has K children, its K most probable draft tokens ([S4000] "EAGLE的创新点"
    item 1: keep top tokens at every step; K^m root-to-leaf paths).
    Returns (parent, rank, row) lists in level order: node i's token is the
    rank[i]-th most probable token of the distribution its parent was
    expanded with, and row[i] is the draft row that node i itself is expanded
    with (-1 for a leaf); expanded nodes take rows 0, 1, ... in node order."""
    parent, rank, row = [-1], [0], []
    level = [0]
    for _ in range(m):
        nxt = []
        for p in level:
            for r in range(K):
                parent.append(p)
                rank.append(r)
                nxt.append(len(parent) - 1)
        level = nxt
    has_kids = set(parent[1:])
    n_rows = 0
    for i in range(len(parent)):
        if i in has_kids:
            row.append(n_rows)
            n_rows += 1
        else:
            row.append(-1)
    return parent, rank, row


def build_static_tree(draft_logp, B: int, tmpl_parent, tmpl_rank, tmpl_row, root_token):
    """EAGLE-1 static draft tree ([EAGLE-2] §2, the fixed top-k tree that the
    dynamic tree replaces; [S4000] "EAGLE的创新点" item 1).

    The tree's shape is a fixed template, the same for every sequence and
    step: template node i (i >= 1) is the tmpl_rank[i]-th most probable token
    (value descending, token ascending) of the draft row its parent
    tmpl_parent[i] was expanded with, row tmpl_row[parent] of the sequence's
    draft_logp [B, R, V].  Its score is fp32(parent score + logp), the same
    cumulative log-prob as the dynamic tree's.  Nodes keep the template's
    numbering (parent before child).  Returns the arrays of
    expand_finalize."""
    lp = np.asarray(draft_logp, dtype=np.float32)
    R, V = lp.shape[-2], lp.shape[-1]
    lp = lp.reshape(B, R, V)
    n = len(tmpl_parent)
    _check_tree(tmpl_parent)
    par, tok, dep, sc, prow = [], [], [], [], []
    for b in range(B):
        order = {}
        t = [int(root_token[b])] + [0] * (n - 1)
        d = [0] * n
        s = [np.float32(0)] * n
        pr = [-1] * n
        for i in range(1, n):
            p = int(tmpl_parent[i])
            r = int(tmpl_row[p])
            if not (0 <= r < R):
                raise ValueError("an expanded template node has no draft row")
            if r not in order:
                order[r] = _topk_tokens(lp[b, r], V)
            k = int(tmpl_rank[i])
            if not (0 <= k < V):
                raise ValueError("template rank outside the vocabulary")
            t[i] = int(order[r][k])
            d[i] = d[p] + 1
            s[i] = np.float32(np.float32(s[p]) + lp[b, r, t[i]])
            pr[i] = b * R + r
        par.append([int(x) for x in tmpl_parent])
        tok.append(t)
        dep.append(d)
        sc.append(s)
        prow.append(pr)
    tree_off = np.arange(B + 1, dtype=np.int32) * n
    cat = lambda xs, dt: np.concatenate([np.asarray(x, dtype=dt) for x in xs])
    return {"tree_off": tree_off, "parent": cat(par, np.int32), "tokens": cat(tok, np.int32),
            "depth": cat(dep, np.int32), "score": cat(sc, np.float32),
            "p_row_of_node": cat(prow, np.int32)}


def draft_head(f_parent, e_token, w_draft):
    """The draft ("auto-regression") head of the loop: the next feature from
    the parent's feature and the embedding of the node's token ([EAGLE]
    workflow paragraph), one matrix: bf16([f ; e] Wd^T), Wd [H, 2H]."""
    x = np.concatenate([np.asarray(f_parent, np.float64), np.asarray(e_token, np.float64)],
                       axis=-1)
    return bf16_round(x @ np.asarray(w_draft, np.float64).T)


def draft_logp_row(feature, w_lm):
    """Draft distribution of a node: the frozen LM head on its feature, as
    fp32 log-probabilities fp32(z - lse(z)) (z and lse in fp64)."""
    z = np.asarray(w_lm, np.float64) @ np.asarray(feature, np.float64)
    m = z.max()
    lse = m + np.log(np.exp(z - m).sum())
    return (z - lse).astype(np.float32)


def build_eagle2_tree_with_head(f_ctx, root_token, emb, w_draft, w_lm, B: int, k: int,
                                depth: int, budget, rows=None):
    """The EAGLE-2 tree drafted level by level: the root's feature is
    draft_head(f_ctx[b], emb[root token]); every frontier node's feature is
    draft_head(its parent's feature, emb[its token]); its draft row is
    draft_logp_row(feature).  Returns (tree, own_rows [B, R, V] fp32).  If
    `rows` [B, R, V] is given, the tree's decisions read those rows (so a
    tree built from another implementation's rows can be checked with
    identical inputs) while own_rows still holds this function's rows,
    computed on that tree's frontiers.  Also returns scale [B, R]: for each
    row, sum_i |f_i| max_j |w_lm[j, i]|, the most a logit of the row moves
    per unit of relative change of every feature entry (the scale against
    which another implementation's rounding of the feature is measured)."""
    V = np.asarray(w_lm).shape[0]
    R = 1 + (depth - 1) * k
    own = np.zeros((B, R, V), dtype=np.float32)
    scale = np.zeros((B, R))
    wmax = np.abs(np.asarray(w_lm, np.float64)).max(axis=0)
    use = own if rows is None else np.asarray(rows, dtype=np.float32).reshape(B, R, V)
    pools = [_Pool() for _ in range(B)]
    feats = [dict() for _ in range(B)]      # pool index (-1: root) -> feature
    for lev in range(depth):
        for b in range(B):
            if lev == 0:
                f = draft_head(f_ctx[b], emb[int(root_token[b])], w_draft)
                feats[b][-1] = f
                own[b, 0] = draft_logp_row(f, w_lm)
                scale[b, 0] = np.abs(f) @ wmax
            else:
                pool = pools[b]
                for r, q in enumerate(pool.frontier):
                    f = draft_head(feats[b][pool.parent[q]], emb[pool.token[q]], w_draft)
                    feats[b][q] = f
                    own[b, 1 + (lev - 1) * k + r] = draft_logp_row(f, w_lm)
                    scale[b, 1 + (lev - 1) * k + r] = np.abs(f) @ wmax
        expand_level(pools, use, lev, k, R)
    return expand_finalize(pools, budget, root_token, R), own, scale


def build_eagle2_tree(draft_logp, B: int, k: int, depth: int, budget, root_token):
    """All expansion levels followed by the rerank."""
    V = draft_logp.shape[-1]
    R = 1 + (depth - 1) * k
    pools = [_Pool() for _ in range(B)]
    for lev in range(depth):
        expand_level(pools, draft_logp.reshape(B, R, V), lev, k, R)
    return expand_finalize(pools, budget, root_token, R)
