"""Seeded synthetic inputs for the EAGLE / EAGLE-2 tree-verify step.

This module only draws random numbers and lays them out; it holds none of the
verify step's arithmetic (no attention, no LM head, no acceptance rule, no
top-k).  Both the oracle-driven tests and the CUDA path are fed from here, so
the two sides always see identical inputs.

The shapes follow the workloads the EAGLE pages evaluate on (LLaMA-3-8B/70B
and Vicuna-7B shaped layers, batch 1 at A100 in the EAGLE-2 analysis page's
§3 speedup table, and a batched case for the page's §4 remark that speedup
collapses at larger batch).  The pages' benchmark suites (MT-Bench, HumanEval,
GSM8K, Alpaca, ShareGPT) and trained weights are not used: every tensor here is
drawn from a seeded distribution of the stated shape.

Generation is numpy's PCG64 Generator, seeded per workload and per tensor name
(so adding a tensor never shifts another tensor's stream).  Values that the
CUDA side stores in bf16 are rounded to bf16 here (round-to-nearest-even) and
kept as float32 arrays holding exactly-representable bf16 values, so the
oracle can up-convert them exactly.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Dict, List, Optional

import numpy as np

U24 = float(2 ** -24)


# --------------------------------------------------------------------------
# workloads
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    dtype: str                 # "f32" or "bf16": storage type of Q/K/V/h/W
    B: int                     # sequences
    Hq: int                    # query heads
    Hkv: int                   # key/value heads
    D: int                     # head dim
    H: int                     # hidden size (LM-head input width)
    V: int                     # vocabulary
    L: tuple                   # KV-cache length per sequence
    tree: str                  # "levels" (random tree of given level sizes), "eagle2"
                               # (dynamic tree) or "static" (full K-ary template)
    k: int = 0                 # EAGLE-2 top-k per expanded node; static: K children
    depth: int = 0             # EAGLE-2 expansion levels; static: draft steps m
    budget: tuple = ()         # EAGLE-2 draft-token budget per sequence
    level_sizes: tuple = ()    # random-tree level sizes (root level first)
    modes: tuple = ("greedy",)
    temperature: float = 1.0
    seed: int = 0
    draft_sigma: float = 3.0   # draft logits ~ N(0, draft_sigma)
    w_sigma: float = 0.02      # LM-head weights ~ N(0, w_sigma)
    # the full decoder layer around the attention (0: attention alone)
    I: int = 0                 # MLP intermediate size
    theta: float = 10000.0     # rotary base
    eps: float = 1e-5          # RMSNorm epsilon

    # ---- derived sizes -------------------------------------------------
    @property
    def n_nodes(self) -> List[int]:
        """Tree nodes per sequence, root included."""
        if self.tree == "levels":
            return [int(sum(self.level_sizes))] * self.B
        if self.tree == "static":
            return [sum(self.k ** i for i in range(self.depth + 1))] * self.B
        pool = self.pool_size
        return [min(int(b), pool) + 1 for b in self.budget]

    @property
    def pool_size(self) -> int:
        """EAGLE-2 candidate pool per sequence: k at level 0, k*k after."""
        if self.tree != "eagle2":
            return 0
        return self.k + (self.depth - 1) * self.k * self.k

    @property
    def rows_per_seq(self) -> int:
        """Draft-distribution rows per sequence.

        EAGLE-2 tree: one row for the root plus k frontier rows per later
        level.  Random tree: one row per node (the distribution its children
        were drafted from)."""
        if self.tree == "eagle2":
            return 1 + (self.depth - 1) * self.k
        if self.tree == "static":
            return sum(self.k ** i for i in range(self.depth))
        return int(sum(self.level_sizes))

    @property
    def T(self) -> int:
        return int(sum(self.n_nodes))

    @property
    def max_depth(self) -> int:
        if self.tree in ("eagle2", "static"):
            return self.depth
        return len(self.level_sizes) - 1

    def static_template(self):
        """The fixed tree shape of a "static" workload, as input structure:
        (parent, rank, row) lists in level order -- every node above the
        last level has k children of ranks 0..k-1, and the expanded nodes
        use draft rows 0, 1, ... in node order (leaves: -1)."""
        parent, rank = [-1], [0]
        level = [0]
        for _ in range(self.depth):
            nxt = []
            for p in level:
                for r in range(self.k):
                    parent.append(p)
                    rank.append(r)
                    nxt.append(len(parent) - 1)
            level = nxt
        expanded = sorted(set(parent[1:]))
        row = [-1] * len(parent)
        for i, node in enumerate(expanded):
            row[node] = i
        return parent, rank, row

    def scaled(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _c5_lists(seed: int):
    rng = np.random.Generator(np.random.PCG64(_seed_for(seed, "c5-shape")))
    L = tuple(int(x) for x in rng.integers(512, 16384 + 1, size=16))
    budget = tuple(int(x) for x in rng.integers(32, 64 + 1, size=16))
    return L, budget


_C5_L, _C5_BUDGET = None, None


def workloads() -> Dict[str, Workload]:
    global _C5_L, _C5_BUDGET
    if _C5_L is None:
        _C5_L, _C5_BUDGET = _c5_lists(5)
    return {
        # tiny fp32 layer: 4 heads x 64, hidden 256, vocab 1024, L=128,
        # random 26-node tree of depth 5 (root, 4 children, <=6 per level).
        "tiny_fp32": Workload(
            name="tiny_fp32", dtype="f32", B=1, Hq=4, Hkv=4, D=64, H=256,
            V=1024, L=(128,), tree="levels", level_sizes=(1, 4, 6, 6, 6, 3),
            modes=("greedy", "stochastic"), temperature=1.0, seed=0,
            draft_sigma=2.0),
        # Vicuna-7B shaped layer: MHA 32 x 128, vocab 32000, L=2048,
        # EAGLE-2 tree budget 60, depth 6, top-10; greedy acceptance.
        "vicuna7b": Workload(
            name="vicuna7b", dtype="bf16", B=1, Hq=32, Hkv=32, D=128, H=4096,
            V=32000, L=(2048,), tree="eagle2", k=10, depth=6, budget=(60,),
            modes=("greedy",), seed=0, I=11008, theta=10000.0, eps=1e-5),
        # LLaMA-3-8B shaped layer: GQA 32/8 x 128, vocab 128256, L=8192,
        # budget 64, depth 7, top-8; stochastic acceptance at T=1.
        "llama3_8b": Workload(
            name="llama3_8b", dtype="bf16", B=1, Hq=32, Hkv=8, D=128, H=4096,
            V=128256, L=(8192,), tree="eagle2", k=8, depth=7, budget=(64,),
            modes=("stochastic",), temperature=1.0, seed=0, I=14336, theta=500000.0),
        # LLaMA-3-70B shaped layer: GQA 64/8 x 128, hidden 8192, vocab 128256,
        # L=4096, budget 64, depth 8, top-8; greedy and stochastic; seed 3.
        "llama3_70b": Workload(
            name="llama3_70b", dtype="bf16", B=1, Hq=64, Hkv=8, D=128, H=8192,
            V=128256, L=(4096,), tree="eagle2", k=8, depth=8, budget=(64,),
            modes=("greedy", "stochastic"), temperature=1.0, seed=3, I=28672,
            theta=500000.0),
        # small bf16 case for the start-up check: three sequences (157 tree
        # rows, so the LM head takes its two-tile cluster path), GQA 32/8,
        # a ragged vocabulary, EAGLE-2 trees; greedy and stochastic.
        "smoke_bf16": Workload(
            name="smoke_bf16", dtype="bf16", B=3, Hq=32, Hkv=8, D=128, H=1024,
            V=4099, L=(512, 300, 700), tree="eagle2", k=8, depth=8,
            budget=(64, 40, 50), modes=("greedy", "stochastic"), temperature=0.8,
            seed=7, I=2816, theta=10000.0),
        # Vicuna-7B shaped layer verifying an EAGLE-1 static tree: the full
        # 4-ary template of 3 draft steps (85 nodes, 64 root-to-leaf paths).
        "vicuna7b_static": Workload(
            name="vicuna7b_static", dtype="bf16", B=1, Hq=32, Hkv=32, D=128, H=4096,
            V=32000, L=(2048,), tree="static", k=4, depth=3,
            modes=("greedy", "stochastic"), seed=11),
        # batched LLaMA-3-8B shaped layer: 16 sequences, L ~ U[512,16384],
        # budget ~ U[32,64], depth 8, top-8, stochastic at T=0.7; seed 5.
        "llama3_8b_batch16": Workload(
            name="llama3_8b_batch16", dtype="bf16", B=16, Hq=32, Hkv=8, D=128,
            H=4096, V=128256, L=_C5_L, tree="eagle2", k=8, depth=8,
            budget=_C5_BUDGET, modes=("stochastic",), temperature=0.7, seed=5,
            I=14336, theta=500000.0),
    }


# --------------------------------------------------------------------------
# seeded streams
# --------------------------------------------------------------------------
def _seed_for(seed: int, name: str) -> int:
    h = hashlib.sha256(f"{seed}/{name}".encode()).digest()
    return int.from_bytes(h[:8], "little")


def rng_for(seed: int, name: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(_seed_for(seed, name)))


def normal(seed: int, name: str, shape, std: float = 1.0) -> np.ndarray:
    x = rng_for(seed, name).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return x


def to_bf16_values(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (nearest-even); return them as float32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # round-to-nearest-even on the upper 16 bits; inputs here are finite
    lsb = (u >> 16) & np.uint32(1)
    r = (u + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def uniforms24(seed: int, name: str, n: int) -> np.ndarray:
    """Uniforms on [0,1) that are exact multiples of 2^-24 (float32)."""
    ints = rng_for(seed, name).integers(0, 1 << 24, size=n, dtype=np.int64)
    return (ints.astype(np.float64) * U24).astype(np.float32)


def draft_rows(seed: int, name: str, rows: int, V: int, sigma: float):
    """Draft-model output rows: logits ~ N(0, sigma), returned as fp32
    log-probabilities and fp32 probabilities, both rounded once from fp64.
    These stand in for the draft head's output distribution."""
    out_logp = np.empty((rows, V), dtype=np.float32)
    out_p = np.empty((rows, V), dtype=np.float32)
    g = rng_for(seed, name)
    chunk = max(1, (1 << 24) // max(V, 1))
    for r0 in range(0, rows, chunk):
        r1 = min(rows, r0 + chunk)
        z = g.standard_normal(size=(r1 - r0, V)) * sigma   # fp64
        m = z.max(axis=1, keepdims=True)
        lse = m + np.log(np.exp(z - m).sum(axis=1, keepdims=True))
        lp = z - lse
        out_logp[r0:r1] = lp.astype(np.float32)
        out_p[r0:r1] = np.exp(lp).astype(np.float32)
    return out_logp, out_p


def random_level_tree(seed: int, level_sizes, V: int):
    """Random tree given per-level node counts: each node's parent is drawn
    uniformly from the previous level; tokens uniform in [0, V).
    Nodes are numbered level by level, so parent[i] < i."""
    g = rng_for(seed, "tree")
    parent = [-1]
    starts = [0]
    for lev in range(1, len(level_sizes)):
        p0 = starts[-1]
        p1 = p0 + level_sizes[lev - 1]
        starts.append(p1)
        for _ in range(level_sizes[lev]):
            parent.append(int(g.integers(p0, p1)))
    parent = np.array(parent, dtype=np.int32)
    tokens = g.integers(0, V, size=len(parent)).astype(np.int32)
    return parent, tokens


# --------------------------------------------------------------------------
# full input sets
# --------------------------------------------------------------------------
def make_inputs(w: Workload, parts=("attn", "lmhead", "draft", "accept"),
                set_index: int = 0) -> Dict[str, np.ndarray]:
    """Build the seeded input arrays for workload `w`.

    `set_index` selects an independent copy (different streams) of the
    per-step tensors, used to rotate input buffers between timed steps.
    Returned arrays are host numpy arrays; bf16 tensors are float32 arrays
    holding bf16 values."""
    s = w.seed
    tag = "" if set_index == 0 else f"#{set_index}"
    out: Dict[str, np.ndarray] = {}
    bf = w.dtype == "bf16"
    cast = to_bf16_values if bf else (lambda a: a)
    n_nodes = w.n_nodes
    T = w.T
    tree_off = np.zeros(w.B + 1, dtype=np.int32)
    tree_off[1:] = np.cumsum(n_nodes)
    out["tree_off"] = tree_off
    kv_off = np.zeros(w.B + 1, dtype=np.int32)
    kv_off[1:] = np.cumsum(w.L)
    out["kv_off"] = kv_off

    if "attn" in parts:
        out["q"] = cast(normal(s, "q" + tag, (T, w.Hq, w.D)))
        out["k_tree"] = cast(normal(s, "k_tree" + tag, (T, w.Hkv, w.D)))
        out["v_tree"] = cast(normal(s, "v_tree" + tag, (T, w.Hkv, w.D)))
        sl = int(kv_off[-1])
        out["k_cache"] = cast(normal(s, "k_cache" + tag, (sl, w.Hkv, w.D)))
        out["v_cache"] = cast(normal(s, "v_cache" + tag, (sl, w.Hkv, w.D)))
    if "lmhead" in parts:
        out["h"] = cast(normal(s, "h" + tag, (T, w.H)))
        out["w_lm"] = cast(normal(s, "w_lm" + tag, (w.V, w.H), std=w.w_sigma))
    if "draft" in parts:
        R = w.rows_per_seq
        lp, p = draft_rows(s, "draft" + tag, w.B * R, w.V, w.draft_sigma)
        out["draft_logp"] = lp
        out["p_rows"] = p
        out["root_token"] = rng_for(s, "root" + tag).integers(
            0, w.V, size=w.B).astype(np.int32)
        if w.tree == "levels":
            parents, toks = [], []
            for b in range(w.B):
                par, tok = random_level_tree(s + 1000 * b, w.level_sizes, w.V)
                parents.append(par)
                toks.append(tok)
            out["parent"] = np.concatenate(parents)
            out["tokens"] = np.concatenate(toks)
            # node i's token was drafted from its parent's row
            prow = np.concatenate([
                np.where(par >= 0, par + b * R, -1).astype(np.int32)
                for b, par in enumerate(parents)])
            out["p_row_of_node"] = prow
        elif w.tree == "static":
            par, rank, row = w.static_template()
            out["tmpl_parent"] = np.array(par, dtype=np.int32)
            out["tmpl_rank"] = np.array(rank, dtype=np.int32)
            out["tmpl_row"] = np.array(row, dtype=np.int32)
        else:
            out["budget"] = np.array(w.budget, dtype=np.int32)
    if "accept" in parts:
        out["u_accept"] = uniforms24(s, "u_accept" + tag, T)
        out["u_sample"] = uniforms24(s, "u_sample" + tag, T)
    return out


def random_probs(seed: int, name: str, rows: int, V: int, sigma: float = 2.0,
                 temperature: float = 1.0) -> np.ndarray:
    """Rows of a softmax over N(0, sigma) logits (fp64 -> fp32); an input
    distribution for acceptance tests that do not run the LM head."""
    z = rng_for(seed, name).standard_normal(size=(rows, V)) * sigma / temperature
    z -= z.max(axis=1, keepdims=True)
    e = np.exp(z)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def make_layer_inputs(w: Workload, set_index: int = 0) -> Dict[str, np.ndarray]:
    """Inputs of the full decoder layer: the residual stream x [T, H] fp32
    entering the layer at every tree node (~ N(0, 1)), the layer's weights
    (rows = output features; ~ N(0, w_sigma), stored as bf16 values), the
    RMSNorm gains (1 + N(0, 0.02), bf16) and the final norm's gain.  The
    weights are the same for every set (they are the model's); x changes."""
    if not w.I:
        raise ValueError(f"workload {w.name} has no layer")
    s = w.seed
    tag = "" if set_index == 0 else f"#{set_index}"
    bf = to_bf16_values
    qd, kd = w.Hq * w.D, w.Hkv * w.D
    out = {"x": normal(s, "layer-x" + tag, (w.T, w.H))}
    for name, shape in (("wq", (qd, w.H)), ("wk", (kd, w.H)), ("wv", (kd, w.H)),
                        ("wo", (w.H, qd)), ("wg", (w.I, w.H)), ("wu", (w.I, w.H)),
                        ("wd", (w.H, w.I))):
        out[name] = bf(normal(s, "layer-" + name, shape, std=w.w_sigma))
    for name in ("g_attn", "g_mlp", "g_final"):
        out[name] = bf(np.float32(1.0) + normal(s, "layer-" + name, (w.H,), std=0.02))
    return out
