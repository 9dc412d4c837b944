"""One tree-verify step on the GPU: device buffers + the launch sequence.

    draft tree   eagle_draft_expand (levels 0..depth-1, then finalize), or
                 eagle_draft_static (EAGLE-1's fixed template), or a
                 caller-given tree (parent/tokens/p_row_of_node)
    attention    eagle_tree_attn
    LM head      eagle_lmhead_softmax (greedy: no [T,V] output; stochastic:
                 writes the logits)
    acceptance   eagle_accept_greedy | eagle_accept_stochastic_logits (which
                 normalises only the rows the walk visits)

Every launch goes through the C ABI on one stream with no host
synchronisation, so `run()` can be captured into a CUDA graph (`capture()`).
Sizes that decide grids (T, max_nodes, max_kv) are known on the host from
the budgets and cache lengths; the kernels read the exact extents from the
device offset arrays.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Sequence

from . import (EPI_ACCUM, EPI_QKV_ROPE, EPI_STORE, EPI_SWIGLU, SAMPLE_NO_REPLACE,
               eagle_accept_greedy, eagle_draft_head_input, eagle_draft_rows, eagle_embed_rows,
               eagle_kv_commit_paged, eagle_loop_advance, eagle_tree_attn_paged,
               eagle_accept_stochastic, eagle_accept_stochastic_logits, eagle_cast_bf16,
               eagle_draft_expand, eagle_draft_expand_all, eagle_draft_pool_bytes,
               eagle_draft_static, eagle_gemm,
               eagle_lmhead_softmax, eagle_lmhead_workspace_bytes, eagle_rmsnorm,
               eagle_tree_attn, eagle_tree_attn_workspace_bytes, eagle_tree_rope_table)


def pack_qkv_weight(wq, wk, wv, Hq: int, Hkv: int, D: int):
    """[Wq; Wk; Wv] in the row order eagle_gemm's QKV_ROPE epilogue reads:
    inside every q and k head, dimension j on row 2j and dimension j + D/2 on
    row 2j + 1 (a weight layout prepared once, when the weights are loaded)."""
    import torch
    half = D // 2
    perm = torch.stack([torch.arange(half), torch.arange(half) + half], dim=1).reshape(-1)

    def pair(w, heads):
        w = w.reshape(heads, D, -1)
        return w[:, perm.to(w.device), :].reshape(heads * D, -1)

    return torch.cat([pair(wq, Hq), pair(wk, Hkv), wv], dim=0).contiguous()


def pack_gate_up_weight(wg, wu):
    """Gate and up projections [I, H] interleaved in groups of 16 rows (16
    gate rows, then the 16 matching up rows), the order eagle_gemm's SWIGLU
    epilogue reads."""
    import torch
    I, H = wg.shape
    if I % 16:
        raise ValueError("the MLP width must be a multiple of 16")
    return torch.stack([wg.reshape(I // 16, 16, H), wu.reshape(I // 16, 16, H)],
                       dim=1).reshape(2 * I, H).contiguous()


@dataclasses.dataclass
class StepShape:
    B: int
    Hq: int
    Hkv: int
    D: int
    H: int
    V: int
    L: Sequence[int]                 # KV-cache length per sequence
    n_nodes: Sequence[int]           # tree nodes per sequence, root included
    rows: int                        # draft-distribution rows (all sequences)
    max_depth: int
    dtype: str = "bf16"              # "bf16" or "f32"
    mode: str = "greedy"             # "greedy" or "stochastic"
    temperature: float = 1.0
    sample_mode: int = SAMPLE_NO_REPLACE
    # EAGLE-2 tree build (k == 0: the caller supplies the tree)
    k: int = 0
    depth: int = 0
    budget: Sequence[int] = ()
    # EAGLE-1 static tree: template (parent, rank, row) lists; k must be 0
    static: tuple = ()
    # the full decoder layer (RMSNorm, Q/K/V + rotary, attention, Wo,
    # RMSNorm, SwiGLU MLP) feeds the attention and the LM head
    layer: bool = False
    I: int = 0
    theta: float = 10000.0
    eps: float = 1e-5
    # paged KV cache: pool of n_pages pages of page_size positions (0: the
    # packed cache of kv_off)
    page_size: int = 0
    n_pages: int = 0
    max_pages: int = 0

    @property
    def builds_tree(self) -> bool:
        return bool(self.k) or bool(self.static)

    @property
    def T(self) -> int:
        return int(sum(self.n_nodes))


class TreeVerifyStep:
    """Owns the device tensors of one step and launches it."""

    def __init__(self, shape: StepShape, device: str = "cuda"):
        import torch
        self.torch = torch
        self.s = shape
        s = shape
        dev = torch.device(device)
        dt = torch.bfloat16 if s.dtype == "bf16" else torch.float32
        i32, f32 = torch.int32, torch.float32
        T, sumL = s.T, int(sum(s.L))
        self.max_nodes = int(max(s.n_nodes))
        self.max_kv = int(max(s.L)) if len(s.L) else 0
        z = lambda *shape_, dtype=f32: torch.zeros(shape_, dtype=dtype, device=dev)
        # Inputs that change every step live in one device buffer (views at
        # 256-byte offsets), so a step's inputs arrive with a single copy.
        if s.layer:
            spec = [("x", (T, s.H), f32)]
        else:
            spec = [("q", (T, s.Hq, s.D), dt), ("k_tree", (T, s.Hkv, s.D), dt),
                    ("v_tree", (T, s.Hkv, s.D), dt), ("h", (T, s.H), dt)]
        spec += [("u_accept", (T,), f32), ("u_sample", (T,), f32)]
        if s.mode == "stochastic":
            spec.append(("p_rows", (max(s.rows, 1), s.V), f32))
        if s.k:
            spec += [("draft_logp", (max(s.rows, 1), s.V), f32), ("budget", (s.B,), i32),
                     ("root_token", (s.B,), i32)]
        elif s.static:
            spec += [("draft_logp", (max(s.rows, 1), s.V), f32), ("root_token", (s.B,), i32)]
        else:
            spec += [("tree_off", (s.B + 1,), i32), ("parent", (T,), i32),
                     ("tokens", (T,), i32), ("p_row_of_node", (T,), i32)]
        offs, total = [], 0
        for _, shp, dty in spec:
            n = 1
            for d in shp:
                n *= d
            offs.append(total)
            total += (n * torch.empty((), dtype=dty).element_size() + 255) // 256 * 256
        self.step_input_names = [n for n, _, _ in spec]
        self.step_inputs = torch.zeros(max(total, 256), dtype=torch.uint8, device=dev)
        for (name, shp, dty), off in zip(spec, offs):
            nb = 1
            for d in shp:
                nb *= d
            nb *= torch.empty((), dtype=dty).element_size()
            setattr(self, name, self.step_inputs[off:off + nb].view(dty).view(shp))
        if s.layer:
            if s.dtype != "bf16":
                raise ValueError("the full layer runs in bf16")
            bf = torch.bfloat16
            # the layer's outputs that the attention and the LM head read
            self.q = z(T, s.Hq, s.D, dtype=bf)
            self.k_tree = z(T, s.Hkv, s.D, dtype=bf)
            self.v_tree = z(T, s.Hkv, s.D, dtype=bf)
            self.h = z(T, s.H, dtype=bf)
            # weights (resident) and work buffers
            qd = s.Hq * s.D
            self.g_attn = z(s.H, dtype=bf)
            self.g_mlp = z(s.H, dtype=bf)
            self.g_final = z(s.H, dtype=bf)
            self.w_qkv = z((s.Hq + 2 * s.Hkv) * s.D, s.H, dtype=bf)
            self.wo = z(s.H, qd, dtype=bf)
            self.w_gu = z(2 * s.I, s.H, dtype=bf)
            self.wd = z(s.H, s.I, dtype=bf)
            self.a = z(T, s.H, dtype=bf)
            self.pos = z(T, dtype=i32)
            self.cos_sin = z(T, s.D // 2, 2)
            self.o_bf = z(T, qd, dtype=bf)
            self.resid = z(T, s.H)
            self.bn = z(T, s.H, dtype=bf)
            self.m = z(T, s.I, dtype=bf)
        # resident inputs
        if s.page_size:
            self.k_pages = z(s.n_pages, s.page_size, s.Hkv, s.D, dtype=dt)
            self.v_pages = z(s.n_pages, s.page_size, s.Hkv, s.D, dtype=dt)
            self.block_table = z(s.B, s.max_pages, dtype=i32)
            self.kv_len = z(s.B, dtype=i32)
            self.max_kv = s.max_pages * s.page_size
        else:
            self.k_cache = z(max(sumL, 1), s.Hkv, s.D, dtype=dt)
            self.v_cache = z(max(sumL, 1), s.Hkv, s.D, dtype=dt)
            self.kv_off = z(s.B + 1, dtype=i32)
        self.w_lm = z(s.V, s.H, dtype=dt)
        if s.mode != "stochastic":
            self.p_rows = z(max(s.rows, 1), s.V)
        if not s.builds_tree:
            self.draft_logp = None
            self.root_token = z(s.B, dtype=i32)
        if not s.k:
            self.budget = z(s.B, dtype=i32)
        self.tmpl = None
        if s.static:
            par, rank, row = s.static
            self.tmpl = [torch.tensor(list(a), dtype=i32, device=dev) for a in (par, rank, row)]
            self.tmpl_max_rank = int(max(list(rank)[1:] or [0])) + 1
        # tree (written by the expand kernels, or loaded)
        if s.builds_tree:
            self.tree_off = z(s.B + 1, dtype=i32)
            self.parent = z(T, dtype=i32)
            self.tokens = z(T, dtype=i32)
            self.p_row_of_node = z(T, dtype=i32)
        self.node_depth = z(T, dtype=i32)
        self.score = z(T)
        self.pool = None
        if s.k:
            nbytes = eagle_draft_pool_bytes(s.B, s.k, s.depth, s.V)
            if nbytes == 0:
                raise ValueError("unsupported EAGLE-2 tree parameters")
            self.pool = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        # outputs / scratch
        self.attn_out = z(T, s.Hq, s.D)
        ws = eagle_tree_attn_workspace_bytes(s.B, T, s.Hq, s.Hkv, s.D, self.max_nodes, self.max_kv)
        self.attn_ws = torch.zeros(max(ws, 16), dtype=torch.uint8, device=dev)
        self.lm_ws = torch.zeros(max(eagle_lmhead_workspace_bytes(T, s.V), 16),
                                 dtype=torch.uint8, device=dev)
        self.argmax = z(T, dtype=i32)
        self.row_max = z(T)
        self.row_lse = z(T)
        self.top2_gap = z(T)
        # stochastic: the target logits; the walk normalises the rows it visits
        self.logits = z(T, s.V) if s.mode == "stochastic" else None
        self._side = None   # second stream of run() (the LM head)
        W = s.max_depth + 1
        self.accept_len = z(s.B, dtype=i32)
        self.accepted_nodes = z(s.B, W, dtype=i32)
        self.out_tokens = z(s.B, W, dtype=i32)
        self.status = z(1, dtype=i32)

    # ------------------------------------------------------------------
    def load(self, arrays: Dict[str, object]) -> None:
        """Copy host arrays (numpy or torch) into the device tensors with the
        same names."""
        torch = self.torch
        for name, val in arrays.items():
            t = getattr(self, name)
            if t is None:
                raise KeyError(f"{name} is not used by this step")
            src = val if isinstance(val, torch.Tensor) else torch.from_numpy(val)
            t.copy_(src.reshape(t.shape).to(t.dtype), non_blocking=False)

    def load_layer(self, arrays: Dict[str, object]) -> None:
        """Copy the layer's weights (standard layouts: wq [Hq*D, H], wk, wv
        [Hkv*D, H], wo [H, Hq*D], wg, wu [I, H], wd [H, I], gains [H]) into
        the device buffers, packing W_qkv and W_gate/up as the GEMM reads
        them."""
        torch = self.torch
        s = self.s
        dev = lambda a: (a if isinstance(a, torch.Tensor) else torch.from_numpy(a)).to(
            device=self.w_qkv.device, dtype=torch.bfloat16)
        for name in ("g_attn", "g_mlp", "g_final", "wo", "wd"):
            getattr(self, name).copy_(dev(arrays[name]).reshape(getattr(self, name).shape))
        self.w_qkv.copy_(pack_qkv_weight(dev(arrays["wq"]), dev(arrays["wk"]), dev(arrays["wv"]),
                                         s.Hq, s.Hkv, s.D))
        self.w_gu.copy_(pack_gate_up_weight(dev(arrays["wg"]), dev(arrays["wu"])))

    def load_paged_cache(self, k, v, lengths: Sequence[int]) -> None:
        """Scatter packed caches k, v [sum L, Hkv, D] (sequence b's rows
        after those of the sequences before it) into the pages its block
        table names, and set kv_len (set-up, not a step)."""
        torch = self.torch
        t = lambda a: a if isinstance(a, torch.Tensor) else torch.from_numpy(a)
        k, v = t(k), t(v)
        table = self.block_table.cpu()
        P = self.s.page_size
        off = 0
        for b, L in enumerate(lengths):
            for j in range((int(L) + P - 1) // P):
                n = min(P, int(L) - j * P)
                page = int(table[b, j])
                self.k_pages[page, :n].copy_(k[off + j * P: off + j * P + n].to(self.k_pages.dtype))
                self.v_pages[page, :n].copy_(v[off + j * P: off + j * P + n].to(self.v_pages.dtype))
            off += int(L)
        self.kv_len.copy_(torch.tensor([int(L) for L in lengths], dtype=torch.int32))

    def assign_pages(self, capacity: Sequence[int]) -> None:
        """A block table giving sequence b the next ceil(capacity[b] /
        page_size) pages of the pool, in order."""
        torch = self.torch
        P = self.s.page_size
        table = torch.full((self.s.B, self.s.max_pages), -1, dtype=torch.int32)
        nxt = 0
        for b, c in enumerate(capacity):
            for j in range((int(c) + P - 1) // P):
                table[b, j] = nxt
                nxt += 1
        if nxt > self.s.n_pages:
            raise ValueError("the page pool is too small")
        self.block_table.copy_(table)

    def host_step_inputs(self, arrays: Dict[str, object]):
        """Pinned host buffer laid out like `step_inputs`, filled from host
        arrays named as the step's inputs: one copy moves a whole step."""
        torch = self.torch
        host = torch.zeros(self.step_inputs.numel(), dtype=torch.uint8).pin_memory()
        base = self.step_inputs.data_ptr()
        for name in self.step_input_names:
            t = getattr(self, name)
            off = t.data_ptr() - base
            nb = t.numel() * t.element_size()
            src = arrays[name]
            src = src if isinstance(src, torch.Tensor) else torch.from_numpy(src)
            host[off:off + nb].view(t.dtype).view(t.shape).copy_(src.reshape(t.shape).to(t.dtype))
        return host

    # ------------------------------------------------------------------
    def run_expand(self, stream=None) -> None:
        s = self.s
        if s.static:
            R = self.draft_logp.shape[0] // s.B
            eagle_draft_static(*self.tmpl, self.draft_logp.view(s.B, R, s.V), self.root_token,
                               self.tree_off, self.parent, self.tokens, self.node_depth,
                               self.score, self.p_row_of_node, self.status,
                               max_rank=self.tmpl_max_rank, stream=stream)
            return
        # every draft row is an input of the step: all levels in one call
        eagle_draft_expand_all(self.pool, self.status, B=s.B, V=s.V, k=s.k, depth=s.depth,
                               draft_logp=self.draft_logp, budget=self.budget,
                               root_token=self.root_token, tree_off=self.tree_off,
                               parent=self.parent, tokens=self.tokens,
                               node_depth=self.node_depth, score=self.score,
                               p_row_of_node=self.p_row_of_node, stream=stream)

    def run_layer(self, stream=None) -> None:
        """The decoder layer over every tree node, ending in the final
        RMSNorm that feeds the LM head (h)."""
        s = self.s
        eagle_rmsnorm(self.x, self.g_attn, self.a, self.status, eps=s.eps, stream=stream)
        cache_len = dict(kv_len=self.kv_len) if s.page_size else dict(kv_off=self.kv_off)
        eagle_tree_rope_table(self.tree_off, self.parent, self.pos, self.cos_sin, self.status,
                              D=s.D, theta=s.theta, stream=stream, **cache_len)
        eagle_gemm(EPI_QKV_ROPE, self.a, self.w_qkv, self.status, q=self.q, k=self.k_tree,
                   v=self.v_tree, cos_sin=self.cos_sin, Hq=s.Hq, Hkv=s.Hkv, D=s.D, stream=stream)
        self.run_attn(stream)
        eagle_cast_bf16(self.attn_out.view(-1), self.o_bf.view(-1), stream=stream)
        eagle_gemm(EPI_ACCUM, self.o_bf, self.wo, self.status, accum=self.resid, resid=self.x,
                   stream=stream)
        eagle_rmsnorm(self.resid, self.g_mlp, self.bn, self.status, eps=s.eps, stream=stream)
        eagle_gemm(EPI_SWIGLU, self.bn, self.w_gu, self.status, y=self.m, stream=stream)
        eagle_gemm(EPI_ACCUM, self.m, self.wd, self.status, accum=self.resid, stream=stream)
        eagle_rmsnorm(self.resid, self.g_final, self.h, self.status, eps=s.eps, stream=stream)

    def run_attn(self, stream=None) -> None:
        if self.s.page_size:
            eagle_tree_attn_paged(self.q, self.k_tree, self.v_tree, self.k_pages, self.v_pages,
                                  self.block_table, self.kv_len, self.tree_off, self.parent,
                                  self.attn_out, self.status, max_nodes=self.max_nodes,
                                  max_kv=self.max_kv, stream=stream)
            return
        eagle_tree_attn(self.q, self.k_tree, self.v_tree, self.k_cache, self.v_cache,
                        self.kv_off, self.tree_off, self.parent, self.attn_out, self.status,
                        max_nodes=self.max_nodes, max_kv=self.max_kv, ws=self.attn_ws,
                        stream=stream)

    def run_lmhead(self, stream=None) -> None:
        eagle_lmhead_softmax(self.h, self.w_lm, self.argmax, self.row_max, self.row_lse,
                             self.top2_gap, self.logits, self.lm_ws, self.status,
                             temperature=self.s.temperature, logits=True, stream=stream)

    def run_accept(self, stream=None) -> None:
        s = self.s
        if s.mode == "greedy":
            eagle_accept_greedy(self.tree_off, self.parent, self.tokens, self.argmax,
                                self.accept_len, self.accepted_nodes, self.out_tokens,
                                self.status, max_nodes=self.max_nodes, max_depth=s.max_depth,
                                stream=stream)
        else:
            eagle_accept_stochastic_logits(self.tree_off, self.parent, self.tokens, self.logits,
                                           self.row_lse, self.p_rows, self.p_row_of_node,
                                           self.u_accept, self.u_sample, self.accept_len,
                                           self.accepted_nodes, self.out_tokens, self.status,
                                           temperature=s.temperature, max_nodes=self.max_nodes,
                                           max_depth=s.max_depth, mode=s.sample_mode,
                                           stream=stream)

    def run_accept_q(self, q, stream=None) -> None:
        """The stochastic walk fed with given probabilities q [T,V] fp32 (a
        device tensor) instead of this step's logits."""
        s = self.s
        eagle_accept_stochastic(self.tree_off, self.parent, self.tokens, q, self.p_rows,
                                self.p_row_of_node, self.u_accept, self.u_sample,
                                self.accept_len, self.accepted_nodes, self.out_tokens,
                                self.status, max_nodes=self.max_nodes, max_depth=s.max_depth,
                                mode=s.sample_mode, stream=stream)

    def run(self, stream=None, build_tree: bool = True) -> None:
        """The whole step: tree build (if EAGLE-2), attention, LM head, accept.
        build_tree=False verifies the tree already in the buffers.

        The LM head needs neither the tree nor the attention output, so it
        runs on a second stream, forked after everything queued so far and
        joined before the acceptance walk: its weight stream overlaps the
        latency-bound tree build (whose CTAs fit beside the LM head's on the
        same SMs) and the attention."""
        torch = self.torch
        main = stream if stream is not None else torch.cuda.current_stream()
        if self.s.layer:
            # the LM head reads the layer's output: one stream, in order
            if self.s.builds_tree and build_tree:
                self.run_expand(main)
            self.run_layer(main)
            self.run_lmhead(main)
            self.run_accept(main)
            return
        if self._side is None:
            self._side = torch.cuda.Stream(device=main.device)
        side = self._side
        side.wait_stream(main)
        self.run_lmhead(side)
        if self.s.builds_tree and build_tree:
            self.run_expand(main)
        self.run_attn(main)
        main.wait_stream(side)
        self.run_accept(main)

    def launches_per_step(self) -> int:
        """Kernels launched by run() (the count the benchmark reports)."""
        n = 0
        if self.s.k:
            # all levels' chunks, then every merge and the finalize (or one
            # merge launch per level and the finalize when the finalize's
            # shared memory is too large), for rows of a multiple of 4
            # entries; else one per level, finalize fused
            k, d = self.s.k, self.s.depth
            fin_smem = (k + (d - 1) * k * k) * 44
            if self.s.V % 4 == 0:
                n += 2 if fin_smem <= 160 * 1024 else d + 2
            else:
                n += d
        elif self.s.static:
            n += 2 if len(self.s.static[0]) > 1 else 1   # ranks + finish
        n += 1                                   # attention
        if self.s.layer:                         # norms, rope table, 4 GEMMs (+ one
            tiles = (self.s.T + 127) // 128      # per extra cluster pass), cast
            n += 3 + 1 + 4 * ((tiles + 7) // 8) + 1
        if self.s.dtype == "bf16":               # LM head: one launch per cluster of
            tiles = (self.s.T + 127) // 128      # up to eight 128-row tiles
            n += (tiles + 7) // 8 + 1            # ... + finalize
        else:
            n += 2                               # LM head tiles + finalize
        n += 1                                   # acceptance
        return n

    def capture(self, stream=None, build_tree: bool = True):
        """Capture run() into a CUDA graph (after one eager warm-up)."""
        torch = self.torch
        st = torch.cuda.Stream() if stream is None else stream
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(st):
            self.run(build_tree=build_tree)
        torch.cuda.current_stream().wait_stream(st)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            self.run(build_tree=build_tree)
        torch.cuda.synchronize()
        return g


@dataclasses.dataclass
class LoopShape:
    """Sizes of a draft -> verify -> accept -> commit loop (greedy or
    stochastic acceptance) over B sequences with paged KV caches."""
    B: int
    Hq: int
    Hkv: int
    D: int
    H: int
    I: int
    V: int
    k: int                           # EAGLE-2 top-k per expanded node
    depth: int                       # EAGLE-2 levels
    budget: Sequence[int]            # draft-token budget per sequence
    L0: Sequence[int]                # cache length per sequence at the start
    steps: int                       # steps the page tables are sized for
    page_size: int = 128
    theta: float = 10000.0
    eps: float = 1e-5
    mode: str = "greedy"
    temperature: float = 1.0


class SpeculativeLoop:
    """The steps on either side of the verify pass, on the GPU.

    Per step: the EAGLE-2 tree is drafted level by level (draft head input
    rows, the head's one matrix, the frozen LM head in logits mode, the
    level's draft rows, the expand level that reads them); the target's one
    decoder layer verifies the tree over the paged cache, the LM head and
    the acceptance walk follow; the root and accepted nodes' K/V are
    committed to the cache and the bonus token becomes the next root.
    Everything is queued on one stream without host synchronisation.

    The draft head is deliberately small: f' = [f ; e] Wd^T (f the parent's
    feature, e the embedding of the node's token, Wd [H, 2H]); the root's
    parent feature is the target's output at the last accepted node."""

    def __init__(self, shape: LoopShape, device: str = "cuda"):
        import torch
        self.torch = torch
        s = self.s = shape
        dev = torch.device(device)
        bf, f32, i32 = torch.bfloat16, torch.float32, torch.int32
        z = lambda *shp, dtype=f32: torch.zeros(shp, dtype=dtype, device=dev)
        n_nodes = [min(int(b), s.k + (s.depth - 1) * s.k * s.k) + 1 for b in s.budget]
        cap = [(int(L) + s.steps * (s.depth + 1) + s.page_size - 1) // s.page_size
               for L in s.L0]
        self.max_pages = max(cap)
        self.n_pages = sum(cap)
        self.step = TreeVerifyStep(StepShape(
            B=s.B, Hq=s.Hq, Hkv=s.Hkv, D=s.D, H=s.H, V=s.V, L=list(s.L0), n_nodes=n_nodes,
            rows=s.B * (1 + (s.depth - 1) * s.k), max_depth=s.depth, dtype="bf16", mode=s.mode,
            temperature=s.temperature, k=s.k, depth=s.depth, budget=list(s.budget), layer=True,
            I=s.I, theta=s.theta, eps=s.eps, page_size=s.page_size, n_pages=self.n_pages,
            max_pages=self.max_pages), device=device)
        st = self.step
        # a fixed page assignment for the whole run (every sequence owns the
        # pages its longest possible context needs)
        st.assign_pages([c * s.page_size for c in cap])
        # model state and draft-loop buffers
        self.emb = z(s.V, s.H, dtype=bf)            # shared token embedding
        self.w_draft = z(s.H, 2 * s.H, dtype=bf)     # the draft head
        self.f_ctx = z(s.B, s.H, dtype=bf)           # context feature per sequence
        self.a_draft = z(s.B * s.k, 2 * s.H, dtype=bf)
        self.feat = [z(s.B * s.k, s.H, dtype=bf) for _ in range(2)]
        self.nodes = [z(s.B * s.k, dtype=i32) for _ in range(2)]
        self.z_draft = z(s.B * s.k, s.V)
        self.d_argmax = z(s.B * s.k, dtype=i32)
        self.d_stats = [z(s.B * s.k) for _ in range(3)]
        self.d_ws = z(max(eagle_lmhead_workspace_bytes(s.B * s.k, s.V), 16), dtype=torch.uint8)
        if st.draft_logp is None:
            raise ValueError("the loop builds its tree")

    def load(self, arrays: Dict[str, object], kv: Dict[str, object]) -> None:
        """Weights (layer weights as TreeVerifyStep.load_layer, w_lm, emb,
        w_draft), the initial context feature f_ctx, root tokens, and the
        initial caches kv["k"], kv["v"] as packed [sum L0, Hkv, D] rows with
        their lengths L0."""
        torch = self.torch
        st = self.step
        st.load_layer(arrays)
        t = lambda a: a if isinstance(a, torch.Tensor) else torch.from_numpy(a)
        st.w_lm.copy_(t(arrays["w_lm"]).to(st.w_lm.dtype))
        self.emb.copy_(t(arrays["emb"]).to(self.emb.dtype))
        self.w_draft.copy_(t(arrays["w_draft"]).to(self.w_draft.dtype))
        self.f_ctx.copy_(t(arrays["f_ctx"]).to(self.f_ctx.dtype))
        st.root_token.copy_(t(arrays["root_token"]).to(torch.int32))
        st.budget.copy_(torch.tensor(list(self.s.budget), dtype=torch.int32))
        # scatter the initial caches into the pages (set-up, not a step)
        st.load_paged_cache(kv["k"], kv["v"], self.s.L0)

    def run_draft(self, stream=None) -> None:
        s, st = self.s, self.step
        R = 1 + (s.depth - 1) * s.k
        logp = st.draft_logp.view(s.B, R, s.V)
        prob = st.p_rows.view(s.B, R, s.V) if s.mode == "stochastic" else None
        for lev in range(s.depth):
            F = 1 if lev == 0 else s.k
            cur, prev = lev % 2, (lev - 1) % 2
            eagle_draft_head_input(st.pool, self.nodes[cur], self.f_ctx, st.root_token, self.emb,
                                   self.a_draft, st.status, B=s.B, V=s.V, k=s.k, depth=s.depth,
                                   level=lev, node_prev=self.nodes[prev],
                                   feat_prev=self.feat[prev], stream=stream)
            feat = self.feat[cur][:s.B * F]
            eagle_gemm(EPI_STORE, self.a_draft[:s.B * F], self.w_draft, st.status, y=feat,
                       stream=stream)
            eagle_lmhead_softmax(feat, st.w_lm, self.d_argmax[:s.B * F],
                                 self.d_stats[0][:s.B * F], self.d_stats[1][:s.B * F],
                                 self.d_stats[2][:s.B * F], self.z_draft[:s.B * F], self.d_ws,
                                 st.status, temperature=1.0, logits=True, stream=stream)
            eagle_draft_rows(self.z_draft[:s.B * F], self.d_stats[1][:s.B * F], logp, prob,
                             B=s.B, k=s.k, depth=s.depth, level=lev, stream=stream)
            last = lev == s.depth - 1
            eagle_draft_expand(st.pool, st.status, B=s.B, V=s.V, k=s.k, depth=s.depth, level=lev,
                               finalize=2 if last else 0, draft_logp=st.draft_logp,
                               budget=st.budget if last else None,
                               root_token=st.root_token if last else None,
                               tree_off=st.tree_off if last else None,
                               parent=st.parent if last else None,
                               tokens=st.tokens if last else None,
                               node_depth=st.node_depth if last else None,
                               score=st.score if last else None,
                               p_row_of_node=st.p_row_of_node if last else None,
                               rows_from_previous_kernel=True, stream=stream)

    def run_verify(self, stream=None) -> None:
        st = self.step
        eagle_embed_rows(st.tokens, self.emb, st.x, st.status, stream=stream)
        st.run_layer(stream)
        st.run_lmhead(stream)
        st.run_accept(stream)

    def run_commit(self, stream=None) -> None:
        s, st = self.s, self.step
        eagle_kv_commit_paged(st.tree_off, st.accept_len, st.accepted_nodes, st.k_tree, st.v_tree,
                              st.k_pages, st.v_pages, st.block_table, st.kv_len, st.status,
                              max_depth=s.depth, stream=stream)
        eagle_loop_advance(st.tree_off, st.accept_len, st.accepted_nodes, st.out_tokens, st.resid,
                           self.f_ctx, st.root_token, st.status, max_depth=s.depth,
                           stream=stream)

    def run(self, stream=None) -> None:
        """One whole step: draft, verify, accept, commit."""
        self.run_draft(stream)
        self.run_verify(stream)
        self.run_commit(stream)
