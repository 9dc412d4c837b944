"""Python binding of libeagle.so, the GB300 (sm_103a) tree-verify library.

Argument marshalling only: every function here checks tensor devices, dtypes
and shapes, derives the sizes the C ABI wants, and calls the C entry point of
the same name on the current CUDA stream.  Every step of the computation runs
in the library's CUDA kernels; there is no fallback.  If the shared library
has not been built (see `build()`), the first call raises.

Tensors are torch CUDA tensors (PyTorch is used for device memory and streams
only).  Outputs are written in place into the tensors the caller passes.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "EagleError", "build", "lib", "status_string", "version", "check_status",
    "EAGLE_F32", "EAGLE_BF16", "LMHEAD_GREEDY", "LMHEAD_PROB", "LMHEAD_LOGITS", "SAMPLE_REPLACE",
    "SAMPLE_NO_REPLACE", "eagle_tree_attn", "eagle_tree_attn_workspace_bytes",
    "eagle_lmhead_softmax", "eagle_lmhead_workspace_bytes", "eagle_accept_greedy",
    "eagle_accept_stochastic", "eagle_accept_stochastic_logits", "eagle_draft_expand",
    "eagle_draft_pool_bytes", "eagle_draft_static", "eagle_tree_attn_paged",
    "eagle_rmsnorm", "eagle_cast_bf16", "eagle_tree_rope_table", "eagle_gemm",
    "eagle_kv_commit_paged", "eagle_draft_expand_dep", "eagle_draft_expand_all",
    "eagle_draft_head_input",
    "eagle_draft_rows", "eagle_embed_rows", "eagle_loop_advance",
    "EPI_STORE", "EPI_ACCUM", "EPI_SWIGLU", "EPI_QKV_ROPE",
    "eagle_lmhead_softmax_noalloc", "eagle_lmhead_noalloc_max_scratch_bytes",
]

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libeagle.so")

EAGLE_F32, EAGLE_BF16 = 0, 1
LMHEAD_GREEDY, LMHEAD_PROB, LMHEAD_LOGITS = 0, 1, 2
SAMPLE_REPLACE, SAMPLE_NO_REPLACE = 0, 1
EPI_STORE, EPI_ACCUM, EPI_SWIGLU, EPI_QKV_ROPE = 0, 1, 2, 3

_STATUS = {0: "ok", 1: "invalid argument", 2: "invalid tree", 3: "unsupported shape",
           4: "numeric error", 5: "device wait timed out", 6: "CUDA error",
           7: "workspace too small"}


class EagleError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn}: {_STATUS.get(code, 'unknown')} (status {code})")
        self.code = code


_lib = None
_i, _f, _p, _sz = ctypes.c_int, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t
_SIGS = {
    "eagle_status_string": ([_i], ctypes.c_char_p),
    "eagle_version": ([], ctypes.c_char_p),
    "eagle_tree_attn_workspace_bytes": ([_i] * 7, _sz),
    "eagle_tree_attn": ([_i, _i, _i, _i, _i, _i, _f, _i, _i, _i] + [_p] * 9 + [_p, _sz, _p, _p],
                        _i),
    "eagle_lmhead_workspace_bytes": ([_i, _i], _sz),
    "eagle_lmhead_softmax": ([_i, _i, _i, _i, _f, _i] + [_p] * 8 + [_sz, _p, _p], _i),
    "eagle_accept_greedy": ([_i, _i, _p, _p, _p, _p, _i, _p, _p, _p, _p, _p], _i),
    "eagle_accept_stochastic": ([_i] * 5 + [_p] * 8 + [_i] + [_p] * 5, _i),
    "eagle_accept_stochastic_logits": ([_i] * 5 + [_p] * 5 + [_f] + [_p] * 4 + [_i] + [_p] * 5,
                                       _i),
    "eagle_draft_pool_bytes": ([_i] * 4, _sz),
    "eagle_lmhead_noalloc_max_scratch_bytes": ([], _sz),
    "eagle_lmhead_softmax_noalloc": ([_i, _i, _i, _i, _f, _i] + [_p] * 9, _i),
    "eagle_draft_expand": ([_i] * 6 + [_p] * 4 + [_sz] + [_p] * 8, _i),
    "eagle_draft_static": ([_i] * 5 + [_p] * 12 + [_p], _i),
    "eagle_tree_attn_paged": ([_i] * 6 + [_f] + [_i] * 5 + [_p] * 12, _i),
    "eagle_rmsnorm": ([_i, _i, _f] + [_p] * 5, _i),
    "eagle_cast_bf16": ([_sz, _p, _p, _p], _i),
    "eagle_tree_rope_table": ([_i, _i, _i, _f] + [_p] * 8, _i),
    "eagle_gemm": ([_i] * 4 + [_p] * 9 + [_i] * 3 + [_p, _p], _i),
    "eagle_kv_commit_paged": ([_i] * 8 + [_p] * 11, _i),
    "eagle_draft_expand_dep": ([_i] * 6 + [_p] * 4 + [_sz] + [_p] * 8, _i),
    "eagle_draft_expand_all": ([_i] * 4 + [_p] * 4 + [_sz] + [_p] * 8, _i),
    "eagle_draft_head_input": ([_i] * 6 + [_p, _sz] + [_p] * 9, _i),
    "eagle_draft_rows": ([_i] * 5 + [_p] * 5, _i),
    "eagle_embed_rows": ([_i] * 3 + [_p] * 5, _i),
    "eagle_loop_advance": ([_i] * 3 + [_p] * 9, _i),
}


def build(verbose: bool = False, force: bool = False) -> str:
    """Compile the CUDA sources into libeagle.so (sm_103a) and return its path."""
    from . import _build
    return _build.build(verbose=verbose, force=force)


def lib() -> ctypes.CDLL:
    """The loaded shared library (raises if it was never built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build the CUDA library first "
                "(eagle_tree_verification_gb300.build())")
        L = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGS.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = res
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().eagle_status_string(int(code)).decode()


def version() -> str:
    return lib().eagle_version().decode()


def check_status(status_tensor, fn: str = "device") -> None:
    """Raise EagleError if a device status word is non-zero (synchronises)."""
    code = int(status_tensor.view(-1)[0].item())
    if code != 0:
        raise EagleError(fn, code)


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return EAGLE_BF16
    if t.dtype == torch.float32:
        return EAGLE_F32
    raise ValueError(f"unsupported dtype {t.dtype}")


def _need(t, dtype, name):
    if t is not None and t.dtype != dtype:
        raise ValueError(f"{name}: expected {dtype}, got {t.dtype}")


def _stream(stream) -> int:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _call(name, *args):
    rc = getattr(lib(), name)(*args)
    if rc != 0:
        raise EagleError(name, rc)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def eagle_tree_attn_workspace_bytes(B, T, Hq, Hkv, D, max_nodes, max_kv) -> int:
    return int(lib().eagle_tree_attn_workspace_bytes(B, T, Hq, Hkv, D, max_nodes, max_kv))


def eagle_tree_attn(q, k_tree, v_tree, k_cache, v_cache, kv_off, tree_off, parent, out,
                    status, *, max_nodes: int, max_kv: int, scale: Optional[float] = None,
                    ws=None, stream=None) -> None:
    """Tree-masked attention; see eagle_tree_attn in include/eagle.h.
    q [T,Hq,D]; k_tree/v_tree [T,Hkv,D]; k_cache/v_cache [sum L,Hkv,D];
    kv_off/tree_off [B+1] int32; parent [T] int32; out [T,Hq,D] fp32."""
    torch = _torch()
    T, Hq, D = q.shape
    Hkv = k_tree.shape[1]
    B = tree_off.numel() - 1
    for name, t in (("k_tree", k_tree), ("v_tree", v_tree), ("k_cache", k_cache),
                    ("v_cache", v_cache)):
        _need(t, q.dtype, name)
    for name, t in (("kv_off", kv_off), ("tree_off", tree_off), ("parent", parent)):
        _need(t, torch.int32, name)
    _need(out, torch.float32, "out")
    ws_bytes = 0 if ws is None else ws.numel() * ws.element_size()
    sc = (1.0 / D ** 0.5) if scale is None else float(scale)
    _call("eagle_tree_attn", _dtype_code(q), B, T, Hq, Hkv, D, sc, max_nodes, max_kv,
          k_cache.shape[0],
          _ptr(q), _ptr(k_tree), _ptr(v_tree), _ptr(k_cache), _ptr(v_cache), _ptr(kv_off),
          _ptr(tree_off), _ptr(parent), _ptr(out), _ptr(ws), ws_bytes,
          _ptr(status), _stream(stream))


def eagle_lmhead_workspace_bytes(T, V) -> int:
    return int(lib().eagle_lmhead_workspace_bytes(T, V))


def eagle_lmhead_softmax(h, w, argmax, row_max, row_lse, top2_gap, q, ws, status, *,
                         temperature: float = 1.0, logits: bool = False, stream=None) -> None:
    """LM head + softmax statistics + argmax; q=None selects greedy mode
    (no [T,V] output).  h [T,H]; w [V,H]; argmax [T] int32; row_max,
    row_lse, top2_gap [T] fp32; q [T,V] fp32 or None.  logits=True stores
    the logits in q instead of the probabilities (for
    eagle_accept_stochastic_logits)."""
    torch = _torch()
    T, H = h.shape
    V = w.shape[0]
    _need(w, h.dtype, "w")
    _need(argmax, torch.int32, "argmax")
    for name, t in (("row_max", row_max), ("row_lse", row_lse), ("top2_gap", top2_gap), ("q", q)):
        _need(t, torch.float32, name)
    mode = LMHEAD_GREEDY if q is None else (LMHEAD_LOGITS if logits else LMHEAD_PROB)
    _call("eagle_lmhead_softmax", _dtype_code(h), T, H, V, float(temperature), mode, _ptr(h),
          _ptr(w), _ptr(argmax), _ptr(row_max), _ptr(row_lse), _ptr(top2_gap), _ptr(q),
          _ptr(ws), ws.numel() * ws.element_size(), _ptr(status), _stream(stream))


def eagle_lmhead_noalloc_max_scratch_bytes() -> int:
    return int(lib().eagle_lmhead_noalloc_max_scratch_bytes())


def eagle_lmhead_softmax_noalloc(h, w, argmax, row_max, row_lse, top2_gap, q, status, *,
                                 temperature: float = 1.0, logits: bool = False,
                                 stream=None) -> None:
    """eagle_lmhead_softmax without a workspace: for callers that cannot
    allocate scratch memory (see include/eagle.h).  Its scratch is a fixed
    16 MiB array inside the library, shared by every call; calls that may
    overlap on the GPU race on it."""
    torch = _torch()
    T, H = h.shape
    V = w.shape[0]
    _need(w, h.dtype, "w")
    _need(argmax, torch.int32, "argmax")
    for name, t in (("row_max", row_max), ("row_lse", row_lse), ("top2_gap", top2_gap), ("q", q)):
        _need(t, torch.float32, name)
    mode = LMHEAD_GREEDY if q is None else (LMHEAD_LOGITS if logits else LMHEAD_PROB)
    _call("eagle_lmhead_softmax_noalloc", _dtype_code(h), T, H, V, float(temperature), mode,
          _ptr(h), _ptr(w), _ptr(argmax), _ptr(row_max), _ptr(row_lse), _ptr(top2_gap), _ptr(q),
          _ptr(status), _stream(stream))


def eagle_accept_greedy(tree_off, parent, tokens, argmax, accept_len, accepted_nodes,
                        out_tokens, status, *, max_nodes: int, max_depth: int,
                        stream=None) -> None:
    """Greedy tree walk.  accepted_nodes/out_tokens [B, max_depth+1] int32."""
    torch = _torch()
    B = tree_off.numel() - 1
    for name, t in (("tree_off", tree_off), ("parent", parent), ("tokens", tokens),
                    ("argmax", argmax), ("accept_len", accept_len),
                    ("accepted_nodes", accepted_nodes), ("out_tokens", out_tokens)):
        _need(t, torch.int32, name)
    if accepted_nodes.numel() < B * (max_depth + 1) or out_tokens.numel() < B * (max_depth + 1):
        raise ValueError("output rows must hold max_depth+1 entries per sequence")
    _call("eagle_accept_greedy", B, max_nodes, _ptr(tree_off), _ptr(parent), _ptr(tokens),
          _ptr(argmax), max_depth, _ptr(accept_len), _ptr(accepted_nodes), _ptr(out_tokens),
          _ptr(status), _stream(stream))


def eagle_accept_stochastic(tree_off, parent, tokens, q, p_rows, p_row_of_node, u_accept,
                            u_sample, accept_len, accepted_nodes, out_tokens, status, *,
                            max_nodes: int, max_depth: int, mode: int = SAMPLE_NO_REPLACE,
                            stream=None) -> None:
    """Multi-round stochastic walk.  q [T,V] fp32; p_rows [R,V] fp32."""
    torch = _torch()
    B = tree_off.numel() - 1
    V = q.shape[1]
    R = p_rows.shape[0]
    for name, t in (("q", q), ("p_rows", p_rows), ("u_accept", u_accept),
                    ("u_sample", u_sample)):
        _need(t, torch.float32, name)
    if p_rows.shape[1] != V:
        raise ValueError("p_rows and q must have the same vocabulary")
    if accepted_nodes.numel() < B * (max_depth + 1) or out_tokens.numel() < B * (max_depth + 1):
        raise ValueError("output rows must hold max_depth+1 entries per sequence")
    _call("eagle_accept_stochastic", B, max_nodes, V, R, int(mode), _ptr(tree_off), _ptr(parent),
          _ptr(tokens), _ptr(q), _ptr(p_rows), _ptr(p_row_of_node), _ptr(u_accept),
          _ptr(u_sample), max_depth, _ptr(accept_len), _ptr(accepted_nodes), _ptr(out_tokens),
          _ptr(status), _stream(stream))


def eagle_accept_stochastic_logits(tree_off, parent, tokens, z, row_lse, p_rows, p_row_of_node,
                                   u_accept, u_sample, accept_len, accepted_nodes, out_tokens,
                                   status, *, temperature: float, max_nodes: int,
                                   max_depth: int, mode: int = SAMPLE_NO_REPLACE,
                                   stream=None) -> None:
    """Multi-round stochastic walk on logits: z [T,V] fp32 and row_lse [T]
    fp32 from eagle_lmhead_softmax(logits=True) at the same temperature."""
    torch = _torch()
    B = tree_off.numel() - 1
    V = z.shape[1]
    R = p_rows.shape[0]
    for name, t in (("z", z), ("row_lse", row_lse), ("p_rows", p_rows),
                    ("u_accept", u_accept), ("u_sample", u_sample)):
        _need(t, torch.float32, name)
    if p_rows.shape[1] != V:
        raise ValueError("p_rows and z must have the same vocabulary")
    if accepted_nodes.numel() < B * (max_depth + 1) or out_tokens.numel() < B * (max_depth + 1):
        raise ValueError("output rows must hold max_depth+1 entries per sequence")
    _call("eagle_accept_stochastic_logits", B, max_nodes, V, R, int(mode), _ptr(tree_off),
          _ptr(parent), _ptr(tokens), _ptr(z), _ptr(row_lse), float(temperature), _ptr(p_rows),
          _ptr(p_row_of_node), _ptr(u_accept), _ptr(u_sample), max_depth, _ptr(accept_len),
          _ptr(accepted_nodes), _ptr(out_tokens), _ptr(status), _stream(stream))


def eagle_draft_pool_bytes(B, k, depth, V) -> int:
    return int(lib().eagle_draft_pool_bytes(B, k, depth, V))


def eagle_draft_expand(pool, status, *, B: int, V: int, k: int, depth: int, level: int = 0,
                       finalize: int = 0, draft_logp=None, budget=None, root_token=None,
                       tree_off=None, parent=None, tokens=None, node_depth=None, score=None,
                       p_row_of_node=None, rows_from_previous_kernel: bool = False,
                       stream=None) -> None:
    """EAGLE-2 expand (one level), finalize (finalize=1), or the last level
    with the finalize fused in (finalize=2); draft_logp [B, R, V] fp32 with
    R = 1 + (depth-1)*k.  rows_from_previous_kernel selects
    eagle_draft_expand_dep (rows written by the kernel just before)."""
    name = "eagle_draft_expand_dep" if rows_from_previous_kernel else "eagle_draft_expand"
    _call(name, B, V, k, depth, int(level), int(finalize),
          _ptr(draft_logp), _ptr(budget), _ptr(root_token), _ptr(pool),
          pool.numel() * pool.element_size(), _ptr(tree_off), _ptr(parent), _ptr(tokens),
          _ptr(node_depth), _ptr(score), _ptr(p_row_of_node), _ptr(status), _stream(stream))


def eagle_draft_expand_all(pool, status, *, B: int, V: int, k: int, depth: int, draft_logp,
                           budget, root_token, tree_off, parent, tokens, node_depth, score,
                           p_row_of_node, stream=None) -> None:
    """EAGLE-2 tree build in one call (every level, then the finalize);
    draft_logp [B, R, V] fp32 with R = 1 + (depth-1)*k, all rows ready."""
    _call("eagle_draft_expand_all", B, V, k, depth, _ptr(draft_logp), _ptr(budget),
          _ptr(root_token), _ptr(pool), pool.numel() * pool.element_size(), _ptr(tree_off),
          _ptr(parent), _ptr(tokens), _ptr(node_depth), _ptr(score), _ptr(p_row_of_node),
          _ptr(status), _stream(stream))


def eagle_draft_static(tmpl_parent, tmpl_rank, tmpl_row, draft_logp, root_token, tree_off,
                       parent, tokens, node_depth, score, p_row_of_node, status, *,
                       max_rank: int, stream=None) -> None:
    """EAGLE-1 static tree from a fixed template (int32 device tensors of N
    entries); draft_logp [B, R, V] fp32; outputs [B*N] (tree_off [B+1])."""
    torch = _torch()
    B, R, V = draft_logp.shape
    N = tmpl_parent.numel()
    for name, t in (("tmpl_parent", tmpl_parent), ("tmpl_rank", tmpl_rank),
                    ("tmpl_row", tmpl_row), ("root_token", root_token), ("tree_off", tree_off),
                    ("parent", parent), ("tokens", tokens), ("node_depth", node_depth),
                    ("p_row_of_node", p_row_of_node)):
        _need(t, torch.int32, name)
    _need(draft_logp, torch.float32, "draft_logp")
    _need(score, torch.float32, "score")
    if parent.numel() < B * N or tree_off.numel() < B + 1:
        raise ValueError("tree outputs must hold B*N nodes")
    _call("eagle_draft_static", B, V, N, R, int(max_rank), _ptr(tmpl_parent), _ptr(tmpl_rank),
          _ptr(tmpl_row), _ptr(draft_logp), _ptr(root_token), _ptr(tree_off), _ptr(parent),
          _ptr(tokens), _ptr(node_depth), _ptr(score), _ptr(p_row_of_node), _ptr(status),
          _stream(stream))


def eagle_tree_attn_paged(q, k_tree, v_tree, k_pages, v_pages, block_table, kv_len, tree_off,
                          parent, out, status, *, max_nodes: int, max_kv: int,
                          scale: Optional[float] = None, stream=None) -> None:
    """Tree attention over a paged KV cache; see eagle_tree_attn_paged in
    include/eagle.h.  k_pages/v_pages [n_pages, page_size, Hkv, D];
    block_table [B, max_pages] int32; kv_len [B] int32."""
    torch = _torch()
    T, Hq, D = q.shape
    Hkv = k_tree.shape[1]
    B = tree_off.numel() - 1
    n_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    max_pages = block_table.shape[1] if block_table.dim() == 2 else 0
    for name, t in (("k_tree", k_tree), ("v_tree", v_tree), ("k_pages", k_pages),
                    ("v_pages", v_pages)):
        _need(t, q.dtype, name)
    for name, t in (("block_table", block_table), ("kv_len", kv_len), ("tree_off", tree_off),
                    ("parent", parent)):
        _need(t, torch.int32, name)
    _need(out, torch.float32, "out")
    if block_table.shape[0] != B or kv_len.numel() != B:
        raise ValueError("block_table and kv_len need one row / entry per sequence")
    sc = (1.0 / D ** 0.5) if scale is None else float(scale)
    _call("eagle_tree_attn_paged", _dtype_code(q), B, T, Hq, Hkv, D, sc, max_nodes, max_kv,
          page_size, n_pages, max_pages, _ptr(q), _ptr(k_tree), _ptr(v_tree), _ptr(k_pages),
          _ptr(v_pages), _ptr(block_table), _ptr(kv_len), _ptr(tree_off), _ptr(parent), _ptr(out),
          _ptr(status), _stream(stream))


def eagle_rmsnorm(x, gain, y, status, *, eps: float, stream=None) -> None:
    """y [T,H] bf16 = rmsnorm(x [T,H] fp32) * gain [H] bf16."""
    torch = _torch()
    T, H = x.shape
    _need(x, torch.float32, "x")
    _need(gain, torch.bfloat16, "gain")
    _need(y, torch.bfloat16, "y")
    _call("eagle_rmsnorm", T, H, float(eps), _ptr(x), _ptr(gain), _ptr(y), _ptr(status),
          _stream(stream))


def eagle_cast_bf16(x, y, stream=None) -> None:
    """y = bf16(x) elementwise (x fp32, y bf16, same number of elements)."""
    torch = _torch()
    _need(x, torch.float32, "x")
    _need(y, torch.bfloat16, "y")
    if x.numel() != y.numel():
        raise ValueError("x and y differ in size")
    _call("eagle_cast_bf16", x.numel(), _ptr(x), _ptr(y), _stream(stream))


def eagle_tree_rope_table(tree_off, parent, pos, cos_sin, status, *, D: int, theta: float,
                          kv_off=None, kv_len=None, stream=None) -> None:
    """Node positions (cache length + depth) and their rotation table
    cos_sin [T, D/2, 2] fp32; give kv_off [B+1] or kv_len [B]."""
    B = tree_off.numel() - 1
    _call("eagle_tree_rope_table", B, parent.numel(), int(D), float(theta), _ptr(tree_off),
          _ptr(parent),
          _ptr(kv_off), _ptr(kv_len), _ptr(pos), _ptr(cos_sin), _ptr(status), _stream(stream))


def eagle_gemm(epilogue, a, w, status, *, y=None, accum=None, resid=None, q=None, k=None, v=None,
               cos_sin=None, Hq: int = 0, Hkv: int = 0, D: int = 0, stream=None) -> None:
    """Y = a [T,K] bf16 x w [N,K]^T bf16 with a layer epilogue (see
    eagle_gemm in include/eagle.h)."""
    torch = _torch()
    T, K = a.shape
    N = w.shape[0]
    _need(a, torch.bfloat16, "a")
    _need(w, torch.bfloat16, "w")
    _call("eagle_gemm", int(epilogue), T, N, K, _ptr(a), _ptr(w), _ptr(y), _ptr(accum),
          _ptr(resid), _ptr(q), _ptr(k), _ptr(v), _ptr(cos_sin), int(Hq), int(Hkv), int(D),
          _ptr(status), _stream(stream))


def eagle_kv_commit_paged(tree_off, accept_len, accepted_nodes, k_tree, v_tree, k_pages, v_pages,
                          block_table, kv_len, status, *, max_depth: int, stream=None) -> None:
    """Append the root and accepted nodes' K/V rows (k_tree/v_tree [T,Hkv,D])
    to the paged cache (k_pages/v_pages [n_pages, page_size, Hkv, D]) and
    advance kv_len [B] in place; accepted_nodes [B, max_depth+1]."""
    torch = _torch()
    B = tree_off.numel() - 1
    T, Hkv, D = k_tree.shape
    n_pages, page_size = k_pages.shape[0], k_pages.shape[1]
    for name, t in (("v_tree", v_tree), ("k_pages", k_pages), ("v_pages", v_pages)):
        _need(t, k_tree.dtype, name)
    for name, t in (("tree_off", tree_off), ("accept_len", accept_len),
                    ("accepted_nodes", accepted_nodes), ("block_table", block_table),
                    ("kv_len", kv_len)):
        _need(t, torch.int32, name)
    if accepted_nodes.numel() < B * (max_depth + 1):
        raise ValueError("accepted_nodes must hold max_depth+1 entries per sequence")
    _call("eagle_kv_commit_paged", _dtype_code(k_tree), B, Hkv, D, page_size, n_pages,
          block_table.shape[1], int(max_depth), _ptr(tree_off), _ptr(accept_len),
          _ptr(accepted_nodes), _ptr(k_tree), _ptr(v_tree), _ptr(k_pages), _ptr(v_pages),
          _ptr(block_table), _ptr(kv_len), _ptr(status), _stream(stream))


def eagle_draft_head_input(pool, node_cur, f_ctx, root_token, emb, a, status, *, B: int, V: int,
                           k: int, depth: int, level: int, node_prev=None, feat_prev=None,
                           stream=None) -> None:
    """Draft-head input rows [B*F, 2H] bf16 for one EAGLE-2 level (see
    include/eagle.h)."""
    H = emb.shape[1]
    _call("eagle_draft_head_input", B, V, k, depth, int(level), H, _ptr(pool),
          pool.numel() * pool.element_size(), _ptr(node_prev), _ptr(node_cur), _ptr(feat_prev),
          _ptr(f_ctx), _ptr(root_token), _ptr(emb), _ptr(a), _ptr(status), _stream(stream))


def eagle_draft_rows(z, lse, logp, prob, *, B: int, k: int, depth: int, level: int,
                     stream=None) -> None:
    """The level's draft rows (log-probs, and probabilities if prob is
    given) from the LM head's logits of its draft nodes."""
    V = z.shape[1]
    _call("eagle_draft_rows", B, V, k, depth, int(level), _ptr(z), _ptr(lse), _ptr(logp),
          _ptr(prob), _stream(stream))


def eagle_embed_rows(tokens, emb, x, status, stream=None) -> None:
    """x [T, H] fp32 = emb[tokens] (emb [V, H] bf16)."""
    V, H = emb.shape
    _call("eagle_embed_rows", tokens.numel(), H, V, _ptr(tokens), _ptr(emb), _ptr(x),
          _ptr(status), _stream(stream))


def eagle_loop_advance(tree_off, accept_len, accepted_nodes, out_tokens, resid, f_ctx,
                       root_token, status, *, max_depth: int, stream=None) -> None:
    """Next step's root token (bonus token) and context feature."""
    B = tree_off.numel() - 1
    H = resid.shape[1]
    _call("eagle_loop_advance", B, H, int(max_depth), _ptr(tree_off), _ptr(accept_len),
          _ptr(accepted_nodes), _ptr(out_tokens), _ptr(resid), _ptr(f_ctx), _ptr(root_token),
          _ptr(status), _stream(stream))
