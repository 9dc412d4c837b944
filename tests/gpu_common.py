"""Helpers shared by the GPU parity tests: build the library once, turn a
seeded workload into device buffers, and compare results with the oracle."""
import numpy as np
import pytest

import synth


def cuda_ready():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import eagle_tree_verification_gb300 as E
    E.build()
    return E


def step_shape(w: synth.Workload, mode: str, **over):
    from eagle_tree_verification_gb300.pipeline import StepShape
    kw = dict(B=w.B, Hq=w.Hq, Hkv=w.Hkv, D=w.D, H=w.H, V=w.V, L=list(w.L),
              n_nodes=w.n_nodes, rows=w.B * w.rows_per_seq, max_depth=w.max_depth,
              dtype=w.dtype, mode=mode, temperature=w.temperature)
    if w.tree == "eagle2":
        kw.update(k=w.k, depth=w.depth, budget=list(w.budget))
    elif w.tree == "static":
        kw.update(static=w.static_template())
    kw.update(over)
    return StepShape(**kw)


def load_step(step, w: synth.Workload, inp):
    """Copy the workload's inputs into a TreeVerifyStep."""
    names = ["q", "k_tree", "v_tree", "k_cache", "v_cache", "kv_off", "h", "w_lm",
             "p_rows", "u_accept", "u_sample", "root_token"]
    arrs = {n: inp[n] for n in names if n in inp}
    if w.tree == "eagle2":
        arrs["draft_logp"] = inp["draft_logp"]
        arrs["budget"] = inp["budget"]
    elif w.tree == "static":
        arrs["draft_logp"] = inp["draft_logp"]
    else:
        arrs["tree_off"] = inp["tree_off"]
        arrs["parent"] = inp["parent"]
        arrs["tokens"] = inp["tokens"]
        arrs["p_row_of_node"] = inp["p_row_of_node"]
    # the step's k_cache/v_cache buffers hold at least one row
    if arrs["k_cache"].shape[0] == 0:
        arrs.pop("k_cache")
        arrs.pop("v_cache")
    step.load(arrs)


def to_np(t):
    return t.detach().cpu().numpy()


def attn_rel_err(got, ref, abs_scale):
    """|g - r| / max(|r|, sum_j p_j |v_j|) per element.

    An output element is the weighted sum sum_j p_j v_j; rounding the
    weights or the terms perturbs it by a fraction of sum_j p_j |v_j| (the
    oracle's `with_abs` output, from its own fp64 weights), which can be far
    larger than |r| when the terms cancel.  So each element's relative error
    is measured against the larger of the two."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.maximum(np.abs(ref), np.asarray(abs_scale, np.float64))
    return np.abs(got - ref) / den


def attn_rel_err_rms(got, ref):
    """|g - r| / max(|r|, 1e-3 * rms(row)) per element (row = one head's
    output): the stricter element-relative metric, reported for the record."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    return np.abs(got - ref) / np.maximum(np.abs(ref), 1e-3 * rms)


def report_attn_err(tag, got, ref, abs_scale):
    """Both error figures of one case, printed for the test log (-s)."""
    e1 = attn_rel_err(got, ref, abs_scale).max()
    e2 = attn_rel_err_rms(got, ref).max()
    print(f"[attn error] {tag}: max |g-r|/max(|r|, sum p|v|) = {e1:.3e}; "
          f"max |g-r|/max(|r|, 1e-3 rms) = {e2:.3e}")
    return e1


def tol_for(dtype: str) -> float:
    return 2e-3 if dtype == "bf16" else 1e-5
