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


def attn_rel_err(got, ref):
    """|g - r| / max(|r|, rms(row)) per element (row = one head's output).

    The output is a weighted mean of value rows; rounding in the weighted
    sum is proportional to sum_j p_j |v_j|, which is of the order of the
    row's RMS, not of the element itself (elements near zero come from
    cancellation).  Relative error is therefore measured against the larger
    of the element and the row RMS."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    rms = np.sqrt(np.mean(ref ** 2, axis=-1, keepdims=True))
    den = np.maximum(np.abs(ref), rms)
    return np.abs(got - ref) / den


def tol_for(dtype: str) -> float:
    return 2e-3 if dtype == "bf16" else 1e-5
