"""GPU parity of the decoder layer around the tree attention.

Kernels one by one against the oracle's definitions (the tensor-core GEMM
and its four epilogues, RMSNorm, the position / rotation table), then the
whole layer over an EAGLE-2 tree through TreeVerifyStep against
oracle.decoder_layer.

Tolerances (bf16 operands, fp32 accumulation; derived from the arithmetic):
  * an fp32 result Y = sum_k a_k w_k may differ from the fp64 sum by the
    accumulation's rounding, a small multiple of 2^-24 * sum_k |a_k w_k|:
    checked at 1e-4 of that magnitude;
  * a bf16 result may in addition land on the other side of a rounding
    boundary: one bf16 step, at most 2^-7 of its magnitude;
  * the whole layer's output, against the scale of the terms that make it
    (|x| + |o|.|Wo| + |m|.|Wd|, the oracle's out_abs): 2e-3, the bf16
    tolerance of the attention."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _t(a, dtype):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def _ab(seed, T, K, N, std=0.02):
    a = O.bf16_round(synth.normal(seed, "gemm-a", (T, K)))
    w = O.bf16_round(synth.normal(seed, "gemm-w", (N, K), std=std))
    return a, w


def _bf_ok(got, ref, scale):
    """bf16 results: within one bf16 step of the exact value, plus the
    accumulation's share."""
    got = np.asarray(got, np.float64)
    return np.abs(got - ref) <= 2.0 ** -7 * np.abs(ref) + 1e-4 * scale


# one row tile with few 256-row blocks splits K over a cluster: (1, 256, 64),
# (65, 4096, 6144), (65, 14336, 4096), (97, 200, 96); the others do not
@pytest.mark.parametrize("T,K,N", [(1, 256, 64), (65, 4096, 6144), (65, 14336, 4096),
                                   (200, 1024, 4096), (767, 512, 1024), (97, 200, 96)])
def test_gemm_store_and_accumulate(T, K, N):
    import torch
    E = cuda_ready()
    a, w = _ab(T + K + N, T, K, N)
    ref = a @ w.T
    scale = np.abs(a) @ np.abs(w).T
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.full((T, N), 7.0, dtype=torch.bfloat16, device="cuda")
    E.eagle_gemm(E.EPI_STORE, _t(a, torch.bfloat16), _t(w, torch.bfloat16), st, y=y)
    r0 = synth.normal(9, "resid", (T, N))
    acc = _t(r0, torch.float32)
    E.eagle_gemm(E.EPI_ACCUM, _t(a, torch.bfloat16), _t(w, torch.bfloat16), st, accum=acc)
    res = _t(r0, torch.float32)
    acc2 = torch.full((T, N), 5.0, dtype=torch.float32, device="cuda")
    E.eagle_gemm(E.EPI_ACCUM, _t(a, torch.bfloat16), _t(w, torch.bfloat16), st, accum=acc2,
                 resid=res)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.all(_bf_ok(to_np(y.float()), ref, scale))
    for out in (acc, acc2):
        err = np.abs(to_np(out).astype(np.float64) - (r0 + ref))
        assert np.all(err <= 1e-4 * (np.abs(r0) + scale))


@pytest.mark.parametrize("T,K,I", [(65, 1024, 2816), (300, 512, 256)])
def test_gemm_swiglu(T, K, I):
    import torch
    E = cuda_ready()
    from eagle_tree_verification_gb300.pipeline import pack_gate_up_weight
    a = O.bf16_round(synth.normal(1, "sw-a", (T, K)))
    wg = O.bf16_round(synth.normal(1, "sw-g", (I, K), std=0.05))
    wu = O.bf16_round(synth.normal(1, "sw-u", (I, K), std=0.05))
    g, u = a @ wg.T, a @ wu.T
    ref = O.silu(g) * u
    # scale of the product's error: |u| * sum|a||wg| + |silu(g)| * sum|a||wu|
    scale = np.abs(u) * (np.abs(a) @ np.abs(wg).T) + np.abs(O.silu(g)) * (np.abs(a) @ np.abs(wu).T)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    w = pack_gate_up_weight(_t(wg, torch.bfloat16), _t(wu, torch.bfloat16))
    y = torch.full((T, I), 7.0, dtype=torch.bfloat16, device="cuda")
    E.eagle_gemm(E.EPI_SWIGLU, _t(a, torch.bfloat16), w, st, y=y)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert np.all(_bf_ok(to_np(y.float()), ref, scale))


def _tree(seed, B, levels):
    parents = [synth.random_level_tree(seed + b, levels, 5)[0] for b in range(B)]
    sizes = [len(p) for p in parents]
    return (np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32),
            np.concatenate(parents).astype(np.int32))


def test_rope_table_and_rmsnorm():
    import torch
    E = cuda_ready()
    tree_off, parent = _tree(4, 3, (1, 4, 4, 4))
    Ls = [0, 700, 16384]
    kv_off = np.concatenate([[0], np.cumsum(Ls)]).astype(np.int32)
    T, D, theta = int(tree_off[-1]), 128, 500000.0
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    pos = torch.zeros(T, dtype=torch.int32, device="cuda")
    cs = torch.zeros(T, D // 2, 2, dtype=torch.float32, device="cuda")
    E.eagle_tree_rope_table(_t(tree_off, torch.int32), _t(parent, torch.int32), pos, cs, st,
                            D=D, theta=theta, kv_off=_t(kv_off, torch.int32))
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref_pos = O.tree_positions(np.diff(kv_off), tree_off, parent)
    np.testing.assert_array_equal(to_np(pos), ref_pos)
    ang = ref_pos[:, None] * theta ** (-2.0 * np.arange(D // 2) / D)
    got = to_np(cs).astype(np.float64)
    # the reduced angle rounded to fp32 (up to 2^-24 pi) and fp32 sine and
    # cosine (about one ulp): a few 1e-7
    assert np.abs(got[..., 0] - np.cos(ang)).max() <= 5e-7
    assert np.abs(got[..., 1] - np.sin(ang)).max() <= 5e-7
    # RMSNorm: bf16 output within one bf16 step of the fp64 definition
    H = 4096
    x = synth.normal(5, "norm-x", (T, H)) * 3.0
    g = O.bf16_round(1.0 + synth.normal(5, "norm-g", (H,), std=0.1))
    y = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    E.eagle_rmsnorm(_t(x, torch.float32), _t(g, torch.bfloat16), y, st, eps=1e-5)
    torch.cuda.synchronize()
    ref = O.rmsnorm(x, g, 1e-5)
    assert np.all(_bf_ok(to_np(y.float()), ref, 1e-3 * np.abs(ref)))


def _layer_case(name):
    w = synth.workloads()[name]
    inp = synth.make_inputs(w)
    lay = synth.make_layer_inputs(w)
    tree = O.build_eagle2_tree(inp["draft_logp"], B=w.B, k=w.k, depth=w.depth,
                               budget=inp["budget"], root_token=inp["root_token"])
    return w, inp, lay, tree


@pytest.mark.parametrize("name", ["smoke_bf16", "llama3_8b"])
def test_full_layer_matches_oracle(name):
    import torch
    E = cuda_ready()
    from eagle_tree_verification_gb300.pipeline import TreeVerifyStep
    from gpu_common import step_shape, load_step
    w, inp, lay, tree = _layer_case(name)
    mode = w.modes[0]
    step = TreeVerifyStep(step_shape(w, mode, layer=True, I=w.I, theta=w.theta, eps=w.eps))
    load_step(step, w, {k: v for k, v in inp.items() if k not in ("q", "k_tree", "v_tree", "h")})
    step.load({"x": lay["x"]})
    step.load_layer(lay)
    step.run()
    torch.cuda.synchronize()
    assert int(step.status.item()) == 0
    for nm in ("tree_off", "parent", "tokens"):
        np.testing.assert_array_equal(to_np(getattr(step, nm)), tree[nm])
    ref = O.decoder_layer(lay["x"], lay, inp["k_cache"], inp["v_cache"], inp["kv_off"],
                          tree["tree_off"], tree["parent"], w.Hq, w.Hkv, w.theta, w.eps,
                          with_abs=True)
    np.testing.assert_array_equal(to_np(step.pos), ref["pos"])
    # q / k / v: bf16 values, within one bf16 step (a rounding boundary)
    for nm, t in (("q", step.q), ("k", step.k_tree), ("v", step.v_tree)):
        g = to_np(t.float()).astype(np.float64)
        r = ref[nm]
        bad = np.abs(g - r) > 2.0 ** -7 * np.abs(r) + 1e-3 * np.abs(r).mean()
        assert bad.mean() < 1e-3, (nm, bad.mean())
    out = to_np(step.resid).astype(np.float64)
    err = np.abs(out - ref["out"]) / np.maximum(np.abs(ref["out"]), ref["out_abs"])
    print(f"[layer error] {name}: max |g-r|/max(|r|, out_abs) = {err.max():.3e}")
    assert err.max() <= 2e-3
    # the LM head on the layer's output, then the walk on identical inputs
    # the final norm: the layer output's error (bounded above) scaled by the
    # norm, plus one bf16 step of the rounded result
    h_ref = O.bf16_round(O.rmsnorm(ref["out"], lay["g_final"], w.eps))
    hb = to_np(step.h.float()).astype(np.float64)
    inv = 1.0 / np.sqrt(np.mean(ref["out"] ** 2, axis=1, keepdims=True) + w.eps)
    tol = 2.0 ** -7 * np.abs(h_ref) + 2e-3 * ref["out_abs"] * inv * np.abs(lay["g_final"])
    assert np.all(np.abs(hb - h_ref) <= tol)
    lm = O.lmhead_softmax(hb, inp["w_lm"], w.temperature, want_q=False)
    gap = lm["top2_gap"]
    am = to_np(step.argmax)
    np.testing.assert_array_equal(am[gap >= 1e-3], lm["argmax"][gap >= 1e-3])
