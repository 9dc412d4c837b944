"""The draft -> verify -> accept -> commit loop on the GPU, step by step
against the oracle.

Every step is checked from the state the GPU left (its caches, context
feature and root token), so one near-tie cannot derail the steps after it:
  * draft: the oracle drafts the tree level by level with the same head and
    LM head; its rows agree with the GPU's rows to 1e-3 (fp32 accumulation
    and a bf16 feature rounding apart), and the tree the oracle builds from
    the GPU's rows equals the GPU's tree bit for bit;
  * verify: the oracle's decoder layer over that tree and the paged cache
    agrees with the GPU's layer output (2e-3 of the terms' scale), the LM
    head's argmax agrees outside near-ties, and the greedy walk fed the
    GPU's argmax gives the GPU's accepted path;
  * commit: the pages equal the oracle's commit of the accepted path, bit
    for bit; the next root is the bonus token and the next context feature
    the layer output at the last accepted node.
The toy draft head's embedding half is close to the identity, so the draft
usually proposes the target's own next token and accepted lengths span the
tree's depth."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu

NEAR_TIE = 1e-3


def _weights(seed, H, Hq, Hkv, D, I, V):
    bf = O.bf16_round
    g = np.random.default_rng(seed)
    w = {"g_attn": bf(1 + 0.02 * g.standard_normal(H)),
         "wq": bf(0.02 * g.standard_normal((Hq * D, H))),
         "wk": bf(0.02 * g.standard_normal((Hkv * D, H))),
         "wv": bf(0.002 * g.standard_normal((Hkv * D, H))),
         "wo": bf(0.002 * g.standard_normal((H, Hq * D))),
         "g_mlp": bf(1 + 0.02 * g.standard_normal(H)),
         "wg": bf(0.02 * g.standard_normal((I, H))),
         "wu": bf(0.02 * g.standard_normal((I, H))),
         "wd": bf(0.002 * g.standard_normal((H, I))),
         "g_final": bf(1 + 0.02 * g.standard_normal(H)),
         "w_lm": bf(0.08 * g.standard_normal((V, H))),
         "emb": bf(g.standard_normal((V, H)))}
    wdr = 0.01 * g.standard_normal((H, 2 * H))
    wdr[:, H:] += np.eye(H)
    w["w_draft"] = bf(wdr)
    return w


def test_loop_steps_match_the_oracle():
    import torch
    E = cuda_ready()
    from eagle_tree_verification_gb300.pipeline import LoopShape, SpeculativeLoop
    B, Hq, Hkv, D, H, I, V = 2, 8, 2, 128, 512, 1024, 4099
    k, depth, budget, L0, steps = 4, 4, [16, 11], [200, 64], 3
    theta, eps = 10000.0, 1e-5
    w = _weights(5, H, Hq, Hkv, D, I, V)
    g = np.random.default_rng(6)
    kc = O.bf16_round(g.standard_normal((sum(L0), Hkv, D)))
    vc = O.bf16_round(g.standard_normal((sum(L0), Hkv, D)))
    f_ctx0 = O.bf16_round(g.standard_normal((B, H)))
    root0 = np.array([17, 4000], np.int32)
    loop = SpeculativeLoop(LoopShape(B=B, Hq=Hq, Hkv=Hkv, D=D, H=H, I=I, V=V, k=k, depth=depth,
                                     budget=budget, L0=L0, steps=steps, theta=theta, eps=eps))
    loop.load(dict(w, f_ctx=f_ctx0, root_token=root0), {"k": kc, "v": vc})
    st = loop.step
    R = 1 + (depth - 1) * k
    alphas = []
    for step in range(steps):
        # ---- state the GPU starts the step from
        kp0, vp0 = to_np(st.k_pages.float()), to_np(st.v_pages.float())
        kv_len0 = to_np(st.kv_len)
        table = to_np(st.block_table)
        f_ctx = to_np(loop.f_ctx.float()).astype(np.float64)
        root = to_np(st.root_token)
        # ---- draft
        loop.run_draft()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        rows = to_np(st.draft_logp).reshape(B, R, V)
        tree, own, scale = O.build_eagle2_tree_with_head(f_ctx, root, w["emb"], w["w_draft"],
                                                         w["w_lm"], B, k, depth, budget,
                                                         rows=rows)
        for nm in ("tree_off", "parent", "tokens", "p_row_of_node"):
            np.testing.assert_array_equal(to_np(getattr(st, nm)), tree[nm], err_msg=nm)
        used = np.zeros((B, R), bool)                      # rows the draft filled
        used[:, 0] = True
        for b in range(B):
            p = tree["p_row_of_node"][tree["tree_off"][b]:tree["tree_off"][b + 1]]
            used[b, p[p >= 0] - b * R] = True
        # a feature entry that lands on the other side of a bf16 rounding
        # boundary moves by one bf16 step (at most 2^-7 of itself): a logit by
        # at most 2^-7 sum_i |f_i| max_j |w_ji|, a log-prob by twice that
        diff = np.abs(rows - own).max(axis=-1)
        assert np.all(diff[used] <= 2 * 2.0 ** -7 * scale[used] + 1e-5)
        # ---- verify
        loop.run_verify()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        toks = tree["tokens"]
        x = w["emb"][toks].astype(np.float64)
        kcache, kv_off = O.gather_pages(kp0, table, kv_len0)
        vcache, _ = O.gather_pages(vp0, table, kv_len0)
        ref = O.decoder_layer(x, w, kcache, vcache, kv_off, tree["tree_off"], tree["parent"], Hq,
                              Hkv, theta, eps, with_abs=True)
        out = to_np(st.resid).astype(np.float64)
        err = np.abs(out - ref["out"]) / np.maximum(np.abs(ref["out"]), ref["out_abs"])
        assert err.max() <= 2e-3, err.max()
        h = to_np(st.h.float()).astype(np.float64)
        lm = O.lmhead_softmax(h, w["w_lm"], 1.0, want_q=False)
        am = to_np(st.argmax)
        clear = lm["top2_gap"] >= NEAR_TIE
        np.testing.assert_array_equal(am[clear], lm["argmax"][clear])
        ref_acc = O.accept_greedy(tree["tree_off"], tree["parent"], toks, am, depth)
        got_acc = (to_np(st.accept_len), to_np(st.accepted_nodes), to_np(st.out_tokens))
        for a_, r_ in zip(got_acc, ref_acc):
            np.testing.assert_array_equal(a_, r_)
        alphas.append(got_acc[0].tolist())
        # ---- commit and advance
        loop.run_commit()
        torch.cuda.synchronize()
        assert int(st.status.item()) == 0
        kt, vt = to_np(st.k_tree.float()), to_np(st.v_tree.float())
        rk, rv, rlen = O.kv_commit_paged(kp0, vp0, table, kv_len0, tree["tree_off"], kt, vt,
                                         got_acc[0], got_acc[1])
        np.testing.assert_array_equal(to_np(st.kv_len), rlen)
        np.testing.assert_array_equal(to_np(st.k_pages.float()), rk)
        np.testing.assert_array_equal(to_np(st.v_pages.float()), rv)
        for b in range(B):
            a = int(got_acc[0][b])
            assert int(to_np(st.root_token)[b]) == int(got_acc[2][b, a])
            last = tree["tree_off"][b] + got_acc[1][b, a]
            np.testing.assert_array_equal(to_np(loop.f_ctx.float())[b],
                                          O.bf16_round(out[last]).astype(np.float32))
    print(f"[loop] accepted lengths per step: {alphas}")
    assert max(max(a) for a in alphas) >= 1          # the draft is accepted at times
