"""GPU parity of the LM head + softmax statistics + argmax against the oracle.

Probabilities: elementwise relative error (q >= 1e-30) within 2e-3 for bf16
inputs and 1e-5 for fp32.  The argmax must match wherever the oracle's top-2
gap is at least 1e-3; inside a near-tie the GPU's pick must be one of the
tied logits (within 1e-3 of the maximum)."""
import numpy as np
import pytest

import oracle as O
import synth
from gpu_common import cuda_ready, to_np, tol_for

pytestmark = pytest.mark.gpu

NEAR_TIE = 1e-3


def _inputs(seed, T, H, V, dtype):
    h = synth.normal(seed, "h", (T, H))
    w = synth.normal(seed, "w", (V, H), std=0.02)
    if dtype == "bf16":
        h, w = synth.to_bf16_values(h), synth.to_bf16_values(w)
    return h, w


def _run(E, h, w, dtype, temperature, prob):
    import torch
    T, H = h.shape
    V = w.shape[0]
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d_h = torch.from_numpy(h).to(tdt).cuda()
    d_w = torch.from_numpy(w).to(tdt).cuda()
    f = lambda: torch.full((T,), -7.0, dtype=torch.float32, device="cuda")
    am = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    rm, lse, gap = f(), f(), f()
    q = torch.full((T, V), -7.0, dtype=torch.float32, device="cuda") if prob else None
    ws = torch.empty(E.eagle_lmhead_workspace_bytes(T, V), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.eagle_lmhead_softmax(d_h, d_w, am, rm, lse, gap, q, ws, st, temperature=temperature)
    torch.cuda.synchronize()
    return (to_np(am), to_np(rm), to_np(lse), to_np(gap), None if q is None else to_np(q),
            int(st.item()))


def _check(dtype, got, ref, rows):
    am, rm, lse, gap, q, st = got
    assert st == 0
    rows = np.asarray(rows)
    z = ref["z"]
    scale = np.maximum(1.0, np.abs(ref["row_max"]))
    np.testing.assert_allclose(rm[rows], ref["row_max"], rtol=0, atol=1e-4 * scale.max())
    np.testing.assert_allclose(lse[rows], ref["row_lse"], rtol=0, atol=1e-4 * scale.max())
    np.testing.assert_allclose(gap[rows], ref["top2_gap"], rtol=0, atol=2e-4)
    clear = ref["top2_gap"] >= NEAR_TIE
    np.testing.assert_array_equal(am[rows][clear], ref["argmax"][clear])
    for j in np.nonzero(~clear)[0]:
        assert z[j, am[rows[j]]] >= z[j].max() - NEAR_TIE
    if q is not None:
        qr = ref["q"].astype(np.float64)
        qg = q[rows].astype(np.float64)
        m = qr >= 1e-30
        rel = np.abs(qg[m] - qr[m]) / qr[m]
        assert rel.max() <= tol_for(dtype), rel.max()


@pytest.mark.parametrize("dtype,T,H,V,temp", [
    ("f32", 26, 256, 1024, 1.0),        # tiny fp32 layer
    ("f32", 1, 64, 1, 1.0),             # a single vocabulary entry
    ("f32", 70, 128, 1000, 0.7),        # ragged row tile and vocab tile
    ("bf16", 61, 4096, 32000, 1.0),     # Vicuna-7B shaped head
    ("bf16", 130, 512, 4099, 0.7),      # two row tiles (one CTA pair) sharing W, ragged vocab
    ("bf16", 256, 1024, 5003, 1.0),     # two full row tiles
    ("bf16", 300, 512, 2111, 0.7),      # three row tiles: two pairs, one CTA past the rows
    ("bf16", 384, 256, 1500, 1.0),      # three full tiles
    ("bf16", 513, 256, 3001, 1.0),      # five tiles, the last of one row
    ("bf16", 1100, 256, 1500, 0.7),     # nine tiles: launches of five and four tiles
    ("bf16", 1153, 256, 2003, 1.0),     # ten tiles, the last of one row
])
@pytest.mark.parametrize("prob", [False, True])
def test_lmhead_matches_oracle(dtype, T, H, V, temp, prob):
    E = cuda_ready()
    h, w = _inputs(T + V, T, H, V, dtype)
    got = _run(E, h, w, dtype, temp, prob)
    ref = O.lmhead_softmax(h, w, temp)
    _check(dtype, got, ref, np.arange(T))


@pytest.mark.parametrize("T,H,temp", [(65, 4096, 1.0), (65, 8192, 1.0), (49, 4096, 0.7),
                                      (790, 4096, 0.7)])   # 16 packed trees
def test_lmhead_full_vocab_sampled_rows(T, H, temp):
    # LLaMA-3 vocabulary (128256); the oracle checks a sample of rows
    E = cuda_ready()
    V = 128256
    h, w = _inputs(T * 3 + H, T, H, V, "bf16")
    got = _run(E, h, w, "bf16", temp, True)
    edges = [r for r in (127, 128, 255, 256, 511, 512) if r < T]   # row-tile and pass edges
    rows = np.unique(np.r_[0, T - 1, np.random.default_rng(T).integers(0, T, size=6),
                           np.asarray(edges, dtype=np.int64)]).astype(np.int64)
    ref = O.lmhead_softmax(h, w, temp, rows=rows)
    _check("bf16", got, ref, rows)


def test_lmhead_planted_ties_pick_the_lowest_index():
    E = cuda_ready()
    T, H, V = 4, 16, 300
    h = np.zeros((T, H), np.float32)
    h[:, 0] = 1.0
    w = np.zeros((V, H), np.float32)
    w[:, 0] = np.linspace(-1, 1, V, dtype=np.float32) * 0.5
    w[[7, 150, 299], 0] = 2.0          # three-way tie for the maximum
    got = _run(E, h, w, "f32", 1.0, True)
    assert list(got[0]) == [7] * T
    assert np.all(got[3] == 0.0)


@pytest.mark.parametrize("dtype,T,H,V,temp", [("f32", 26, 256, 1024, 0.7),
                                               ("bf16", 61, 4096, 32000, 1.0),
                                               ("bf16", 300, 512, 2111, 0.7),
                                               # V % 4 == 0: logits staged and written by
                                               # bulk tensor stores (one tile, then three
                                               # sharing W), ragged last 8-column box
                                               ("bf16", 100, 512, 4100, 1.0),
                                               ("bf16", 300, 512, 2116, 0.7),
                                               ("bf16", 1100, 256, 1504, 0.7)])
def test_lmhead_logits_mode(dtype, T, H, V, temp):
    # LOGITS mode stores z itself and the same statistics as the other modes
    import torch
    E = cuda_ready()
    h, w = _inputs(T + V, T, H, V, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    d_h = torch.from_numpy(h).to(tdt).cuda()
    d_w = torch.from_numpy(w).to(tdt).cuda()
    f = lambda: torch.full((T,), -7.0, dtype=torch.float32, device="cuda")
    am = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    rm, lse, gap = f(), f(), f()
    z = torch.full((T, V), -7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(E.eagle_lmhead_workspace_bytes(T, V), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    E.eagle_lmhead_softmax(d_h, d_w, am, rm, lse, gap, z, ws, st, temperature=temp, logits=True)
    torch.cuda.synchronize()
    ref = O.lmhead_softmax(h, w, temp)
    _check(dtype, (to_np(am), to_np(rm), to_np(lse), to_np(gap), None, int(st.item())), ref,
           np.arange(T))
    zr = ref["z"]
    atol = (1e-4 if dtype == "bf16" else 1e-5) * max(1.0, float(np.abs(zr).max()))
    np.testing.assert_allclose(to_np(z), zr, rtol=0, atol=atol)
