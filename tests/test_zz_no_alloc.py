"""The allocation-free LM head entry point, through the C ABI.

eagle_lmhead_softmax_noalloc serves callers that cannot give the library a
scratch buffer (for example a serving loop that must not allocate
mid-step).  It keeps
its scratch in a fixed array inside the library.  Its results must match
eagle_lmhead_softmax's on the same inputs, call after call (the array keeps
the previous call's contents, which must not leak into the next result).
This file is collected last so that a failure here stops a `-x` run only
after every other test has run."""
import numpy as np
import pytest

import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu


def _bufs(torch, T, V, prob):
    f = lambda: torch.full((T,), -7.0, dtype=torch.float32, device="cuda")
    am = torch.full((T,), -7, dtype=torch.int32, device="cuda")
    q = torch.full((T, V), -7.0, dtype=torch.float32, device="cuda") if prob else None
    return am, f(), f(), f(), q


@pytest.mark.parametrize("dtype,T,H,V,temp", [
    ("bf16", 61, 4096, 32000, 1.0),      # Vicuna-7B shaped head, one row tile
    ("bf16", 200, 4096, 32000, 0.7),     # two row tiles: a cluster sharing W
    ("f32", 26, 256, 1024, 0.7),         # tiny fp32 head, CUDA-core path
])
def test_noalloc_matches_the_workspace_entry_point_on_consecutive_calls(dtype, T, H, V, temp):
    # Consecutive calls in the three modes (greedy, probabilities, logits),
    # each on fresh inputs: the allocation-free call must reproduce the
    # workspace call bit for bit (same kernels, same inputs), and a call
    # must not see what the previous one left in the shared scratch.
    import torch
    E = cuda_ready()
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call, mode in enumerate(("greedy", "prob", "logits")):
        full = mode != "greedy"
        h = synth.normal(100 + call, "h", (T, H))
        w = synth.normal(100 + call, "w", (V, H), std=0.02)
        d_h = torch.from_numpy(h).to(tdt).cuda()
        d_w = torch.from_numpy(w).to(tdt).cuda()
        ref = _bufs(torch, T, V, full)
        ws = torch.empty(E.eagle_lmhead_workspace_bytes(T, V), dtype=torch.uint8, device="cuda")
        E.eagle_lmhead_softmax(d_h, d_w, *ref[:4], ref[4], ws, st, temperature=temp,
                               logits=(mode == "logits"))
        got = _bufs(torch, T, V, full)
        E.eagle_lmhead_softmax_noalloc(d_h, d_w, *got[:4], got[4], st, temperature=temp,
                                       logits=(mode == "logits"))
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        for a, b in zip(got, ref):
            if a is not None:
                np.testing.assert_array_equal(to_np(a), to_np(b), err_msg=mode)
        # and the outputs are real results, not an untouched fill
        assert np.all(to_np(got[0]) >= 0) and np.all(to_np(got[0]) < V)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import torch
    E = cuda_ready()
    T, H, V = 128, 64, 131072 + 16          # one 16-row unit past the limit
    assert E.eagle_lmhead_workspace_bytes(T, V) > E.eagle_lmhead_noalloc_max_scratch_bytes()
    h = torch.zeros((T, H), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((V, H), dtype=torch.bfloat16, device="cuda")
    am, a, b, c, _ = _bufs(torch, T, V, False)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(E.EagleError) as ei:
        E.eagle_lmhead_softmax_noalloc(h, w, am, a, b, c, None, st)
    assert ei.value.code == 7                     # EAGLE_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert int(st.item()) == 0
