"""A bounded device wait that runs out, on the GPU, without a fault.

Every mbarrier wait of the tensor-core kernels gives up after a cycle
budget, records EAGLE_ERR_TIMEOUT in the caller's status word, raises the
CTA's abort flag, lets its own copies in flight land, drains its MMAs and
frees its tensor memory before returning.  The product build's budget is
about two seconds, which a healthy pipeline never reaches; this test builds
a second copy of the LM head (a separate shared library) whose pipeline
waits give up after 64 cycles, far less than one TMA load takes, so the
first wait runs out.  Checked: the call returns, the status word says
TIMEOUT, and the product library's next call on the same GPU context is
correct (bit-identical to its call before)."""
import ctypes

import numpy as np
import pytest

import synth
from gpu_common import cuda_ready, to_np

pytestmark = pytest.mark.gpu

EAGLE_ERR_TIMEOUT = 5


def _outs(torch, T):
    f = lambda: torch.full((T,), -7.0, dtype=torch.float32, device="cuda")
    return torch.full((T,), -7, dtype=torch.int32, device="cuda"), f(), f(), f()


def test_pipeline_wait_times_out_and_the_context_stays_usable():
    import torch
    E = cuda_ready()
    from eagle_tree_verification_gb300 import _build
    path = _build.build_variant("libeagle_waittest.so", ["lmhead.cu", "capi.cu"],
                                defines=["EAGLE_WAIT_CYCLES=64ll"])
    tl = ctypes.CDLL(path)
    fn = tl.eagle_lmhead_softmax
    fn.argtypes = E._SIGS["eagle_lmhead_softmax"][0]
    fn.restype = ctypes.c_int

    T, H, V = 61, 4096, 32000               # one row tile: the tensor-core path
    h = torch.from_numpy(synth.normal(41, "h", (T, H))).to(torch.bfloat16).cuda()
    w = torch.from_numpy(synth.normal(41, "w", (V, H), std=0.02)).to(torch.bfloat16).cuda()
    ws = torch.empty(E.eagle_lmhead_workspace_bytes(T, V), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")

    before = _outs(torch, T)
    E.eagle_lmhead_softmax(h, w, *before, None, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0

    timed = _outs(torch, T)
    rc = fn(E.EAGLE_BF16, T, H, V, 1.0, E.LMHEAD_GREEDY, h.data_ptr(), w.data_ptr(),
            *[t.data_ptr() for t in timed], None, ws.data_ptr(),
            ws.numel(), st.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == 0                          # queued; the time-out is seen on the device
    torch.cuda.synchronize()                # the kernel returned
    assert int(st.item()) == EAGLE_ERR_TIMEOUT

    st.zero_()
    after = _outs(torch, T)
    E.eagle_lmhead_softmax(h, w, *after, None, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    for a, b in zip(after, before):
        np.testing.assert_array_equal(to_np(a), to_np(b))
