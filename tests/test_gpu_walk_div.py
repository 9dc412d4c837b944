"""The rejection rounds' division against the IEEE quotient, bit for bit.

A rejection round renormalises every entry of the target (and, without
replacement, the draft) slice: q <- fp32(W) / fp32(Z), one division rounded
to nearest with the same divisor for the whole round.  The walk computes it
from a reciprocal estimate with one correction, keeps the result only when
the exact remainder proves it is the nearest float, and otherwise divides.
This test builds a copy of the walk's source with that division exported
and compares it with numpy's float32 division (IEEE, round to nearest) on
operands shaped like the walk's -- integer-valued floats below 2^41 -- and
on the cases where rounding is delicate: quotients at and just below powers
of two, divisors with all-ones significands, exact quotients and halfway
neighbours."""
import ctypes

import numpy as np
import pytest

from gpu_common import cuda_ready

pytestmark = pytest.mark.gpu


def _operands(rng):
    xs, zs = [], []
    n = 1 << 24
    # the walk's own shape: sums near 2^40, entries anywhere below them
    z = np.floor(rng.uniform(2.0 ** 39, 2.0 ** 40, n)).astype(np.float32)
    x = np.floor(rng.uniform(0.0, 1.0, n) ** 4 * z.astype(np.float64)).astype(np.float32)
    xs.append(x); zs.append(z)
    # integers of every magnitude below 2^41
    e1 = rng.integers(0, 41, n); e2 = rng.integers(0, 41, n)
    x = np.floor(np.ldexp(rng.uniform(1.0, 2.0, n), e1)).astype(np.float32)
    z = np.floor(np.ldexp(rng.uniform(1.0, 2.0, n), e2)).astype(np.float32)
    xs.append(x); zs.append(np.maximum(z, 1.0).astype(np.float32))
    # divisors with all-ones significands and powers of two; numerators at,
    # just above and just below multiples of them (quotients near powers of
    # two and exact quotients)
    k = np.arange(24, 41, dtype=np.float64)
    zspecial = np.concatenate([np.ldexp(2.0 ** 24 - 1, (k - 24).astype(int)),
                               np.ldexp(1.0, k.astype(int)),
                               np.ldexp(2.0 ** 23 + 1, (k - 23).astype(int))]).astype(np.float32)
    for zv in zspecial:
        m = rng.integers(1, 1 << 16, 4096).astype(np.float64)
        base = np.floor(np.float64(zv) / m)
        zd = np.float64(zv)
        cand = np.concatenate([base, base + 1, base - 1, [np.floor(zd / 2), zd, zd - 1]])
        cand = cand[(cand >= 0) & (cand < 2.0 ** 41)]
        x = cand.astype(np.float32)
        xs.append(x); zs.append(np.full(x.shape, zv, np.float32))
    x = np.concatenate(xs); z = np.concatenate(zs)
    keep = np.isfinite(x) & (z >= 1.0)
    return x[keep], z[keep]


def test_round_division_is_the_ieee_quotient():
    import torch
    E = cuda_ready()
    from eagle_tree_verification_gb300 import _build
    path = _build.build_variant("libeagle_walkdivtest.so", ["accept.cu", "capi.cu"],
                                defines=["EAGLE_WALK_DIV_TEST=1"])
    lib = ctypes.CDLL(path)
    fn = lib.eagle_test_walk_div
    fn.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p]
    fn.restype = ctypes.c_int
    x, z = _operands(np.random.default_rng(20251203))
    want = (x / z).astype(np.float32)          # numpy: IEEE division, round to nearest
    dx = torch.from_numpy(x).cuda()
    dz = torch.from_numpy(z).cuda()
    out = torch.empty_like(dx)
    assert fn(dx.data_ptr(), dz.data_ptr(), out.data_ptr(), int(x.size),
              torch.cuda.current_stream().cuda_stream) == 0
    got = out.cpu().numpy()
    bad = np.flatnonzero(got.view(np.uint32) != want.view(np.uint32))
    assert bad.size == 0, (int(bad.size), [(float(x[i]), float(z[i]), float(got[i]), float(want[i]))
                                           for i in bad[:5]])
