"""CPU checks of the C ABI: the library builds, loads, exports every symbol
include/eagle.h declares, and its host-side argument checks answer without
touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def E():
    import eagle_tree_verification_gb300 as E
    E.build()
    return E


def _declared():
    with open(os.path.join(ROOT, "include", "eagle.h")) as f:
        text = f.read()
    return re.findall(r"EAGLE_API\s+[\w\s\*]+?\b(eagle_\w+)\s*\(", text)


def test_every_declared_symbol_is_exported(E):
    names = _declared()
    assert len(names) == 26
    lib = ctypes.CDLL(E.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    # and the binding wraps each of them under the same name
    for n in names:
        assert n in E._SIGS


def test_status_strings_and_version(E):
    assert E.status_string(0) == "ok"
    assert E.status_string(2) == "invalid tree"
    assert E.status_string(99) == "unknown status"
    assert "sm_103a" in E.version()


def test_workspace_sizes_are_host_computable(E):
    assert E.eagle_lmhead_workspace_bytes(65, 128256) > 0
    assert E.eagle_lmhead_workspace_bytes(0, 128256) == 0
    assert E.eagle_draft_pool_bytes(1, 8, 7, 128256) > 0
    assert E.eagle_draft_pool_bytes(1, 33, 7, 128256) == 0      # k above the limit
    assert E.eagle_draft_pool_bytes(1, 8, 17, 128256) == 0      # depth above the limit
    assert E.eagle_draft_pool_bytes(1, 8, 7, 4) == 0            # k > V
    assert E.eagle_tree_attn_workspace_bytes(1, 65, 32, 8, 128, 65, 8192) >= 0


def test_host_argument_checks_return_before_any_device_work(E):
    L = E.lib()
    null = None
    # head dim 96 is not implemented
    assert L.eagle_tree_attn(1, 1, 4, 4, 4, 96, 0.1, 4, 0, 0, *([null] * 9), null, 0, null, null) == 3
    # Hq not a multiple of Hkv
    assert L.eagle_tree_attn(1, 1, 4, 6, 4, 128, 0.1, 4, 0, 0, *([null] * 9), null, 0, null, null) == 3
    # NULL pointers with work to do
    assert L.eagle_tree_attn(1, 1, 4, 4, 4, 128, 0.1, 4, 0, 0, *([null] * 9), null, 0, null, null) == 1
    # more nodes than the implementation allows
    assert L.eagle_accept_greedy(1, 257, *([null] * 4), 3, *([null] * 5)) == 3
    # temperature must be positive
    assert L.eagle_lmhead_softmax(1, 4, 8, 8, 0.0, 0, *([null] * 8), 0, null, null) == 1
    # unknown sampling mode
    assert L.eagle_accept_stochastic(1, 8, 10, 10, 7, *([null] * 8), 3, *([null] * 5)) == 1
    # the logits walk: temperature must be positive, row_lse given
    fake = ctypes.c_void_p(256)         # never dereferenced: the calls return first
    ptrs = [fake] * 5
    assert L.eagle_accept_stochastic_logits(1, 8, 10, 10, 1, *ptrs, 0.0, *([fake] * 4), 3,
                                            *([fake] * 4), null) == 1
    ptrs[4] = null                      # no row_lse
    assert L.eagle_accept_stochastic_logits(1, 8, 10, 10, 1, *ptrs, 1.0, *([fake] * 4), 3,
                                            *([fake] * 4), null) == 1
    # LM head: an unknown mode
    assert L.eagle_lmhead_softmax(1, 4, 8, 8, 1.0, 3, *([null] * 8), 0, null, null) == 1
    # pool too small
    fake = ctypes.c_void_p(256)         # never dereferenced: the call returns first
    assert L.eagle_draft_expand(1, 100, 4, 3, 0, 0, null, null, null, fake, 16,
                                *([null] * 6), fake, null) == 7
    # static tree: more template nodes than allowed, a rank set above the
    # top-k limit, missing pointers
    assert L.eagle_draft_static(1, 100, 257, 4, 2, *([null] * 12), null) == 3
    assert L.eagle_draft_static(1, 100, 7, 4, 33, *([null] * 12), null) == 3
    assert L.eagle_draft_static(1, 100, 7, 4, 2, *([null] * 12), null) == 1
    # empty batches are no-ops
    assert L.eagle_accept_greedy(0, 8, *([null] * 4), 3, *([null] * 5)) == 0
    assert L.eagle_draft_static(0, 100, 7, 4, 2, *([null] * 12), null) == 0


def test_product_path_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "eagle_tree_verification_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                with open(os.path.join(dirpath, f)) as fh:
                    src = fh.read()
                assert not re.search(r"^\s*(import|from)\s+oracle", src, re.M), f
                assert "oracle/" not in src, f


def test_binding_argument_counts_match_the_header(E):
    # every ctypes signature of the binding has as many arguments as the
    # C prototype in include/eagle.h
    with open(os.path.join(ROOT, "include", "eagle.h")) as f:
        text = f.read()
    for m in re.finditer(r"EAGLE_API\s+[\w\s\*]+?\b(eagle_\w+)\s*\(([^)]*)\)", text):
        name, params = m.group(1), m.group(2).strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert len(E._SIGS[name][0]) == n, name
