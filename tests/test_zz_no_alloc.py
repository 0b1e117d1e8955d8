"""bsa_select_mask_noalloc: the selection entry point for callers that cannot
allocate device memory (its scratch is a fixed array in the library's device
image).  Its kept lists and masks must equal those of bsa_select_mask, which
uses a caller-provided workspace, on two calls in a row, for both query
aggregations (block mean and per-token maximum).

This file is named to be collected last, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from parity_util import gpu_mask_build, shape_of, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from block_sparse_long_kv_gb300 import build, _lib
    build.build()
    return _lib.load()


def _noalloc_select(lib, w, lay, flags=0):
    import block_sparse_long_kv_gb300 as bsa
    from block_sparse_long_kv_gb300 import _lib
    s = shape_of(w)
    q, k = to_dev(lay["q"]), to_dev(lay["k"])
    meta = bsa.alloc_meta(s)
    sel = bsa.alloc_select(s, with_mask=True)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    bsa.block_meta(s, k, meta["centroid"], meta["radius"], meta["quant"], meta["alpha"], dev_status=st)
    prm = _lib.SelectParams(w.centroid_keep, w.rescue_keep, flags)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    code = lib.bsa_select_mask_noalloc(
        ctypes.byref(s), ctypes.byref(prm), p(q), p(meta["centroid"]), p(meta["radius"]),
        p(meta["alpha"]), p(sel["kv_idx"]), p(sel["kv_cnt"]), p(sel["mask"]), p(st),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0, _lib.STATUS.get(code, code)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {x: v.cpu().numpy() for x, v in sel.items()}


@pytest.mark.parametrize("flags", [0, 1])   # block-mean and per-token (BSA_SELECT_TOKEN_MAX) scores
def test_noalloc_matches_workspace_entry_point_twice(lib, flags):
    w = synth.workload("gqa32x4_n32768_d128_b128")
    for layer in (0, 1):                     # two calls in a row, different inputs
        lay = synth.make_layer(w, layer=layer)
        ref = gpu_mask_build(w, lay, flags=flags)  # bsa_select_mask with its own workspace
        got = _noalloc_select(lib, w, lay, flags)
        np.testing.assert_array_equal(got["kv_cnt"], ref["kv_cnt"])
        np.testing.assert_array_equal(got["mask"], ref["mask"])
        for b in range(w.batch):
            for g in range(w.hkv):
                for i in range(w.nb):
                    c = ref["kv_cnt"][b, g, i]
                    np.testing.assert_array_equal(got["kv_idx"][b, g, i, :c], ref["kv_idx"][b, g, i, :c])


def test_noalloc_rejects_shapes_beyond_its_scratch(lib):
    from block_sparse_long_kv_gb300 import _lib
    w = synth.workload("gqa32x4_n131072_d128_b128")      # needs 71.4 MB of scratch
    s = shape_of(w)
    prm = _lib.SelectParams(0.1, 0.02, 0)
    f = ctypes.c_void_p(0x10000)
    code = lib.bsa_select_mask_noalloc(ctypes.byref(s), ctypes.byref(prm), f, f, f, f, f, f, None,
                                       None, None)
    assert code == 4                                      # BSA_ERR_WORKSPACE, nothing launched
