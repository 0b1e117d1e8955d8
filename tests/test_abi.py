"""libbsa loads, exports every symbol include/bsa.h declares, and rejects bad
arguments on the host before any launch (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_long_kv_gb300 import build, _lib
    build.build()
    return _lib.load()


def header_functions():
    text = open(os.path.join(ROOT, "include", "bsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(lib):
    from block_sparse_long_kv_gb300 import _lib
    names = header_functions()
    assert "bsa_prefill_fwd" in names and len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
        assert n in _lib.SIGNATURES, f"binding lacks {n}"


def test_status_strings(lib):
    from block_sparse_long_kv_gb300 import _lib
    for code, name in _lib.STATUS.items():
        assert lib.bsa_status_string(code).decode() == name
    assert lib.bsa_version() >= 100


FAKE = 0x10000          # aligned, never dereferenced: every call below fails validation first
MIS = 0x10001


def shp(**kw):
    from block_sparse_long_kv_gb300 import _lib
    base = dict(batch=1, seq=1024, hq=2, hkv=1, head_dim=64, block=64)
    base.update(kw)
    return _lib.Shape(**base)


@pytest.mark.parametrize("kw, code", [
    (dict(seq=1000), 2), (dict(hq=3, hkv=2), 2), (dict(batch=0), 2), (dict(seq=0), 2),
    (dict(head_dim=96), 3), (dict(block=32), 3),
    (dict(seq=64 * 4100), 3), (dict(hq=3, hkv=1, block=64), 3),               # nb > 4096; odd group
    (dict(hq=24, hkv=1, block=128), 3),                                         # group 24
])
def test_shape_validation(lib, kw, code):
    s = shp(**kw)
    p = [ctypes.c_void_p(FAKE)] * 6
    assert lib.bsa_block_meta(ctypes.byref(s), *p[:5], None, None) == code
    assert lib.bsa_prefill_dense_fwd(ctypes.byref(s), *p[:3], ctypes.c_float(0.1), p[0], None,
                                     None, None) == code
    assert lib.bsa_prefill_layer_workspace_bytes(ctypes.byref(s)) == 0


def test_null_and_misaligned_pointers(lib):
    from block_sparse_long_kv_gb300 import _lib
    s = shp()
    f = ctypes.c_void_p(FAKE)
    assert lib.bsa_block_meta(None, f, f, f, f, f, None, None) == 1
    assert lib.bsa_block_meta(ctypes.byref(s), None, f, f, f, f, None, None) == 1
    assert lib.bsa_block_meta(ctypes.byref(s), ctypes.c_void_p(MIS), f, f, f, f, None, None) == 1
    prm = _lib.SelectParams(0.25, 0.05, 0)
    args = [f] * 6
    big = ctypes.c_size_t(1 << 40)
    assert lib.bsa_select_mask(ctypes.byref(s), None, *args, None, f, big, None, None) == 1
    for bad in (_lib.SelectParams(1.5, 0.0, 0), _lib.SelectParams(0.1, -0.1, 0),
                _lib.SelectParams(float("nan"), 0.0, 0), _lib.SelectParams(0.1, 0.1, 2),
                _lib.SelectParams(0.1, 0.1, -1)):
        assert lib.bsa_select_mask(ctypes.byref(s), ctypes.byref(bad), *args, None, f, big,
                                   None, None) == 1
    need = lib.bsa_select_workspace_bytes(ctypes.byref(s))
    # q_hi, q_lo (8192 B each) + nbar (128 B) + c_hi, c_lo (4096 B each) + two 16 x 16
    # score matrices (1 KB each), each region 256-aligned
    assert need == 2 * 8192 + 256 + 2 * 4096 + 2 * 1024
    assert lib.bsa_select_mask(ctypes.byref(s), ctypes.byref(prm), *args, None, None, big,
                               None, None) == 4
    assert lib.bsa_select_mask(ctypes.byref(s), ctypes.byref(prm), *args, None, f,
                               ctypes.c_size_t(need - 1), None, None) == 4
    assert lib.bsa_prefill_fwd(ctypes.byref(s), f, f, f, None, f, ctypes.c_float(0.1), f, None,
                               None, None) == 1
    assert lib.bsa_prefill_fwd(ctypes.byref(s), f, f, f, f, f, ctypes.c_float(0.0), f, None,
                               None, None) == 1
    assert lib.bsa_prefill_fwd(ctypes.byref(s), f, f, f, f, f, ctypes.c_float(float("inf")), f,
                               None, None, None) == 1


def test_layer_workspace_layout(lib):
    s = shp(batch=2, seq=8192, hq=32, hkv=4, head_dim=128, block=128)
    total = lib.bsa_prefill_layer_workspace_bytes(ctypes.byref(s))
    offs = (ctypes.c_size_t * 6)()
    assert lib.bsa_prefill_layer_views(ctypes.byref(s), offs) == 0
    nb = 64
    sizes = [2 * 4 * 128 * nb * 4, 2 * 4 * nb * 4, 2 * 4 * 2 * 4, 2 * 4 * nb * 4,
             2 * 4 * nb * nb * 4, 2 * 4 * nb * 4]
    for x in range(6):
        assert offs[x] % 256 == 0
        if x:
            assert offs[x] >= offs[x - 1] + sizes[x - 1]
    assert total >= offs[5] + sizes[5]
    f = ctypes.c_void_p(FAKE)
    from block_sparse_long_kv_gb300 import _lib
    prm = _lib.SelectParams(0.25, 0.05, 0)
    assert lib.bsa_prefill_layer(ctypes.byref(s), ctypes.byref(prm), f, f, f, ctypes.c_float(0.1),
                                 f, None, f, ctypes.c_size_t(total - 1), None, None) == 4
    assert lib.bsa_prefill_layer(ctypes.byref(s), ctypes.byref(prm), f, f, f, ctypes.c_float(0.1),
                                 f, None, ctypes.c_void_p(FAKE + 16), ctypes.c_size_t(total),
                                 None, None) == 4


def test_product_path_has_no_oracle_or_fallback():
    pkg = os.path.join(ROOT, "block_sparse_long_kv_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "oracle" not in src.replace("oracle-free", ""), fn
                assert "import synth" not in src, fn


def vshape(**kw):
    from block_sparse_long_kv_gb300 import _lib
    base = dict(batch=3, total_tokens=2000, max_seqlen=1000, hq=4, hkv=2, head_dim=64, block=64)
    base.update(kw)
    return _lib.VarlenShape(**base)


@pytest.mark.parametrize("kw, code", [
    (dict(batch=0), 2), (dict(total_tokens=0), 2), (dict(max_seqlen=0), 2),
    (dict(max_seqlen=2001), 2), (dict(hq=3), 2),
    (dict(head_dim=96), 3), (dict(block=32), 3), (dict(hq=3, hkv=1), 3),
    (dict(total_tokens=300000, max_seqlen=64 * 4097), 3),                     # nb > 4096
])
def test_varlen_shape_validation(lib, kw, code):
    s = vshape(**kw)
    f = ctypes.c_void_p(FAKE)
    assert lib.bsa_varlen_block_meta(ctypes.byref(s), f, f, f, f, f, f, None, None) == code
    assert lib.bsa_varlen_prefill_dense_fwd(ctypes.byref(s), f, f, f, f, ctypes.c_float(0.1), f,
                                            None, None, None) == code
    assert lib.bsa_varlen_block_stride(ctypes.byref(s)) == 0
    assert lib.bsa_varlen_select_workspace_bytes(ctypes.byref(s)) == 0


def test_varlen_stride_workspace_and_pointer_checks(lib):
    from block_sparse_long_kv_gb300 import _lib
    # ceil(max_seqlen / block) rounded up to a multiple of 4
    for mx, blk, want in [(1000, 64, 16), (1025, 64, 20), (64, 64, 4), (1, 128, 4), (8192, 128, 64)]:
        s = vshape(max_seqlen=mx, total_tokens=max(mx, 2000), block=blk)
        assert lib.bsa_varlen_block_stride(ctypes.byref(s)) == want
    s = vshape()                                            # nbs = 16, rows = 3 * 4 * 16
    need = lib.bsa_varlen_select_workspace_bytes(ctypes.byref(s))
    r256 = lambda x: (x + 255) // 256 * 256
    rows, blocks = 3 * 4 * 16, 3 * 2 * 16
    assert need == 2 * r256(rows * 64 * 4) + r256(rows * 4) + 2 * r256(blocks * 64 * 4) + \
        2 * r256(blocks * 16 * 4)
    f = ctypes.c_void_p(FAKE)
    prm = _lib.SelectParams(0.25, 0.05, 0)
    big = ctypes.c_size_t(1 << 40)
    # cu_seqlens missing or misaligned
    assert lib.bsa_varlen_block_meta(ctypes.byref(s), None, f, f, f, f, f, None, None) == 1
    assert lib.bsa_varlen_block_meta(ctypes.byref(s), ctypes.c_void_p(FAKE + 2), f, f, f, f, f,
                                     None, None) == 1
    assert lib.bsa_varlen_select_mask(ctypes.byref(s), ctypes.byref(prm), f, f, f, f, f, f, f, None,
                                      None, big, None, None) == 4
    assert lib.bsa_varlen_select_mask(ctypes.byref(s), ctypes.byref(prm), f, f, f, f, f, f, f, None,
                                      f, ctypes.c_size_t(need - 1), None, None) == 4
    assert lib.bsa_varlen_prefill_fwd(ctypes.byref(s), f, f, f, f, None, f, ctypes.c_float(0.1), f,
                                      None, None, None) == 1


def test_fp8_entry_point_validation(lib):
    from block_sparse_long_kv_gb300 import _lib
    s = shp(batch=1, seq=1024, hq=4, hkv=2, head_dim=128, block=64)
    f = ctypes.c_void_p(FAKE)
    one = ctypes.c_float(1.0)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        b = ctypes.c_float(bad)
        assert lib.bsa_block_meta_fp8(ctypes.byref(s), f, b, f, f, f, f, None, None) == 1
        assert lib.bsa_prefill_dense_fwd_fp8(ctypes.byref(s), f, f, f, one, b, one, ctypes.c_float(0.1),
                                             f, None, f, ctypes.c_size_t(1 << 40), None, None) == 1
    s64 = shp(head_dim=64)                                   # e4m3 attention needs head_dim 128
    assert lib.bsa_prefill_dense_fwd_fp8(ctypes.byref(s64), f, f, f, one, one, one, ctypes.c_float(0.1),
                                         f, None, f, ctypes.c_size_t(1 << 40), None, None) == 3
    assert lib.bsa_prefill_fp8_workspace_bytes(ctypes.byref(s64)) == 0
    need = lib.bsa_prefill_fp8_workspace_bytes(ctypes.byref(s))
    assert need == 1 * 1024 * 2 * 128 * 2                    # V widened to bf16
    assert lib.bsa_prefill_dense_fwd_fp8(ctypes.byref(s), f, f, f, one, one, one, ctypes.c_float(0.1),
                                         f, None, f, ctypes.c_size_t(need - 1), None, None) == 4
    tok = _lib.SelectParams(0.1, 0.1, 1)                     # per-token aggregation reads bf16 Q
    assert lib.bsa_select_mask_fp8(ctypes.byref(s), ctypes.byref(tok), f, one, f, f, f, f, f, None, f,
                                   ctypes.c_size_t(1 << 40), None, None) == 3


def test_selftest_argument_validation(lib):
    import ctypes
    INVALID = 1
    assert lib.bsa_selftest_wait_timeout(None, ctypes.c_uint64(10_000_000), 1, None) == INVALID
    buf = (ctypes.c_int32 * 4)()
    base = ctypes.addressof(buf)
    for limit, ctas in ((999_999, 1), (1_000_000_001, 1), (10_000_000, 0), (10_000_000, 9)):
        assert lib.bsa_selftest_wait_timeout(ctypes.c_void_p(base), ctypes.c_uint64(limit), ctas, None) == INVALID
    assert lib.bsa_selftest_wait_timeout(ctypes.c_void_p(base + 2), ctypes.c_uint64(10_000_000), 1, None) == INVALID


@pytest.mark.parametrize("nb", [1, 2, 3, 5, 9, 65])
def test_any_block_count_accepted(lib, nb):
    """Only seq % block == 0 is required: block counts that are not a multiple of 4 are taken.
    The caller's per-block arrays keep the plain [b, hkv, nb, ...] layout; only the select
    scratch pads its score rows to a multiple of 4 entries."""
    for block, hq, hkv, d in ((128, 32, 4, 128), (64, 4, 2, 64)):
        s = shp(batch=2, seq=nb * block, hq=hq, hkv=hkv, head_dim=d, block=block)
        need = lib.bsa_select_workspace_bytes(ctypes.byref(s))
        rows, blocks, nbw = 2 * hq * nb, 2 * hkv * nb, (nb + 3) // 4 * 4
        r256 = lambda x: (x + 255) // 256 * 256
        assert need == (2 * r256(rows * d * 4) + r256(rows * 4) + 2 * r256(blocks * d * 4)
                        + 2 * r256(blocks * nbw * 4))
        total = lib.bsa_prefill_layer_workspace_bytes(ctypes.byref(s))
        offs = (ctypes.c_size_t * 6)()
        assert lib.bsa_prefill_layer_views(ctypes.byref(s), offs) == 0
        sizes = [blocks * d * 4, blocks * 4, 2 * hkv * 2 * 4, blocks * 4, blocks * nb * 4, blocks * 4]
        for x in range(1, 6):
            assert offs[x] >= offs[x - 1] + sizes[x - 1] and offs[x] % 256 == 0
        assert total >= offs[5] + sizes[5] + need
        # argument checks still run (and fail) before anything is launched
        f = ctypes.c_void_p(FAKE)
        assert lib.bsa_block_meta(ctypes.byref(s), None, f, f, f, f, None, None) == 1


def test_noalloc_scratch_boundary(lib):
    """bsa_select_mask_noalloc holds 12 MiB of scratch.  At 32 query heads over 4 KV heads,
    head_dim 128 and block 128 the largest layer it takes has 35072 tokens (274 blocks); the
    next block count needs more and is refused with BSA_ERR_WORKSPACE before any launch."""
    from block_sparse_long_kv_gb300 import _lib
    limit = 12 << 20
    fits = shp(seq=35072, hq=32, hkv=4, head_dim=128, block=128)
    over = shp(seq=35072 + 128, hq=32, hkv=4, head_dim=128, block=128)
    assert lib.bsa_select_workspace_bytes(ctypes.byref(fits)) <= limit
    assert lib.bsa_select_workspace_bytes(ctypes.byref(over)) > limit
    f = ctypes.c_void_p(FAKE)
    for flags in (0, _lib.SELECT_TOKEN_MAX):
        prm = _lib.SelectParams(0.1, 0.02, flags)
        assert lib.bsa_select_mask_noalloc(ctypes.byref(over), ctypes.byref(prm), f, f, f, f, f, f,
                                           None, None, None) == 4
    # shape errors are reported as by bsa_select_mask
    bad = shp(seq=1000)
    prm = _lib.SelectParams(0.1, 0.02, 0)
    assert lib.bsa_select_mask_noalloc(ctypes.byref(bad), ctypes.byref(prm), f, f, f, f, f, f,
                                       None, None, None) == 2


def test_mask_build_validation_and_workspace(lib):
    """bsa_mask_build: shape, parameter, pointer and workspace errors before any launch; its
    workspace is the select scratch plus one counter per (batch, KV head), 256-byte rounded."""
    from block_sparse_long_kv_gb300 import _lib
    s = shp(batch=2, seq=9 * 128, hq=32, hkv=4, head_dim=128, block=128)
    sel = lib.bsa_select_workspace_bytes(ctypes.byref(s))
    need = lib.bsa_mask_build_workspace_bytes(ctypes.byref(s))
    assert need == (sel + 255) // 256 * 256 + 2 * 4 * 4
    bad = shp(seq=1000)
    assert lib.bsa_mask_build_workspace_bytes(ctypes.byref(bad)) == 0
    f = ctypes.c_void_p(FAKE)
    m = ctypes.c_void_p(MIS)
    ok = _lib.SelectParams(0.1, 0.02, 0)

    def call(shape=s, prm=ok, q=f, k=f, outs=(f,) * 6, mask=None, ws=f, nbytes=need):
        return lib.bsa_mask_build(ctypes.byref(shape), None if prm is None else ctypes.byref(prm), q, k,
                                  *outs, mask, ws, ctypes.c_size_t(nbytes), None, None)

    assert call(shape=bad) == 2
    assert call(prm=None) == 1
    assert call(prm=_lib.SelectParams(0.1, 0.02, 1)) == 1      # per-token aggregation: two-call path
    assert call(prm=_lib.SelectParams(1.5, 0.02, 0)) == 1
    assert call(prm=_lib.SelectParams(float("nan"), 0.02, 0)) == 1
    assert call(q=None) == 1 and call(k=None) == 1
    assert call(q=m) == 1 and call(k=m) == 1
    for x in range(6):
        outs = [f] * 6
        outs[x] = None
        assert call(outs=tuple(outs)) == 1
        outs[x] = m
        assert call(outs=tuple(outs)) == 1
    assert call(mask=m) == 1
    assert call(ws=None) == 4 and call(ws=m) == 4
    assert call(nbytes=need - 1) == 4


def test_decode_step_validation(lib):
    """bsa_decode_step: the argument checks of bsa_decode_select and bsa_decode_fwd together,
    before any launch; its workspace is bsa_decode_workspace_bytes (which holds the barrier
    words)."""
    from block_sparse_long_kv_gb300 import _lib
    s = vshape()
    need = lib.bsa_decode_workspace_bytes(ctypes.byref(s))
    assert need > 0
    f = ctypes.c_void_p(FAKE)
    m = ctypes.c_void_p(MIS)
    ok = _lib.SelectParams(0.1, 0.02, 0)

    def call(shape=s, prm=ok, cu=f, ptrs=(f,) * 6, scale=0.1, outs=(f, f, f), lse=None, ws=f, nbytes=need):
        return lib.bsa_decode_step(ctypes.byref(shape), None if prm is None else ctypes.byref(prm), cu, *ptrs,
                                   ctypes.c_float(scale), *outs, lse, ws, ctypes.c_size_t(nbytes), None, None)

    assert call(shape=vshape(batch=0)) == 2
    assert call(cu=None) == 1 and call(cu=ctypes.c_void_p(FAKE + 2)) == 1
    assert call(prm=None) == 1
    assert call(prm=_lib.SelectParams(0.1, 0.02, 1)) == 1
    assert call(prm=_lib.SelectParams(-0.1, 0.02, 0)) == 1
    for x in range(6):                       # q_new, k, v, centroid, radius, alpha
        p = [f] * 6
        p[x] = None
        assert call(ptrs=tuple(p)) == 1
        p[x] = m
        assert call(ptrs=tuple(p)) == 1
    for x in range(3):                       # kv_idx, kv_cnt, o
        o = [f] * 3
        o[x] = None
        assert call(outs=tuple(o)) == 1
        o[x] = m
        assert call(outs=tuple(o)) == 1
    assert call(lse=m) == 1
    assert call(scale=0.0) == 1 and call(scale=float("inf")) == 1 and call(scale=float("nan")) == 1
    assert call(shape=vshape(batch=4097, total_tokens=5000, max_seqlen=64)) == 3   # batch * hkv > 4096
    assert call(ws=None) == 4 and call(ws=m) == 4
    assert call(nbytes=need - 1) == 4
