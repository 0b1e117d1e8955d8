"""Python binding of the libbsa C ABI, on torch CUDA tensors.

The functions carry the C entry points' names without the ``bsa_`` prefix and
do argument marshalling only (dtype / device / contiguity checks, pointers,
the current CUDA stream); every step of the path runs in libbsa's kernels.
PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
import math

import torch

from . import _lib

__all__ = [
    "Shape", "SelectParams", "SELECT_TOKEN_MAX", "make_shape", "block_meta", "select_workspace_bytes", "select_mask", "mask_build_workspace_bytes", "mask_build", "prefill_fwd",
    "prefill_dense_fwd", "prefill_layer", "prefill_layer_workspace_bytes", "layer_views",
    "alloc_meta", "alloc_select", "alloc_layer_workspace", "status_string", "version",
    "selftest_wait_timeout",
    "VarlenShape", "make_varlen_shape", "varlen_block_stride", "varlen_block_meta",
    "varlen_select_workspace_bytes", "varlen_select_mask", "varlen_prefill_fwd",
    "varlen_prefill_dense_fwd", "alloc_varlen_meta", "alloc_varlen_select",
    "decode_workspace_bytes", "decode_select", "decode_fwd", "decode_step",
    "block_meta_fp8", "select_mask_fp8", "prefill_fwd_fp8", "prefill_dense_fwd_fp8",
    "prefill_fp8_workspace_bytes",
]

Shape = _lib.Shape
SelectParams = _lib.SelectParams
SELECT_TOKEN_MAX = _lib.SELECT_TOKEN_MAX
VarlenShape = _lib.VarlenShape


def make_shape(batch: int, seq: int, hq: int, hkv: int, head_dim: int, block: int) -> Shape:
    return Shape(batch, seq, hq, hkv, head_dim, block)


def _ptr(t, name, dtype=None, numel=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _dims(s: Shape):
    nb = s.seq // s.block
    return s.batch, s.seq, s.hq, s.hkv, s.head_dim, nb


def block_meta(shape: Shape, k, centroid, radius, quant, alpha, dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    _lib.check("bsa_block_meta", lib.bsa_block_meta(
        ctypes.byref(shape), _ptr(k, "k", torch.bfloat16, b * n * hkv * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * d * nb),
        _ptr(radius, "radius", torch.float32, b * hkv * nb),
        _ptr(quant, "quant", torch.float32, b * hkv * 2),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nb),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def select_workspace_bytes(shape: Shape) -> int:
    return int(_lib.load().bsa_select_workspace_bytes(ctypes.byref(shape)))


def select_mask(shape: Shape, params: SelectParams, q, centroid, radius, alpha, kv_idx, kv_cnt,
                mask=None, workspace=None, dev_status=None, stream=None):
    """bsa_select_mask.  ``workspace``: uint8 CUDA tensor of select_workspace_bytes(shape)
    bytes (allocated here on the current device if None)."""
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(select_workspace_bytes(shape), dtype=torch.uint8, device=q.device)
    _lib.check("bsa_select_mask", lib.bsa_select_mask(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16, b * n * hq * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * d * nb),
        _ptr(radius, "radius", torch.float32, b * hkv * nb),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nb),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nb * nb),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nb),
        _ptr(mask, "mask", torch.uint8, b * hkv * nb * nb),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def mask_build_workspace_bytes(shape: Shape) -> int:
    return int(_lib.load().bsa_mask_build_workspace_bytes(ctypes.byref(shape)))


def mask_build(shape: Shape, params: SelectParams, q, k, centroid, radius, quant, alpha, kv_idx, kv_cnt,
               mask=None, workspace=None, dev_status=None, stream=None):
    """bsa_mask_build (bsa_block_meta then bsa_select_mask in three launches).  ``workspace``:
    uint8 CUDA tensor of mask_build_workspace_bytes(shape) bytes (allocated here if None)."""
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(mask_build_workspace_bytes(shape), dtype=torch.uint8, device=q.device)
    _lib.check("bsa_mask_build", lib.bsa_mask_build(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16, b * n * hq * d),
        _ptr(k, "k", torch.bfloat16, b * n * hkv * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * d * nb),
        _ptr(radius, "radius", torch.float32, b * hkv * nb),
        _ptr(quant, "quant", torch.float32, b * hkv * 2),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nb),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nb * nb),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nb),
        _ptr(mask, "mask", torch.uint8, b * hkv * nb * nb),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def prefill_fwd(shape: Shape, q, k, v, kv_idx, kv_cnt, softmax_scale, o, lse=None,
                dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    _lib.check("bsa_prefill_fwd", lib.bsa_prefill_fwd(
        ctypes.byref(shape), _ptr(q, "q", torch.bfloat16, b * n * hq * d),
        _ptr(k, "k", torch.bfloat16, b * n * hkv * d), _ptr(v, "v", torch.bfloat16, b * n * hkv * d),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nb * nb),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nb), ctypes.c_float(softmax_scale),
        _ptr(o, "o", torch.bfloat16, b * n * hq * d), _ptr(lse, "lse", torch.float32, b * hq * n),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def prefill_dense_fwd(shape: Shape, q, k, v, softmax_scale, o, lse=None, dev_status=None,
                      stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    _lib.check("bsa_prefill_dense_fwd", lib.bsa_prefill_dense_fwd(
        ctypes.byref(shape), _ptr(q, "q", torch.bfloat16, b * n * hq * d),
        _ptr(k, "k", torch.bfloat16, b * n * hkv * d), _ptr(v, "v", torch.bfloat16, b * n * hkv * d),
        ctypes.c_float(softmax_scale), _ptr(o, "o", torch.bfloat16, b * n * hq * d),
        _ptr(lse, "lse", torch.float32, b * hq * n),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def prefill_layer_workspace_bytes(shape: Shape) -> int:
    return int(_lib.load().bsa_prefill_layer_workspace_bytes(ctypes.byref(shape)))


def prefill_layer(shape: Shape, params: SelectParams, q, k, v, softmax_scale, o, lse, workspace,
                  dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    _lib.check("bsa_prefill_layer", lib.bsa_prefill_layer(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.bfloat16, b * n * hq * d),
        _ptr(k, "k", torch.bfloat16, b * n * hkv * d), _ptr(v, "v", torch.bfloat16, b * n * hkv * d),
        ctypes.c_float(softmax_scale), _ptr(o, "o", torch.bfloat16, b * n * hq * d),
        _ptr(lse, "lse", torch.float32, b * hq * n), _ptr(workspace, "workspace", torch.uint8),
        ctypes.c_size_t(workspace.numel()), _ptr(dev_status, "dev_status", torch.int32),
        _stream(stream)))


def layer_views(shape: Shape, workspace: torch.Tensor) -> dict:
    """Tensor views of the intermediates bsa_prefill_layer leaves in its workspace."""
    b, n, hq, hkv, d, nb = _dims(shape)
    offs = (ctypes.c_size_t * 6)()
    _lib.check("bsa_prefill_layer_views", _lib.load().bsa_prefill_layer_views(ctypes.byref(shape), offs))

    def view(i, dtype, shp):
        cnt = math.prod(shp)
        return workspace[offs[i]:offs[i] + cnt * 4].view(dtype).view(*shp)

    return {
        "centroid": view(0, torch.float32, (b, hkv, nb, d)),
        "radius": view(1, torch.float32, (b, hkv, nb)),
        "quant": view(2, torch.float32, (b, hkv, 2)),
        "alpha": view(3, torch.float32, (b, hkv, nb)),
        "kv_idx": view(4, torch.int32, (b, hkv, nb, nb)),
        "kv_cnt": view(5, torch.int32, (b, hkv, nb)),
    }


def alloc_meta(shape: Shape, device="cuda") -> dict:
    b, n, hq, hkv, d, nb = _dims(shape)
    f32 = dict(dtype=torch.float32, device=device)
    return {"centroid": torch.empty(b, hkv, nb, d, **f32), "radius": torch.empty(b, hkv, nb, **f32),
            "quant": torch.empty(b, hkv, 2, **f32), "alpha": torch.empty(b, hkv, nb, **f32)}


def alloc_select(shape: Shape, device="cuda", with_mask: bool = True) -> dict:
    b, n, hq, hkv, d, nb = _dims(shape)
    out = {"kv_idx": torch.empty(b, hkv, nb, nb, dtype=torch.int32, device=device),
           "kv_cnt": torch.empty(b, hkv, nb, dtype=torch.int32, device=device)}
    out["mask"] = torch.empty(b, hkv, nb, nb, dtype=torch.uint8, device=device) if with_mask else None
    return out


def alloc_layer_workspace(shape: Shape, device="cuda") -> torch.Tensor:
    return torch.empty(prefill_layer_workspace_bytes(shape), dtype=torch.uint8, device=device)


# ---------------------------------------------------------------- fp8 (e4m3) inputs
# q, k, v: uint8 CUDA tensors of e4m3 codes in the bf16 layouts; value = code * scale.

def block_meta_fp8(shape: Shape, k, k_scale, centroid, radius, quant, alpha, dev_status=None,
                   stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    _lib.check("bsa_block_meta_fp8", lib.bsa_block_meta_fp8(
        ctypes.byref(shape), _ptr(k, "k", torch.uint8, b * n * hkv * d), ctypes.c_float(k_scale),
        _ptr(centroid, "centroid", torch.float32, b * hkv * d * nb),
        _ptr(radius, "radius", torch.float32, b * hkv * nb),
        _ptr(quant, "quant", torch.float32, b * hkv * 2),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nb),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def select_mask_fp8(shape: Shape, params: SelectParams, q, q_scale, centroid, radius, alpha, kv_idx,
                    kv_cnt, mask=None, workspace=None, dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(select_workspace_bytes(shape), dtype=torch.uint8, device=q.device)
    _lib.check("bsa_select_mask_fp8", lib.bsa_select_mask_fp8(
        ctypes.byref(shape), ctypes.byref(params), _ptr(q, "q", torch.uint8, b * n * hq * d),
        ctypes.c_float(q_scale),
        _ptr(centroid, "centroid", torch.float32, b * hkv * d * nb),
        _ptr(radius, "radius", torch.float32, b * hkv * nb),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nb),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nb * nb),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nb),
        _ptr(mask, "mask", torch.uint8, b * hkv * nb * nb),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def prefill_fp8_workspace_bytes(shape: Shape) -> int:
    return int(_lib.load().bsa_prefill_fp8_workspace_bytes(ctypes.byref(shape)))


def _fp8_ws(shape, workspace, like):
    if workspace is None:
        workspace = torch.empty(prefill_fp8_workspace_bytes(shape), dtype=torch.uint8, device=like.device)
    return workspace


def prefill_fwd_fp8(shape: Shape, q, k, v, q_scale, k_scale, v_scale, kv_idx, kv_cnt, softmax_scale,
                    o, lse=None, workspace=None, dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    workspace = _fp8_ws(shape, workspace, q)
    _lib.check("bsa_prefill_fwd_fp8", lib.bsa_prefill_fwd_fp8(
        ctypes.byref(shape), _ptr(q, "q", torch.uint8, b * n * hq * d),
        _ptr(k, "k", torch.uint8, b * n * hkv * d), _ptr(v, "v", torch.uint8, b * n * hkv * d),
        ctypes.c_float(q_scale), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nb * nb),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nb), ctypes.c_float(softmax_scale),
        _ptr(o, "o", torch.bfloat16, b * n * hq * d), _ptr(lse, "lse", torch.float32, b * hq * n),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def prefill_dense_fwd_fp8(shape: Shape, q, k, v, q_scale, k_scale, v_scale, softmax_scale, o,
                          lse=None, workspace=None, dev_status=None, stream=None):
    b, n, hq, hkv, d, nb = _dims(shape)
    lib = _lib.load()
    workspace = _fp8_ws(shape, workspace, q)
    _lib.check("bsa_prefill_dense_fwd_fp8", lib.bsa_prefill_dense_fwd_fp8(
        ctypes.byref(shape), _ptr(q, "q", torch.uint8, b * n * hq * d),
        _ptr(k, "k", torch.uint8, b * n * hkv * d), _ptr(v, "v", torch.uint8, b * n * hkv * d),
        ctypes.c_float(q_scale), ctypes.c_float(k_scale), ctypes.c_float(v_scale),
        ctypes.c_float(softmax_scale), _ptr(o, "o", torch.bfloat16, b * n * hq * d),
        _ptr(lse, "lse", torch.float32, b * hq * n),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


# ---------------------------------------------------------------- packed ragged batches

def make_varlen_shape(batch: int, total_tokens: int, max_seqlen: int, hq: int, hkv: int,
                      head_dim: int, block: int) -> VarlenShape:
    return VarlenShape(batch, total_tokens, max_seqlen, hq, hkv, head_dim, block)


def varlen_block_stride(shape: VarlenShape) -> int:
    """nbs: per-sequence stride of every per-block array (0 for an invalid shape)."""
    return int(_lib.load().bsa_varlen_block_stride(ctypes.byref(shape)))


def _vdims(s: VarlenShape):
    nbs = varlen_block_stride(s)
    if nbs == 0:
        raise _lib.BsaError("bsa_varlen_block_stride", 2)
    return s.batch, s.total_tokens, s.hq, s.hkv, s.head_dim, nbs


def _cu(cu_seqlens, batch):
    return _ptr(cu_seqlens, "cu_seqlens", torch.int32, batch + 1)


def varlen_block_meta(shape: VarlenShape, cu_seqlens, k, centroid, radius, quant, alpha,
                      dev_status=None, stream=None):
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    _lib.check("bsa_varlen_block_meta", lib.bsa_varlen_block_meta(
        ctypes.byref(shape), _cu(cu_seqlens, b), _ptr(k, "k", torch.bfloat16, t * hkv * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * nbs * d),
        _ptr(radius, "radius", torch.float32, b * hkv * nbs),
        _ptr(quant, "quant", torch.float32, b * hkv * 2),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nbs),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def varlen_select_workspace_bytes(shape: VarlenShape) -> int:
    return int(_lib.load().bsa_varlen_select_workspace_bytes(ctypes.byref(shape)))


def varlen_select_mask(shape: VarlenShape, params: SelectParams, cu_seqlens, q, centroid, radius,
                       alpha, kv_idx, kv_cnt, mask=None, workspace=None, dev_status=None,
                       stream=None):
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(varlen_select_workspace_bytes(shape), dtype=torch.uint8,
                                device=q.device)
    _lib.check("bsa_varlen_select_mask", lib.bsa_varlen_select_mask(
        ctypes.byref(shape), ctypes.byref(params), _cu(cu_seqlens, b),
        _ptr(q, "q", torch.bfloat16, t * hq * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * nbs * d),
        _ptr(radius, "radius", torch.float32, b * hkv * nbs),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nbs),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nbs * nbs),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nbs),
        _ptr(mask, "mask", torch.uint8, b * hkv * nbs * nbs),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def varlen_prefill_fwd(shape: VarlenShape, cu_seqlens, q, k, v, kv_idx, kv_cnt, softmax_scale, o,
                       lse=None, dev_status=None, stream=None):
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    _lib.check("bsa_varlen_prefill_fwd", lib.bsa_varlen_prefill_fwd(
        ctypes.byref(shape), _cu(cu_seqlens, b), _ptr(q, "q", torch.bfloat16, t * hq * d),
        _ptr(k, "k", torch.bfloat16, t * hkv * d), _ptr(v, "v", torch.bfloat16, t * hkv * d),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nbs * nbs),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv * nbs), ctypes.c_float(softmax_scale),
        _ptr(o, "o", torch.bfloat16, t * hq * d), _ptr(lse, "lse", torch.float32, hq * t),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def varlen_prefill_dense_fwd(shape: VarlenShape, cu_seqlens, q, k, v, softmax_scale, o, lse=None,
                             dev_status=None, stream=None):
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    _lib.check("bsa_varlen_prefill_dense_fwd", lib.bsa_varlen_prefill_dense_fwd(
        ctypes.byref(shape), _cu(cu_seqlens, b), _ptr(q, "q", torch.bfloat16, t * hq * d),
        _ptr(k, "k", torch.bfloat16, t * hkv * d), _ptr(v, "v", torch.bfloat16, t * hkv * d),
        ctypes.c_float(softmax_scale), _ptr(o, "o", torch.bfloat16, t * hq * d),
        _ptr(lse, "lse", torch.float32, hq * t),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def alloc_varlen_meta(shape: VarlenShape, device="cuda") -> dict:
    b, t, hq, hkv, d, nbs = _vdims(shape)
    f32 = dict(dtype=torch.float32, device=device)
    return {"centroid": torch.empty(b, hkv, nbs, d, **f32), "radius": torch.empty(b, hkv, nbs, **f32),
            "quant": torch.empty(b, hkv, 2, **f32), "alpha": torch.empty(b, hkv, nbs, **f32)}


def alloc_varlen_select(shape: VarlenShape, device="cuda", with_mask: bool = True) -> dict:
    b, t, hq, hkv, d, nbs = _vdims(shape)
    out = {"kv_idx": torch.empty(b, hkv, nbs, nbs, dtype=torch.int32, device=device),
           "kv_cnt": torch.empty(b, hkv, nbs, dtype=torch.int32, device=device)}
    out["mask"] = (torch.empty(b, hkv, nbs, nbs, dtype=torch.uint8, device=device)
                   if with_mask else None)
    return out


# ---------------------------------------------------------------- decode

def decode_workspace_bytes(shape: VarlenShape) -> int:
    return int(_lib.load().bsa_decode_workspace_bytes(ctypes.byref(shape)))


def decode_select(shape: VarlenShape, params: SelectParams, cu_seqlens, q_new, centroid, radius,
                  alpha, kv_idx, kv_cnt, workspace=None, dev_status=None, stream=None):
    """bsa_decode_select: kept blocks of each sequence's new token (kv_idx [b, hkv, nbs],
    kv_cnt [b, hkv]).  ``workspace``: uint8 tensor of decode_workspace_bytes(shape) bytes."""
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(shape), dtype=torch.uint8, device=q_new.device)
    _lib.check("bsa_decode_select", lib.bsa_decode_select(
        ctypes.byref(shape), ctypes.byref(params), _cu(cu_seqlens, b),
        _ptr(q_new, "q_new", torch.bfloat16, b * hq * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * nbs * d),
        _ptr(radius, "radius", torch.float32, b * hkv * nbs),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nbs),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nbs),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def decode_fwd(shape: VarlenShape, cu_seqlens, q_new, k, v, kv_idx, kv_cnt, softmax_scale, o,
               lse=None, workspace=None, dev_status=None, stream=None):
    """bsa_decode_fwd: o [b, hq, d] of each sequence's new token over its kept blocks."""
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(shape), dtype=torch.uint8, device=q_new.device)
    _lib.check("bsa_decode_fwd", lib.bsa_decode_fwd(
        ctypes.byref(shape), _cu(cu_seqlens, b), _ptr(q_new, "q_new", torch.bfloat16, b * hq * d),
        _ptr(k, "k", torch.bfloat16, t * hkv * d), _ptr(v, "v", torch.bfloat16, t * hkv * d),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nbs),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv), ctypes.c_float(softmax_scale),
        _ptr(o, "o", torch.bfloat16, b * hq * d), _ptr(lse, "lse", torch.float32, b * hq),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def decode_step(shape: VarlenShape, params: SelectParams, cu_seqlens, q_new, k, v, centroid, radius,
                alpha, softmax_scale, kv_idx, kv_cnt, o, lse=None, workspace=None, dev_status=None,
                stream=None):
    """bsa_decode_step: decode_select then decode_fwd in one cooperative launch."""
    b, t, hq, hkv, d, nbs = _vdims(shape)
    lib = _lib.load()
    if workspace is None:
        workspace = torch.empty(decode_workspace_bytes(shape), dtype=torch.uint8, device=q_new.device)
    _lib.check("bsa_decode_step", lib.bsa_decode_step(
        ctypes.byref(shape), ctypes.byref(params), _cu(cu_seqlens, b),
        _ptr(q_new, "q_new", torch.bfloat16, b * hq * d),
        _ptr(k, "k", torch.bfloat16, t * hkv * d), _ptr(v, "v", torch.bfloat16, t * hkv * d),
        _ptr(centroid, "centroid", torch.float32, b * hkv * nbs * d),
        _ptr(radius, "radius", torch.float32, b * hkv * nbs),
        _ptr(alpha, "alpha", torch.float32, b * hkv * nbs), ctypes.c_float(softmax_scale),
        _ptr(kv_idx, "kv_idx", torch.int32, b * hkv * nbs),
        _ptr(kv_cnt, "kv_cnt", torch.int32, b * hkv),
        _ptr(o, "o", torch.bfloat16, b * hq * d), _ptr(lse, "lse", torch.float32, b * hq),
        _ptr(workspace, "workspace", torch.uint8), ctypes.c_size_t(workspace.numel()),
        _ptr(dev_status, "dev_status", torch.int32), _stream(stream)))


def selftest_wait_timeout(dev_status, limit_ns: int, ctas: int = 1, stream=None):
    """bsa_selftest_wait_timeout: CTAs that wait on a barrier nothing completes; CTA 0 gives
    up after limit_ns and writes BSA_ERR_DEVICE_TIMEOUT into dev_status, the others stop on
    seeing it."""
    lib = _lib.load()
    _lib.check("bsa_selftest_wait_timeout", lib.bsa_selftest_wait_timeout(
        _ptr(dev_status, "dev_status", torch.int32, 1), ctypes.c_uint64(limit_ns), ctypes.c_int32(ctas),
        _stream(stream)))


def status_string(code: int) -> str:
    return _lib.load().bsa_status_string(code).decode()


def version() -> int:
    return int(_lib.load().bsa_version())
