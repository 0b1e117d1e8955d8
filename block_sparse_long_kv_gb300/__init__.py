"""Radius-rescued block-sparse long-context prefill attention for GB300.

The hot path (key-block meta, selection, sparse attention) runs in libbsa's
hand-written sm_103a CUDA kernels behind the C ABI in ``include/bsa.h``;
``api`` is its thin torch binding.  Build with
``python -m block_sparse_long_kv_gb300.build``.
"""
from .api import *  # noqa: F401,F403
from .api import __all__  # noqa: F401
