"""fp64 CPU oracle for radius-rescued block-sparse causal prefill.

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the package's
``smoke()`` check and the benchmark's CPU-baseline leg may import it.  It shares
no code with the CUDA path and imports nothing from it.
"""
from .bsa_oracle import (  # noqa: F401
    block_meta, radius_quantiles, rescue_coefficient, query_summary,
    block_scores, token_block_scores, keep_count, select_row, select_blocks, kv_lists,
    sparse_attention, dense_attention, sparse_attention_rows, nearest_rank,
    ratio_ppm, PPM, FORCED, CENTROID, RESCUE,
    seq_bounds, varlen_select_blocks, varlen_attention_rows, varlen_dense_attention,
    decode_select, decode_attention, varlen_decode,
)
