"""CPU oracle for the paged block-sparse attend (float64, numpy).

TEST INFRASTRUCTURE ONLY: used by ``tests/``, ``__graft_entry__.smoke()`` and
the cpu_baseline leg of ``bench.py``; never by the product path. It shares no
code with the CUDA kernels.
"""
from .sparse_attend import (  # noqa: F401
    PAGES_PER_BLOCK, PAGE_ROWS, SPARSE_BLOCK_SIZE, attend, attend_lse, attended_positions,
    build_sparse_block_table_decode, build_sparse_block_table_prefill, decode_query_positions,
    gather_kv, insert_index_cache, prefill_query_positions, sparse_block_table_row,
    sparse_decode_attention, sparse_prefill_attention)
from .formats import bf16_bits_to_float, e2m1_to_float, e4m3_to_float, nvfp4_slot_rows  # noqa: F401
