"""CPU oracle for the DSA sparse-attention step: test infrastructure, not product code.

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg may import,
call or execute anything in this package. The CUDA library and its Python
binding never import it, and it imports nothing from them.
"""
from .fp8 import E4M3_TABLE, decode_bf16, decode_e4m3, decode_f32le  # noqa: F401
from .dsa import (  # noqa: F401
    query_positions, physical_rows, decode_index_q, decode_index_keys, decode_kv_rows,
    indexer_scores, topk_row, topk, sparse_mla, masked_dense_mla, dsa_step,
)
