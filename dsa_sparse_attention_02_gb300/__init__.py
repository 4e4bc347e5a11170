"""GB300 (sm_103a) DSA sparse-attention step behind a C ABI (include/dsa.h).

The CUDA library is libdsa.so in this directory (built by `build.py`); `_lib`
is its ctypes binding. Nothing here computes the method in Python.
"""
from ._lib import (  # noqa: F401
    DSA_BF16, DSA_E4M3, DsaError, Geometry, dsa_abi_version, dsa_clear_error, dsa_decode_step,
    dsa_decode_step_workspace_size, dsa_get_error, dsa_indexer_scores,
    dsa_indexer_scores_workspace_size, dsa_sparse_mla_attend, dsa_sparse_mla_attend_workspace_size,
    dsa_topk, dsa_topk_workspace_size, load, make_step_args, workspace,
)
