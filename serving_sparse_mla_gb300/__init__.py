"""GB300 (sm_103a) DSA sparse-MLA attention (forward, backward) and the DSA
indexer that produces its index lists: a C-ABI CUDA library (csrc/,
include/sparse_mla.h) and its thin Python binding."""
from .binding import (  # noqa: F401
    SparseMLAError,
    clear_device_error,
    decode_workspace_size,
    dsa_indexer_scores,
    dsa_indexer_scores_paged,
    dsa_indexer_topk,
    dsa_indexer_topk_paged,
    dsa_indexer_workspace_size,
    dsa_topk,
    get_device_error,
    load,
    set_wait_timeout_ns,
    sparse_mla_bwd,
    sparse_mla_bwd_varlen,
    sparse_mla_decode,
    sparse_mla_fwd,
    sparse_mla_fwd_causal,
    sparse_mla_fwd_varlen,
)
