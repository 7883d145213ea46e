"""CPU float64 oracle (test infrastructure only; see sparse_mla_oracle)."""
from .sparse_mla_oracle import (  # noqa: F401
    attend,
    sparse_mla_decode,
    sparse_mla_fwd,
    sparse_mla_fwd_varlen,
    valid_count_dense,
)
