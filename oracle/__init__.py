"""fp64 CPU oracle (test infrastructure only; never used by the product path)."""
from .sdpa_oracle import attention_dense, attention_one_head, attention_varlen  # noqa: F401
