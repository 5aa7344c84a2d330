"""CPU oracle for exact attention (test infrastructure only; see attention.py)."""
from .attention import (  # noqa: F401
    attention,
    attention_rows,
    bf16_round,
    flash_fa1,
    flash_fa2,
    naive_bf16_attention,
    safe_softmax,
)
from .backward import (  # noqa: F401
    attention_bwd,
    attention_bwd_heads,
    attention_bwd_recompute,
    naive_bf16_attention_bwd,
)
from .gqa import (  # noqa: F401
    attention_gqa,
    attention_gqa_rows,
    attention_split,
    merge_partials,
)
