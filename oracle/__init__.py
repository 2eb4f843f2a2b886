"""fp64 CPU oracle for exact attention: test infrastructure, never the product path.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline legs
may import it.  It shares no code with the CUDA library.
"""

from .attention import (  # noqa: F401
    attn_blockwise_normalised_sum,
    attn_bwd_dq_rows,
    attn_bwd_kv_rows,
    attn_bwd_ref,
    attn_fwd_ref,
    attn_fwd_rows,
    attn_online_ref,
    attn_probs,
    brute_force_fwd,
)
from .varlen import (  # noqa: F401
    attn_bwd_qk,
    attn_fwd_qk,
    attn_varlen_bwd_ref,
    attn_varlen_fwd_ref,
    brute_force_fwd_qk,
)
