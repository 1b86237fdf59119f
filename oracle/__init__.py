"""fp64 CPU oracle for causal multi-head attention (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
arm may import this package. The CUDA product path never does.
"""

from .attention import (  # noqa: F401
    attention_backward,
    attention_forward,
    contract,
    default_scale,
    group_reference,
    head_backward,
    head_forward,
)
from .decode import gather_positions, paged_decode  # noqa: F401
from .materialized import (  # noqa: F401
    attention_probs,
    causal_softmax,
    causal_softmax_vjp,
    head_backward_probs,
    materialized_backward,
)
from .varlen import attention_backward_varlen, attention_forward_varlen  # noqa: F401
