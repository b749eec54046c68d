"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

Only the test suite, the package's smoke check and the benchmark's CPU
baseline leg may import this package.  The product path (the CUDA library
and its Python binding) never imports, calls or links anything here, and
nothing here imports the product package.
"""

from .attention import (  # noqa: F401
    TILE,
    allowed_mask,
    attention_forward,
    attention_backward,
    attention_forward_online,
    attention_forward_rows,
    attention_backward_varlen,
    attention_forward_varlen,
    live_tiles,
)
from .philox import dropout_keep, dropout_p8, philox4x32_10  # noqa: F401
from .kvcache import (  # noqa: F401
    attention_forward_kvcache,
    kvcache_allowed,
    merge_partial_states,
)
