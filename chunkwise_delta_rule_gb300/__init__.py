"""GB300-native chunkwise gated delta rule (DeltaNet / Gated DeltaNet / KDA).

Forward and complete ReWY backward as hand-written CUDA kernels for sm_103a
behind the C ABI in include/kda.h; this package is the thin Python binding.
Build the shared library with ``python -m chunkwise_delta_rule_gb300.build``.
"""

from .ops import (  # noqa: F401
    ChunkKDAFunction,
    Problem,
    chunk_kda,
    kda_chunk_bwd,
    kda_chunk_fwd,
    kda_device_status,
    kda_last_error,
    kda_recurrent_fwd,
    kda_saved_size,
    kda_workspace_size,
    make_problem,
)
