"""Seeded synthetic inputs for the chunkwise gated delta-rule operator.

This package is shared by the tests, the benchmark and the oracle harness. It
only draws random tensors and applies the input recipe (L2 normalisation of q
and k, log-sigmoid gates, sigmoid betas, dtype rounding); it contains none of
the operator's own arithmetic.
"""

from .configs import CONFIGS, Case, make_case, make_config_case, varlen_lengths  # noqa: F401
