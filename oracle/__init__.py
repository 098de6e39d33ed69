"""Float64 CPU oracle of the triangle multiplicative update (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package. It shares no code with the CUDA library.
"""
from .trimul import (LN_EPS, DIRECTIONS, sigmoid, layer_norm, round_to_bf16, normalise_input,  # noqa: F401
                     gated_projection, contract, output, full, intermediates, sampled,
                     half_ulp_bf16, errors)
from .trimul_backward import (WEIGHT_NAMES, layer_norm_backward, contract_backward,  # noqa: F401
                              gated_projection_backward, output_backward, full_backward)
from . import triangle_attention  # noqa: F401
