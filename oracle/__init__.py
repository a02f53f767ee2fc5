"""Float64 CPU oracle of the RankMixer block (test infrastructure only).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may
import this package.  It shares no code with the CUDA path.
"""

from .rmx_oracle import (  # noqa: F401
    EPS_INNER, EPS_OUTER, backward, dense_ffn_v2_forward, forward,
    forward_backward, layer_norm, layer_norm_backward, sigmoid, silu,
    silu_grad, token_mixer,
)
