"""fp64 CPU oracle of the Muse Spark Open latent-MoE block.

TEST INFRASTRUCTURE ONLY.  Only tests/, the smoke check in __graft_entry__ and
the benchmark's CPU-baseline leg may import this package.  It never imports
the CUDA library, and the library never imports it.
"""
from .block import (BlockParams, ExpertStack, Trace, forward_batched, forward_per_token,  # noqa: F401
                    forward_norm_after_sum, rms_norm, route, silu, softmax, top_k, expert_ffn)
from . import formats  # noqa: F401
from .params import params_from_inputs, params_for_workload  # noqa: F401
