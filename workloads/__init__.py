"""Seeded synthetic inputs for the latent-MoE block (shared by the tests, the
benchmark and the smoke check; holds none of the block's arithmetic)."""
from .configs import (WORKLOADS, DECODE_SWEEP_T, Workload, BlockInputs, make_inputs,  # noqa: F401
                      dense_weight, nvfp4_weight, gammas, x_tensor, zipf_bias,
                      forced_routing, hot_experts, nvfp4_tensor_scale, to_device)
