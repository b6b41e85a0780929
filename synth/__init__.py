"""Seeded synthetic inputs for the DMTP round: model dimensions, weights and prompts.

This package holds no arithmetic of the method. It only draws random numbers
(weights N(0, std), prompt ids) in a fixed, seeded order and lays them out under
fixed names. Both the CPU oracle (through the tests) and the CUDA library (through
the Python binding) receive the same tensors from here.
"""
from .configs import CONFIGS, DmtpConfig, config_by_name, tap_layers
from .gen import make_prompts, make_weights, weight_specs

__all__ = ["CONFIGS", "DmtpConfig", "config_by_name", "tap_layers",
           "make_prompts", "make_weights", "weight_specs"]
