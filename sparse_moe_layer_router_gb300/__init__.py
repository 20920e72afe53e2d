"""GB300-native routed sparse-MoE FFN layer (router, dispatch, grouped GEMM, combine).

The compute path is the CUDA library ``libmoe_gb300.so`` (sm_103a kernels behind
a C ABI declared in ``include/moe.h``); ``binding`` marshals torch tensors into
that ABI and nothing else.  Importing this package does not load the library;
the first call does, and raises if the library is missing or no GPU is present.
"""
from .synthetic import CONFIGS, MoEConfig, MoEInputs, make_inputs  # noqa: F401

__all__ = ["CONFIGS", "MoEConfig", "MoEInputs", "make_inputs"]
