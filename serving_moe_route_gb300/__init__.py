"""GB300 (sm_103a) fused mixture-of-experts layer forward.

NaN-safe top-k routing, atomic-free permutation by expert, tcgen05/TMEM
grouped GEMMs (TF32, BF16, FP8 e4m3 with [128,128] block scales) with SiLU
and the top-k weighted combine fused into their epilogues, behind the C ABI
in ``include/moe_route.h``.
"""
from ._binding import MoeError, MoePlan, lib, moe_plan  # noqa: F401
from .ep import ep_forward  # noqa: F401
from .layer import BF16, F32, FP8, SIGMOID, SOFTMAX, MoELayer, route_topk  # noqa: F401

__all__ = ["MoELayer", "MoePlan", "MoeError", "route_topk", "ep_forward", "moe_plan", "lib",
           "F32", "BF16", "FP8", "SOFTMAX", "SIGMOID"]
