"""GB300 MoE layer hot path: route -> dispatch -> grouped SwiGLU FFN -> combine.

The compute lives in libmoe.so (CUDA, sm_103a) behind the C ABI in
include/moe.h; ``expert_moe_route_gb300.binding`` is its thin Python binding
and ``expert_moe_route_gb300.synth`` draws the seeded synthetic workloads.
Submodules are imported on demand so that the input generators work on hosts
without a GPU.
"""
__version__ = "0.1.0"
