"""GB300-native (sm_103a) single-GPU MoE layer: route -> permute -> grouped FFN -> combine.

The compute path is the C-ABI library ``libmoe.so`` (hand-written CUDA for
sm_103a); ``mixture_experts_layer_02_gb300.moe`` is its thin ctypes binding.
Importing the package itself loads nothing; ``synth`` holds the seeded
synthetic workloads.
"""
__all__ = ["moe", "synth"]
