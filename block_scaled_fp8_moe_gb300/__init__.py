"""GB300-native routed-expert MoE layer (FP8 activations x FP4 weights, block-scaled tcgen05).

The compute path is libmoe.so (hand-written CUDA for sm_103a, C ABI in include/moe.h);
`binding` is its thin ctypes wrapper and raises on import if the library is not built.
`synth` holds the seeded synthetic inputs.
"""
