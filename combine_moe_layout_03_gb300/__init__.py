"""MoE token dispatch and combine on one GB300 GPU (sm_103a).

The hot path is libmoe.so (C ABI in include/moe.h); `combine_moe_layout_03_gb300.moe`
is its Python binding and raises on import if the library has not been built.
`combine_moe_layout_03_gb300.synth` holds the seeded synthetic inputs.
"""
__all__ = ["moe", "synth"]
