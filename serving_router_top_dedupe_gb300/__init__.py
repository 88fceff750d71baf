"""GB300-native MoE-layer expert-cache hot path (FreeToken-style), behind libftmoe.

`ftmoe` is the thin ctypes binding of the C ABI in include/ft_moe.h; `build`
compiles the CUDA library in-tree for sm_103a.
"""
