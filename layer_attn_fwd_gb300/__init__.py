"""GB300-native attention forward: a C-ABI CUDA library and its thin binding.

Importing the package loads nothing; the CUDA library is loaded on the first
call into ``layer_attn_fwd_gb300.api`` and a missing library raises.
"""
