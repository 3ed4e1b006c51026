"""GB300-native (sm_103a) DFlash draft-and-verify step: KV injection, one block-diffusion
draft pass and greedy verification behind a C ABI (include/dflash.h).

`binding` holds the ctypes marshalling of libdflash.so; `build` compiles it in-tree.
"""
from .build import LIB_PATH, build  # noqa: F401
