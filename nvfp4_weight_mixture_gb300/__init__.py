"""GB300-native NVFP4-weight mixture-of-experts layer.

The compute path is the CUDA library ``libmoe_nvfp4.so`` (C ABI declared in
``include/moe_nvfp4.h``); :mod:`nvfp4_weight_mixture_gb300.moe` is its thin
Python binding and :mod:`nvfp4_weight_mixture_gb300.synth` draws seeded
inputs.  Importing this package loads nothing: the library is opened on first
use of the binding, and fails loudly if it is missing.
"""
