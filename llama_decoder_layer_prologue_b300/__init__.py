"""B300-native forward pass of one Llama-style decoder layer.

The compute lives in ``libllama_layer.so`` (hand-written sm_103a kernels
behind a C ABI, declared in ``include/llama_layer.h``); ``binding`` marshals
arguments to it.  Importing this package loads nothing; ``binding.lib()``
loads the library and raises if it is missing.
"""
