"""GB300-native backward of packed variable-length (TND) attention.

The compute path is the C-ABI library ``libfavarlen.so`` built from
``csrc/`` for sm_103a; :mod:`varlen_flashattention_backward_gb300.binding`
marshals torch tensors into it.  The library is loaded on first use, and
every entry point raises if it is missing: there is no CPU fallback.

Submodules: ``binding`` (the library calls), ``workloads`` (seeded synthetic
inputs), ``build`` (compiles the library in-tree).
"""
