"""GB300-native (sm_103a) fused exact-attention forward.

The compute path is the C-ABI library ``libattn_gb300.so`` built from ``csrc/``;
``binding`` wraps it with ctypes. ``inputs`` draws seeded synthetic workloads.
Importing the package does not load the library; ``binding.lib()`` does, and
raises if it has not been built.
"""
