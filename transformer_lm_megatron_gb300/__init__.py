"""Tensor-sliced transformer MLP block (forward, backward, fp32 gradient
accumulation) on one GB300 GPU, behind the C ABI in ``include/gb_mlp.h``.

``inputs``  seeded synthetic workloads;  ``mlp``  ctypes binding of the library;
``build``   nvcc build of ``libgb_mlp.so`` for sm_103a.
"""
