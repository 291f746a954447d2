"""Batched gapped (affine, y-drop) seed extension on one GB300.

The compute path is a C-ABI shared library of hand-written sm_103a CUDA
kernels (``csrc/``); ``fz`` is its thin Python binding.  ``workloads`` makes
seeded synthetic inputs.
"""
