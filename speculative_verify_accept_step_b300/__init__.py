"""ISD verify/accept step for B300 (sm_103a): Python binding of libidlm.so.

The binding only marshals arguments: every step of the path runs in the CUDA
kernels of ``csrc/``.  Importing the package does not load the library; the
first call does, and raises if the library was not built.
"""
