"""Tensor-parallel (Megatron-style) transformer block on one B300.

``tp`` is the ctypes binding of the C-ABI library ``libtp.so``
(``include/tp.h``); ``inputs`` holds the seeded synthetic workloads;
``runtime`` allocates device buffers with torch and drives the library.
The binding is imported lazily so that ``inputs`` stays usable on machines
where the library has not been built.
"""
__all__ = ["tp", "inputs", "runtime", "build"]
