"""OSDN forward pass on GB300 (sm_103a): Python binding of the C-ABI library.

The binding is filled in by ``ops.py``; ``synth`` holds the seeded input
generators.  Importing the package does not load the CUDA library: the first
call to an operation does, and fails loudly if it is missing.
"""
