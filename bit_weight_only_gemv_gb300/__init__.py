"""GB300-native W4A16 group-32 decode GEMV library (Python binding).

The compute path is the C-ABI shared library built from ``csrc/``; this package
only marshals arguments to it (see ``lib``).  ``synth`` draws seeded inputs.
"""
