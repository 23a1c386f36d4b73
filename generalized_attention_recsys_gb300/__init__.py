"""GB300-native Generalized Dot Product Attention (GDPA).

The compute runs in the CUDA library ``libgdpa.so`` (built from ``csrc/``);
this package only marshals arguments to its C-ABI. Importing the package does
not load the library; the first call does, and raises if it is missing.
"""
