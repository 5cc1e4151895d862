"""GB300-native causal-convolution stack of the Wan2.2 video VAE decoder.

The compute lives in libcc.so (C ABI in include/cc.h, sm_103a kernels);
``api`` is its Python binding and ``inputs`` the seeded synthetic inputs.
Importing the package does not load the library; the first call does, and
fails loudly if it has not been built.
"""

__version__ = "0.1.0"
