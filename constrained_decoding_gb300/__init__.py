"""GB300-native parallel constrained decoding (PCD).

A thin Python binding over the C-ABI library ``lib/libpcd.so`` (see
``include/pcd.h``): it marshals arguments only; every step of the hot path
runs in the library's CUDA kernels for sm_103a.
"""
from ._lib import load, LIB_PATH  # noqa: F401
