"""GB300-native NVFP4 quantize-and-multiply path of one linear layer.

The compute path is libnvfp4.so (hand-written CUDA for sm_103a, C ABI in
include/nvfp4.h); ``binding`` marshals torch tensors to it.  ``workloads``
draws the seeded synthetic inputs.
"""
from . import workloads  # noqa: F401
