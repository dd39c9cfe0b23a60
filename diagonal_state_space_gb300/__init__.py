"""GB300-native S5 layer: a C-ABI CUDA library for sm_103a and its thin binding.

The compute path lives in ``libs5.so`` (``csrc/``); ``api`` marshals torch
tensors into the C entry points declared in ``include/s5.h``.  Importing the
package does not load the library; the first API call does, and raises if the
library has not been built.
"""
__all__ = ["workloads"]
