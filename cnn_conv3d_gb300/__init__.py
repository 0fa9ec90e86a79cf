"""GB300-native conv3d block for CosmoFlow-style volumetric CNNs.

The compute path is the C-ABI library ``libcfconv3d.so`` built from
``csrc/`` (hand-written sm_103a kernels); ``cnn_conv3d_gb300.cfconv`` binds it
with ctypes.  Importing this package does not load the library; importing
``cfconv`` does, and raises if it is missing.
"""
__all__ = ["flops", "build", "cfconv"]
