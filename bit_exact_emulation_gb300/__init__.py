"""GB300-native bit-exact emulation of matrix-multiplier arithmetic.

The compute path is the CUDA library ``libmcemu.so`` (C ABI in ``include/mcemu.h``);
``binding`` marshals device buffers and streams into it.  Importing this package
loads nothing: the library is opened on first use and every call fails loudly
when it is missing.
"""
__all__ = ["binding", "workloads"]
