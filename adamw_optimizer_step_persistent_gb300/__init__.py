"""Fused Adam/AdamW over one data-parallel rank's optimizer shard, for GB300.

The work happens in ``_build/libfadam.so`` (hand-written sm_103a kernels and
a C ABI declared in ``include/fadam.h``); this package is its thin Python
binding.  Importing the package does not load the library; the first call
that needs it does, and fails loudly when it has not been built.
"""
from ._abi import FadamError, lib  # noqa: F401
from .optimizer import FusedAdamShard, dtype_code, step_once  # noqa: F401

__all__ = ["FusedAdamShard", "FadamError", "step_once", "dtype_code", "lib"]
