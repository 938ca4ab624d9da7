"""GB300-native whole-model decode megakernel.

The product is the C-ABI library ``libmk.so`` (include/mk.h) built from ``csrc/``; this package holds
its sources, the build step and a thin ctypes binding with the same entry points.
"""
from .binding import Megakernel, MKError, load, lib_path, EXPORTS  # noqa: F401
