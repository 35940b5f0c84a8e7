"""GB300-native DFlash KV-injection draft attention.

``dflash`` is the ctypes binding of the C-ABI library ``libdflash.so``
(built from ``csrc/`` by ``build.build()``); ``synth`` draws the seeded
synthetic workloads. Neither is imported here, so that importing the package
does not load the CUDA library.
"""
__all__ = ["dflash", "synth", "build"]
