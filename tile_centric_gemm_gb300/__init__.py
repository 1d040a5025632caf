"""Tile-centric compute/communication overlap on one GB300 (sm_103a).

The library is ``libtilelink.so`` (C ABI, declared in ``include/tilelink.h``).
``tile_centric_gemm_gb300.binding`` is a thin ctypes layer over it with the same
function names; ``tile_centric_gemm_gb300.inputs`` draws the seeded synthetic
inputs.  Submodules are imported on first use so that the input generators work
on machines without the built library.
"""
import importlib

__all__ = ["binding", "inputs"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
