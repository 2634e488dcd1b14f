"""GB300-native uniform spatial grid build: count -> scan -> scatter -> gather.

The compute path is libugrid.so (hand-written CUDA for sm_103a behind a C
ABI, ``include/ugrid.h``); ``uniform_grid_particle_gb300.ugrid`` is its Python
binding and ``uniform_grid_particle_gb300.scenes`` draws seeded synthetic
particle scenes.  The binding is imported on first use so that the scene
generator works on machines without the library.
"""
import importlib

__all__ = ["ugrid", "scenes"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
