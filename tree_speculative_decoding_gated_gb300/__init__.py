"""tgdn — rollback-free verification of speculative draft trees through Gated DeltaNet layers.

The compute path is the C-ABI library ``libtgdn.so`` (hand-written CUDA for
sm_103a, declared in ``include/tgdn.h``); ``tgdn.py`` is its thin Python
binding.  ``synth.py`` draws the seeded synthetic workloads.  Nothing is
imported eagerly: loading the binding loads the CUDA library and fails loudly
when it has not been built.
"""

__all__ = ["synth", "tgdn"]


def __getattr__(name):
    if name in __all__:
        import importlib
        return importlib.import_module(f"{__name__}.{name}")
    raise AttributeError(name)
