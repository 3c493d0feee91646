"""GB300 (sm_103a) routed-MoE forward over int4-grouped expert weights.

The public API is the binding of the C ABI (``binding.py``, same names as
``include/coli.h``).  It is loaded on first use, so that the build script
(``build``) and the seeded input generators (``synth``) import without the
compiled library; the binding itself raises ImportError when ``libcoli.so``
has not been built.
"""
import importlib

_SUBMODULES = ("binding", "build", "synth")


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    if name in _SUBMODULES:
        return importlib.import_module(__name__ + "." + name)
    return getattr(importlib.import_module(__name__ + ".binding"), name)
