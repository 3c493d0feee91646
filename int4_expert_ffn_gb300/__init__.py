"""GB300 (sm_103a) routed-MoE forward over int4-grouped expert weights.

The public API is the binding of the C ABI (``binding.py``, same names as
``include/coli.h``).  It is loaded on first use, so that the seeded input
generators (``synth``) import without the compiled library; the binding itself
raises ImportError when ``libcoli.so`` has not been built.
"""
import importlib


def __getattr__(name):
    if name.startswith("__"):
        raise AttributeError(name)
    mod = importlib.import_module(__name__ + ".binding")
    if name == "binding":
        return mod
    return getattr(mod, name)
