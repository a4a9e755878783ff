"""GB300-native kernelised linear attention (phi(x) = elu(x) + 1).

The compute path is the C-ABI library ``liblinattn.so`` (hand-written sm_103a
CUDA); :mod:`weight_recurrence_gb300.la` is its thin ctypes binding.  The
binding is imported lazily so that :mod:`weight_recurrence_gb300.inputs` is
usable without a GPU; the first call into the binding fails loudly if the
library has not been built.
"""
import importlib

__all__ = ["la", "inputs", "ranks"]


def __getattr__(name):
    if name in __all__:
        return importlib.import_module("." + name, __name__)
    raise AttributeError(name)
