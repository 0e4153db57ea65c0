"""libtranspose for GB300 (sm_103a): out-of-place matrix transpose staged
through bank-conflict-free shared-memory tiles.

The compute path is the C-ABI shared library ``libtranspose.so`` built from
``csrc/``; ``binding`` marshals arguments into it with ctypes.  Importing this
package loads nothing: the library is opened on first use, and every call
fails loudly when it is missing -- there is no CPU fallback.
"""
from . import workloads  # noqa: F401  (pure numpy, no device code)

__all__ = ["workloads", "binding"]


def __getattr__(name):
    if name == "binding":
        import importlib
        return importlib.import_module(".binding", __name__)
    raise AttributeError(name)
