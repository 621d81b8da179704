"""GB300-native depth-decoder frame: one persistent sm_103a launch per frame.

The product is the C-ABI library ``_lib/libcp.so`` (include/cp.h). ``cp`` is
its ctypes binding, ``build`` compiles it in-tree and ``torch_io`` turns numpy
inputs into the torch tensors the binding takes.
"""
from . import cp  # noqa: F401
from .cp import Frame, CPError  # noqa: F401
