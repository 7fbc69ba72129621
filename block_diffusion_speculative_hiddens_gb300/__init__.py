"""GB300-native DFlash drafting round: C-ABI CUDA library + thin Python binding.

The compute path is libdflash.so (sm_103a kernels, see include/dflash.h);
``binding`` marshals torch tensors into its C calls.  Importing this package
does not load the library; ``binding.load()`` does, and fails loudly if the
library has not been built.
"""
from . import binding  # noqa: F401
from .binding import Drafter, load, weights_to_device  # noqa: F401
