"""libdspark: GB300-native candidate selection and rejection-sampling verification for
DFlash/DSpark block speculative decoding. The compute path is the CUDA library
``lib/libdspark.so`` (built from ``csrc/`` by ``build.build()``); this package is its thin
ctypes binding, with PyTorch used for device memory and streams only."""
from ._binding import *  # noqa: F401,F403
from ._binding import DsparkError, QRecord, lib  # noqa: F401
