"""GB300-native fused RankMixer block (forward + backward).

The compute lives in librmx.so (hand-written sm_103a CUDA behind the C ABI of
include/rmx.h).  ``binding`` is the ctypes layer with the same names;
``device`` keeps the block's buffers in torch device memory and calls the
library; ``inputs`` draws the seeded synthetic inputs.  Importing the package
does not load the library; the first call does, and raises if it is missing.
"""

__all__ = ["binding", "device", "inputs"]
