"""GB300 (sm_103a) INT8 mixed-precision linear layers.

The compute lives in libint8mp.so (hand-written CUDA kernels behind the C ABI
of include/int8mp.h); this package is its thin Python binding.  The library
is loaded on first use and raises if it has not been built.
"""
from .binding import *  # noqa: F401,F403
from .binding import (EXPORTED, Int8mpError, int8mp_linear_cfg, linear_cfg, load,  # noqa: F401
                      library_path)
from .autograd import Int8MixedPrecisionLinear, Int8MixedPrecisionLinearFunction  # noqa: F401,E402
from .decoder import Int8MixedPrecisionDecoderLinears  # noqa: F401,E402
