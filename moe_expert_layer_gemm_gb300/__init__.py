"""GB300-native (sm_103a) single-GPU mixture-of-experts layer: router, top-k, routing maps,
permute, grouped SwiGLU experts on tcgen05 tensor cores, weighted combine, shared expert, and
the backward pass.  The compute lives in libmoe_gb300.so (C ABI: include/moe_gb300.h); this
package is its thin Python binding.
"""
from ._lib import *  # noqa: F401,F403
from ._lib import lib, header_functions  # noqa: F401
