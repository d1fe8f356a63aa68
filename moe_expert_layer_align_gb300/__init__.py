"""GB300-native (sm_103a) fused Mixture-of-Experts layer.

The compute path is the CUDA library ``lib/libmoe_gb300.so`` behind the C ABI
declared in ``include/moe.h``; this package is its thin ctypes binding (same
function names) plus the seeded synthetic workloads used by tests and
benchmarks.  Build the library with ``moe_expert_layer_align_gb300.build``.
"""
from ._binding import *  # noqa: F401,F403
from ._binding import (LIB_PATH, SYMBOLS, MoeError, alloc_index, device_status_bits,  # noqa: F401
                       layer_shape, make_opts, make_shape, workspace_views)
