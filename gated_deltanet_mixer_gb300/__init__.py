"""libgdn: the Gated DeltaNet token mixer on one GB300 (sm_103a).

The compute path is the C-ABI library ``libgdn.so`` (``include/gdn.h``),
hand-written CUDA kernels; ``gdn`` is its thin ctypes binding.
"""
from .gdn import (GdnError, alloc_prefill_outputs, gdn_abi_version, gdn_decode_ex, gdn_decode_step,  # noqa: F401
                  gdn_device_status, gdn_linear, gdn_prefill, gdn_prefill_ex,
                  gdn_selftest_wait_timeout, gdn_status_str, lib)
