"""GB300 (sm_103a) causal Polar Attention: C-ABI library + thin binding.

The compute lives in libpolarattn.so (CUDA kernels for sm_103a); this
package only builds it, loads it and marshals torch tensors into it.
"""
from .polar import (  # noqa: F401
    Consts,
    bwd,
    bwd_stats,
    bwd_workspace_bytes,
    PolarError,
    combine,
    decode,
    decode_paged,
    decode_static_scratch,
    decode_paged_workspace_bytes,
    decode_num_splits,
    decode_workspace_bytes,
    default_consts,
    device_status,
    fwd,
    fwd_host,
    fwd_host_workspace_bytes,
    fwd_stats,
    lib,
    memory_step,
    selftest_wait_timeout,
    strerror,
    version,
)
