"""GB300 (sm_103a) mixture-of-experts layer: routing, int4 grouped expert GEMMs and
decode; grouped-query decode attention over a fixed-block KV cache; and the
Gated DeltaNet scan.

The compute lives in liblily_moe.so (CUDA kernels behind a C ABI, see
include/lily_moe.h); ``_abi`` is its ctypes binding.  Importing this package
loads nothing; the library is built / loaded on first use.
"""
from ._abi import (LilyError, alloc_attn_workspace, alloc_routing, lily_attn_decode, lily_attn_workspace_bytes,  # noqa: F401
                   make_attn_shape, lily_gdn_scan, alloc_workspace, lily_moe_block_capacity, lily_moe_check_shape,  # noqa: F401
                   lily_moe_clear_status, lily_moe_decode, lily_moe_device_status, lily_moe_forward,
                   lily_moe_forward_timed, lily_moe_grouped_gemm, lily_moe_last_error_detail, lily_moe_route, lily_moe_route_noalloc, lily_moe_status_string,
                   lily_moe_version, lily_moe_workspace_bytes, load, make_routing, make_shape, make_weights)
