"""GB300 (sm_103a) paged KV-cache attention: store_kv, paged decode and
extend attention, and the log-sum-exp merge, as hand-written CUDA kernels
behind the C ABI of include/pkv.h. This package holds the ctypes binding
(same names as the C entry points), the nvcc build and the seeded
synthetic-input generator used by the tests and the benchmark.
"""
from .binding import (PkvError, pkv_cascade_workspace_size,  # noqa: F401
                      pkv_decode_workspace_size, pkv_extend_workspace_size, pkv_init,
                      pkv_kv_store, pkv_paged_cascade_decode_attn,
                      pkv_merge_lse, pkv_paged_decode_attn, pkv_paged_decode_attn_noalloc, pkv_paged_decode_attn_store,
                      pkv_paged_extend_attn, pkv_paged_extend_attn_store,
                      pkv_read_device_errors)
