"""GB300 (sm_103a) paged GQA split-KV decode attention with a C ABI.

The compute lives in ``_build/libpagedgqa.so`` (hand-written CUDA); this package
only marshals torch tensors into its C entry points (see include/pagedgqa.h).
"""
from .binding import (BF16, FP16, FP32, POOL_STABLE, PagedGQAError, Plan, append_run,  # noqa: F401
                      decode_static_scratch, kv_append, kv_append_rope, load, plan_create, plan_destroy,
                      plan_get_info,
                      plan_update, read_device_flags, run)
