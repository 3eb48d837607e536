"""GB300 (sm_103a) paged GQA split-KV decode attention with a C ABI.

The compute lives in ``_build/libpagedgqa.so`` (hand-written CUDA); this package
only marshals torch tensors into its C entry points (see include/pagedgqa.h).

A decode step, one layer (pools ``[pages, page_size, Hkv, d]`` on the device; the page
table as host int32 arrays plus its indices on the device)::

    import torch, paged_kv_gqa_05_gb300 as pg
    with pg.Plan(num_qo_heads=14, num_kv_heads=2, head_dim=64, page_size=16,
                 dtype=torch.bfloat16, max_batch=128, max_q_rows=128) as plan:
        plan.update(kv_indptr, last_page_len, kv_indices_dev, num_pages)  # once per step
        out = plan.append_run(k_new, v_new, q, k_pool, v_pool)            # per layer

``plan.update(..., qo_indptr=..., causal=True)`` describes a ragged call, in which
requests with several query rows (a prefill chunk) ride along with decode rows.
"""
from .binding import (BF16, FP16, FP32, POOL_STABLE, PagedGQAError, Plan, append_run,  # noqa: F401
                      decode_static_scratch, kv_append, kv_append_rope, load, plan_create, plan_destroy,
                      plan_get_info, plan_schedule, plan_update, read_device_flags, run)
