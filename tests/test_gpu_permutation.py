"""GPU: moving pages to other pool slots, with the page table remapped to match,
changes nothing, bit for bit.

The "flashlet" README's design bullets put the KV cache in a pool of fixed-size
pages addressed through a page table, so where a page sits in the pool is
bookkeeping only: a permuted pool read through the remapped table must give
exactly the output and log-sum-exp of the original, on every kernel the call
runs (decode slices, merge, prefill tiles).  The oracle's side of the same
invariant is pinned in tests/oracle_pins.py; here both GPU runs must also match
the oracle within the stated tolerance.
"""
import numpy as np
import pytest
import torch

from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu


def permuted(w: W.Workload, seed: int) -> W.Workload:
    """The same workload with pool page p moved to slot inv[p] (a seeded permutation),
    kv_indices and the append's slot mapping remapped to follow it."""
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(seed))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_pages)
    w2 = W.Workload(**{**w.__dict__})
    w2.k_pool = w.k_pool[perm].clone()
    w2.v_pool = w.v_pool[perm].clone()
    w2.kv_indices = inv.numpy()[w.kv_indices].astype(np.int32)
    if w.slot_mapping is not None:
        s = w.slot_mapping.copy()
        ok = s >= 0
        s[ok] = inv.numpy()[s[ok] // w.page_size] * w.page_size + s[ok] % w.page_size
        w2.slot_mapping = s
    return w2


CASES = [
    ("qwen05_decode", {}),                   # 256 unsplit rows, fused-append workload
    ("qwen05_decode", {"split_tokens": 64}),  # forced split: partials + merge
    ("ragged", {}),                          # prefill tiles + split decode rows + merge
    ("long_context_b1", {}),                 # 147 slices per kv head, block merge
]


@pytest.mark.parametrize("name,opts", CASES, ids=[f"{n}-{'split64' if o else 'auto'}" for n, o in CASES])
def test_page_permutation_is_bit_identical(name, opts):
    w = W.make(name)
    w2 = permuted(w, seed=1234)
    assert not np.array_equal(w.kv_indices, w2.kv_indices)
    ro, rl = H.oracle_outputs(w)
    o1, l1, i1 = H.gpu_outputs(w, torch.float32, **opts)
    o2, l2, i2 = H.gpu_outputs(w2, torch.float32, **opts)
    assert i1 == i2, "the plan depends on the lengths only"
    assert np.array_equal(o1, o2), f"{name}: permuted pool changed the output"
    assert np.array_equal(l1, l2), f"{name}: permuted pool changed the lse"
    H.compare(o1, l1, ro, rl, f"{name} {opts}")


def test_page_permutation_native_out_and_append():
    """16-bit outputs, and the pool bytes after the append, follow the permutation exactly."""
    w = W.make("qwen05_decode")
    w2 = permuted(w, seed=77)
    dt = W.TORCH_DTYPES[w.dtype]
    d1, d2 = H.to_device(w), H.to_device(w2)
    o1, l1, _ = H.gpu_outputs(w, dt, dev=d1)
    o2, l2, _ = H.gpu_outputs(w2, dt, dev=d2)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(77)).cuda()
    assert torch.equal(d1["k_pool"][perm].view(torch.int16), d2["k_pool"].view(torch.int16))
    assert torch.equal(d1["v_pool"][perm].view(torch.int16), d2["v_pool"].view(torch.int16))
