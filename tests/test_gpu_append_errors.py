"""GPU: paged KV append bit-exactness, device-side bounds checks, and the
status codes of malformed calls."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dtype,hkv,d,ps", [("bf16", 2, 64, 16), ("fp16", 2, 128, 256),
                                             ("bf16", 8, 128, 64), ("fp16", 1, 64, 32)])
def test_append_bit_exact(dtype, hkv, d, ps):
    gen = torch.Generator().manual_seed(hkv * d + ps)
    P = 40
    tdt = W.TORCH_DTYPES[dtype]
    kp = torch.randn(P, ps, hkv, d, generator=gen).to(tdt)
    vp = torch.randn(P, ps, hkv, d, generator=gen).to(tdt)
    T = 300
    k = torch.randn(T, hkv, d, generator=gen).to(tdt)
    v = torch.randn(T, hkv, d, generator=gen).to(tdt)
    slots = torch.randperm(P * ps, generator=gen)[:T].to(torch.int64)
    slots[::17] = -1  # padding rows are skipped
    rk, rv = W.raw16(kp).copy(), W.raw16(vp).copy()
    oracle.get().kv_append(rk, rv, W.raw16(k), W.raw16(v), slots.numpy())
    dk, dv = kp.cuda(), vp.cuda()
    pg.kv_append(dk, dv, k.cuda(), v.cuda(), slots.cuda())
    torch.cuda.synchronize()
    assert np.array_equal(W.raw16(dk), rk) and np.array_equal(W.raw16(dv), rv)
    assert pg.read_device_flags() == 0


def test_append_then_decode_matches_oracle():
    w = W.qwen05_decode(batch=16, cached=100, num_pages=512)
    ro, rl = H.oracle_outputs(w)
    out, lse, _ = H.gpu_outputs(w)
    H.compare(out, lse, ro, rl, "append+decode")
    # without the append, the new token's pool rows are NaN and must poison the output
    out2, _, _ = H.gpu_outputs(w, append=False)
    assert np.isnan(out2).all(axis=(1, 2)).all()


def test_append_out_of_range_slot_flagged():
    kp = torch.zeros(4, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    vp = torch.zeros_like(kp)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device="cuda")
    slots = torch.tensor([3, 4 * 16 + 5], dtype=torch.int64, device="cuda")
    pg.read_device_flags(clear=True)
    pg.kv_append(kp, vp, k, k, slots)
    flags = pg.read_device_flags(clear=True)
    assert flags & 2, "out-of-range slot must raise the slot flag"
    assert kp.view(-1, 2, 64)[3].float().eq(1).all()
    assert pg.read_device_flags() == 0


def test_bad_page_index_without_mirror_is_flagged():
    """An index past the pool, with no host mirror to catch it, is skipped by the
    kernel and reported through the flag word instead of being read."""
    w = W.custom("bad", [20, 40], 16, 4, 2, 64, "bf16", 16, seed=2)
    w.kv_indices = w.kv_indices.copy()
    w.kv_indices[1] = 1000
    pg.read_device_flags(clear=True)
    H.gpu_outputs(w, host_mirror=False)
    assert pg.read_device_flags(clear=True) & 1


def _plan(**kw):
    args = dict(num_qo_heads=4, num_kv_heads=2, head_dim=64, page_size=16, dtype=torch.bfloat16,
                max_batch=4, max_q_rows=8)
    args.update(kw)
    return pg.Plan(**args)


@pytest.mark.parametrize("kw,status", [
    (dict(head_dim=96), "PGQA_ERR_UNSUPPORTED"),
    (dict(page_size=48), "PGQA_ERR_UNSUPPORTED"),
    (dict(num_qo_heads=5), "PGQA_ERR_INVALID_ARG"),
    (dict(num_qo_heads=34), "PGQA_ERR_UNSUPPORTED"),                         # 17 heads per kv head
    (dict(num_qo_heads=18, decode_kernel="cuda_core"), "PGQA_ERR_UNSUPPORTED"),  # 9: CUDA-core limit is 8
    (dict(dtype=torch.float32), "PGQA_ERR_UNSUPPORTED"),
    (dict(max_batch=0), "PGQA_ERR_INVALID_ARG"),
])
def test_plan_create_rejects(kw, status):
    with pytest.raises(pg.PagedGQAError) as e:
        _plan(**kw)
    assert e.value.name == status


@pytest.mark.parametrize("indptr,last,indices,status", [
    ([0, 2, 1], [16, 3], [0, 1, 2], "PGQA_ERR_BAD_PAGE_TABLE"),     # indptr decreases
    ([0, 2, 3], [17, 3], [0, 1, 2], "PGQA_ERR_BAD_PAGE_TABLE"),     # last_page_len > page_size
    ([0, 2, 3], [0, 3], [0, 1, 2], "PGQA_ERR_BAD_PAGE_TABLE"),      # last_page_len 0 with pages
    ([0, 0, 1], [5, 3], [0], "PGQA_ERR_BAD_PAGE_TABLE"),            # no pages, nonzero fill
    ([0, 2, 3], [16, 3], [0, 1, 99], "PGQA_ERR_BAD_PAGE_TABLE"),    # index outside the pool
    ([1, 2, 3], [16, 3], [0, 1, 2], "PGQA_ERR_BAD_PAGE_TABLE"),     # indptr[0] != 0
    ([0, 1, 2, 3, 4, 5], [1] * 5, [0, 1, 2, 3, 4], "PGQA_ERR_CAPACITY"),  # batch > max_batch
])
def test_plan_update_rejects(indptr, last, indices, status):
    p = _plan()
    idx = torch.tensor(indices, dtype=torch.int32, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        p.update(np.array(indptr), np.array(last), idx, 8, kv_indices_host=np.array(indices))
    assert e.value.name == status
    with pytest.raises(pg.PagedGQAError) as e2:  # a rejected plan cannot be run
        p.run(torch.zeros(2, 4, 64, dtype=torch.bfloat16, device="cuda"),
              torch.zeros(8, 16, 2, 64, dtype=torch.bfloat16, device="cuda"),
              torch.zeros(8, 16, 2, 64, dtype=torch.bfloat16, device="cuda"))
    assert e2.value.name == "PGQA_ERR_INVALID_ARG"


def test_run_rejects_wrong_out_dtype_and_misalignment():
    w = W.custom("x", [5], 16, 4, 2, 64, "bf16", 4, seed=0)
    dev = H.to_device(w)
    p = _plan()
    p.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages)
    with pytest.raises(pg.PagedGQAError) as e:
        p.run(dev["q"], dev["k_pool"], dev["v_pool"], out_dtype=torch.float16)
    assert e.value.name == "PGQA_ERR_UNSUPPORTED"
    buf = torch.zeros(w.q.numel() + 8, dtype=torch.bfloat16, device="cuda")
    q_mis = buf[1:1 + w.q.numel()].view(w.q.shape)
    q_mis.copy_(dev["q"])
    with pytest.raises(pg.PagedGQAError) as e:
        pg.run(p.handle, q_mis, dev["k_pool"], dev["v_pool"])
    assert e.value.name == "PGQA_ERR_INVALID_ARG"
