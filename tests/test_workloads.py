"""CPU tests of the seeded input recipe: each workload has the shapes, lengths, page
tables and poison the pages' workloads call for, and the byte count behind the
benchmark's GB/s is the plain sum of what a call must read and write."""
import numpy as np
import pytest
import torch

from paged_kv_gqa_05_gb300 import workloads as W


def table_ok(w):
    """CSR page table over distinct pool pages; kv_len from the last page's fill."""
    npages = np.diff(w.kv_indptr)
    assert w.kv_indptr[0] == 0 and np.all(npages >= 0)
    assert len(w.kv_indices) == w.kv_indptr[-1]
    assert np.all((w.kv_indices >= 0) & (w.kv_indices < w.num_pages))
    assert len(np.unique(w.kv_indices)) == len(w.kv_indices), "a page serves two requests"
    lens = np.where(npages == 0, 0, (npages - 1) * w.page_size + w.last_page_len)
    assert np.array_equal(lens, w.kv_lens)
    assert np.all((npages == 0) == (w.last_page_len == 0))
    assert np.all(w.last_page_len <= w.page_size)


def poison_ok(w):
    """NaN everywhere outside the table; finite on every attended row except the slots
    the step's append writes."""
    for pool in (w.k_pool, w.v_pool):
        finite = torch.isfinite(pool.float()).all(dim=(2, 3)).numpy()  # [pages, page_size]
        nan = torch.isnan(pool.float()).all(dim=(2, 3)).numpy()
        used = np.zeros(finite.shape, bool)
        for b in range(w.batch):
            n = int(w.kv_lens[b])
            for j in range(n):
                used[w.kv_indices[w.kv_indptr[b] + j // w.page_size], j % w.page_size] = True
        appended = np.zeros(finite.shape, bool)
        if w.slot_mapping is not None:
            s = w.slot_mapping[w.slot_mapping >= 0]
            appended[s // w.page_size, s % w.page_size] = True
        assert np.all(nan[~used]), "a row outside the table is not NaN"
        assert np.all(finite[used & ~appended]), "an attended row is not finite"
        assert np.all(nan[appended]), "a row the append writes is not poisoned"


def test_tiny():
    w = W.tiny()
    assert list(w.kv_lens) == [1, 17, 64, 200]
    assert list(np.diff(w.kv_indptr)) == [1, 2, 4, 13] and list(w.last_page_len) == [1, 1, 16, 8]
    assert (w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype, w.num_pages) == \
        (16, 14, 2, 64, "bf16", 64)
    table_ok(w)
    poison_ok(w)


def test_qwen05_decode_step():
    """128 requests of 300 cached tokens, each appending its 301st (position 300) and
    attending over all 301: 19 pages of 16, the last holding 13 rows."""
    w = W.qwen05_decode()
    assert w.batch == 128 and w.rows == 128 and np.all(w.kv_lens == 301)
    assert np.all(np.diff(w.kv_indptr) == 19) and np.all(w.last_page_len == 13)
    assert (w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype, w.num_pages) == \
        (16, 14, 2, 64, "bf16", 8192)
    last_pages = w.kv_indices[w.kv_indptr[1:] - 1]
    assert np.array_equal(w.slot_mapping, last_pages.astype(np.int64) * 16 + 12), "append slot = position 300"
    assert w.k_new.shape == (128, 2, 64) and w.qo_indptr is None and not w.causal
    table_ok(w)
    poison_ok(w)
    # bytes of one layer call: K/V rows attended, q, out (bf16) and the page-table words read
    a = W.algorithmic_bytes(w)
    assert a["kv"] == 128 * 301 * 2 * 2 * 64 * 2 == 19_726_336
    assert a["q"] == a["o"] == 128 * 14 * 64 * 2 == 229_376
    assert a["page_table"] == 4 * (129 + 128 * 19 + 128) == 10_756
    assert a["total"] == 19_726_336 + 2 * 229_376 + 10_756
    assert a["kv_whole_pages"] == 128 * 19 * 16 * 2 * 2 * 64 * 2


def test_qwen15_mixed_lengths():
    """Prompt lengths from {16, 64, 256, 1024, 4096} plus 64..256 generated tokens."""
    w = W.qwen15_mixed()
    allowed = {p + g for p in W.PROMPT_CHOICES for g in range(64, 257)}
    assert w.batch == 32 and set(w.kv_lens.tolist()) <= allowed
    assert (w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype, w.num_pages) == \
        (256, 12, 2, 128, "fp16", 1024)
    table_ok(w)
    # a long draw reaches both ends: the shortest prompt with few generated tokens and
    # the longest prompt with many
    lens = W.qwen15_mixed_lens(torch.Generator("cpu").manual_seed(0), 4000)
    assert set(lens.tolist()) <= allowed
    assert lens.min() < 16 + 100 and lens.max() > 4096 + 220


@pytest.mark.parametrize("batch", [1, 4])
def test_long_context(batch):
    w = W.make(f"long_context_b{batch}")
    assert w.batch == batch and np.all(w.kv_lens == 32768)
    assert np.all(np.diff(w.kv_indptr) == 128) and np.all(w.last_page_len == 256)
    assert (w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype) == (256, 12, 2, 128, "bf16")
    table_ok(w)
    assert W.algorithmic_bytes(w)["kv"] == batch * 32768 * 2 * 2 * 128 * 2


def test_ragged_call():
    """One 512-row causal chunk over 1024 cached + its own 512 keys, then 127 decode rows:
    qo_indptr is the prefix sum of the lengths [512, 1, 1, ...]."""
    w = W.ragged()
    assert w.batch == 128 and w.causal
    assert np.array_equal(w.qo_indptr, np.concatenate([[0], 512 + np.arange(128)]))
    assert w.kv_lens[0] == 1536 and np.all((w.kv_lens[1:] >= 16) & (w.kv_lens[1:] <= 4096))
    assert (w.page_size, w.num_qo_heads, w.num_kv_heads, w.head_dim, w.dtype) == (64, 14, 2, 64, "bf16")
    table_ok(w)
    # the chunk's causal (row, key) pairs per head: sum over i of 1024 + i + 1
    decode = int(w.kv_lens[1:].sum())
    assert W.algorithmic_flops(w) == (512 * 1024 + 512 * 513 // 2 + decode) * 14 * 4 * 64


def test_prefill_chunk_flops():
    """655,616 causal (row, key) pairs per head: 2.35 GFLOP for the chunk."""
    w = W.prefill_chunk()
    assert w.batch == 1 and w.rows == 512 and int(w.kv_lens[0]) == 1536 and w.causal
    assert W.algorithmic_flops(w) == 655_616 * 14 * 4 * 64 == 2_349_727_744


def test_wide_group():
    w = W.wide_group()
    assert w.batch == 64 and np.all(w.kv_lens == 2049) and w.group == 16 and w.head_dim == 128
    table_ok(w)


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_seeded(name):
    """The same seed gives the same inputs; another seed gives other values."""
    a, b, c = W.make(name, 0), W.make(name, 0), W.make(name, 1)
    assert np.array_equal(a.kv_indices, b.kv_indices) and np.array_equal(W.raw16(a.q), W.raw16(b.q))
    assert np.array_equal(W.raw16(a.k_pool), W.raw16(b.k_pool))
    assert not np.array_equal(W.raw16(a.q), W.raw16(c.q))
