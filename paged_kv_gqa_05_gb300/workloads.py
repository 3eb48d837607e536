"""Seeded synthetic inputs for paged GQA decode attention.

This module builds inputs only; it holds none of the attention arithmetic and
is the one piece shared by the CUDA path's tests/benchmark and the CPU oracle.

Each workload restates, with N(0,1) data, the shapes the pages run:
  * "flashlet" README, benchmark paragraph: 128 sequences x 300-token prompts in
    pure decode on Qwen2.5-0.5B (14 query heads, 2 KV heads, head_dim 64, bf16)
    over a pool of 8192 pages;
  * "A library kernel for decode", section "What changed" / setup: Qwen2.5-1.5B in
    fp16 (12 query heads, 2 KV heads, head_dim 128), 256-slot pages, prompts drawn
    from {16, 64, 256, 1024, 4096} tokens plus 64..256 generated tokens, seed 0;
  * "flashlet" README, design bullets: one ragged call with qo_indptr lengths
    [512, 1, 1, ...] serving a chunked prefill and decode rows together.

Random draws use torch's CPU generator seeded per workload, in the order
lengths -> page permutation -> q -> k -> v (-> appended k, v).  Float samples
are fp32 N(0,1) cast to the 16-bit type with round-to-nearest-even.  Pool
pages no request references, and rows past last_page_len in a request's last
page, are filled with NaN so that any read outside the page table shows up
as NaN in the output.
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

TORCH_DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}
PROMPT_CHOICES = (16, 64, 256, 1024, 4096)


@dataclasses.dataclass
class Workload:
    name: str
    dtype: str                  # "bf16" | "fp16"
    page_size: int
    num_qo_heads: int
    num_kv_heads: int
    head_dim: int
    num_pages: int
    kv_lens: np.ndarray         # [B] int64, keys each request attends over
    kv_indptr: np.ndarray       # [B+1] int32
    kv_indices: np.ndarray      # [nnz] int32
    last_page_len: np.ndarray   # [B] int32
    qo_indptr: Optional[np.ndarray]  # [B+1] int32, None = one decode row per request
    causal: bool
    q: torch.Tensor             # [rows, Hq, d]
    k_pool: torch.Tensor        # [P, ps, Hkv, d]
    v_pool: torch.Tensor
    k_new: Optional[torch.Tensor] = None        # [T, Hkv, d] rows to append
    v_new: Optional[torch.Tensor] = None
    slot_mapping: Optional[np.ndarray] = None   # [T] int64 flat slot per appended row
    description: str = ""

    @property
    def batch(self) -> int:
        return len(self.kv_lens)

    @property
    def rows(self) -> int:
        return self.q.shape[0]

    @property
    def group(self) -> int:
        return self.num_qo_heads // self.num_kv_heads


def raw16(t: torch.Tensor) -> np.ndarray:
    """The 16-bit patterns of a bf16/fp16 tensor as a numpy uint16 array."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def _randn(gen: torch.Generator, shape, dtype: str, device="cpu") -> torch.Tensor:
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    return x.to(TORCH_DTYPES[dtype])


def page_table(kv_lens: np.ndarray, page_size: int, num_pages: int,
               gen: torch.Generator):
    """CSR page table over a seeded random permutation of the pool's pages."""
    npages = [(int(n) + page_size - 1) // page_size for n in kv_lens]
    nnz = sum(npages)
    if nnz > num_pages:
        raise ValueError(f"pool of {num_pages} pages cannot hold {nnz}")
    perm = torch.randperm(num_pages, generator=gen)[:nnz].numpy().astype(np.int32)
    kv_indptr = np.zeros(len(kv_lens) + 1, np.int32)
    kv_indptr[1:] = np.cumsum(npages)
    last = np.array([(int(n) - (p - 1) * page_size) if p > 0 else 0
                     for n, p in zip(kv_lens, npages)], np.int32)
    return kv_indptr, perm, last


def poison_pool(pool: torch.Tensor, kv_indptr: np.ndarray, kv_indices: np.ndarray,
                last_page_len: np.ndarray) -> None:
    """NaN over every page outside the table and every row past a last page's fill."""
    num_pages, page_size = pool.shape[0], pool.shape[1]
    used = torch.zeros(num_pages, dtype=torch.bool)
    if len(kv_indices):
        used[torch.from_numpy(kv_indices.astype(np.int64))] = True
    pool[~used.to(pool.device)] = float("nan")
    for b in range(len(last_page_len)):
        if kv_indptr[b + 1] > kv_indptr[b]:
            page = int(kv_indices[kv_indptr[b + 1] - 1])
            pool[page, int(last_page_len[b]):] = float("nan")


def make_pools(num_pages, page_size, num_kv_heads, head_dim, dtype, kv_indptr, kv_indices,
               last_page_len, gen: torch.Generator, device="cpu"):
    shape = (num_pages, page_size, num_kv_heads, head_dim)
    k_pool = _randn(gen, shape, dtype, device)
    v_pool = _randn(gen, shape, dtype, device)
    poison_pool(k_pool, kv_indptr, kv_indices, last_page_len)
    poison_pool(v_pool, kv_indptr, kv_indices, last_page_len)
    return k_pool, v_pool


def custom(name: str, kv_lens, page_size: int, num_qo_heads: int, num_kv_heads: int,
           head_dim: int, dtype: str, num_pages: int, seed: int = 0,
           qo_lens=None, causal: bool = False, append_last: bool = False,
           description: str = "") -> Workload:
    """Generic builder.  qo_lens=None gives one decode row per request.

    append_last=True models "cached history + one appended token": the page table
    covers kv_lens, the pool row of each request's final token is NaN before the
    append, and k_new / v_new / slot_mapping carry that token's rows.
    """
    gen = torch.Generator("cpu").manual_seed(seed)
    kv_lens = np.asarray(kv_lens, dtype=np.int64)
    kv_indptr, kv_indices, last = page_table(kv_lens, page_size, num_pages, gen)
    if qo_lens is None:
        qo_indptr = None
        rows = len(kv_lens)
    else:
        qo_indptr = np.zeros(len(kv_lens) + 1, np.int32)
        qo_indptr[1:] = np.cumsum(np.asarray(qo_lens, np.int64))
        rows = int(qo_indptr[-1])
    q = _randn(gen, (rows, num_qo_heads, head_dim), dtype)
    k_pool, v_pool = make_pools(num_pages, page_size, num_kv_heads, head_dim, dtype,
                                kv_indptr, kv_indices, last, gen)
    w = Workload(name, dtype, page_size, num_qo_heads, num_kv_heads, head_dim, num_pages,
                 kv_lens, kv_indptr, kv_indices, last, qo_indptr, causal, q, k_pool, v_pool,
                 description=description)
    if append_last:
        k_new = _randn(gen, (len(kv_lens), num_kv_heads, head_dim), dtype)
        v_new = _randn(gen, (len(kv_lens), num_kv_heads, head_dim), dtype)
        slots = np.full(len(kv_lens), -1, np.int64)
        for b, n in enumerate(kv_lens):
            if n == 0:
                continue
            page = int(kv_indices[kv_indptr[b] + (n - 1) // page_size])
            slots[b] = page * page_size + (n - 1) % page_size
            k_pool.view(-1, num_kv_heads, head_dim)[slots[b]] = float("nan")
            v_pool.view(-1, num_kv_heads, head_dim)[slots[b]] = float("nan")
        w.k_new, w.v_new, w.slot_mapping = k_new, v_new, slots
    return w


# ---------------------------------------------------------------------------
# The five workloads
# ---------------------------------------------------------------------------

def tiny(seed: int = 0) -> Workload:
    return custom("tiny", [1, 17, 64, 200], 16, 14, 2, 64, "bf16", 64, seed=seed,
                  description="batch 4, kv_len {1,17,64,200}, page 16, Hq14/Hkv2/d64, bf16, "
                              "pool 64 pages")


def qwen05_decode(seed: int = 0, batch: int = 128, cached: int = 300,
                  num_pages: int = 8192) -> Workload:
    return custom("qwen05_decode_128x300", [cached + 1] * batch, 16, 14, 2, 64, "bf16",
                  num_pages, seed=seed, append_last=True,
                  description=f"{batch} requests x {cached} cached tokens + 1 appended, page 16, "
                              f"Hq14/Hkv2/d64, bf16, pool {num_pages} pages")


def qwen15_mixed_lens(gen: torch.Generator, batch: int) -> np.ndarray:
    prompt_idx = torch.randint(0, len(PROMPT_CHOICES), (batch,), generator=gen)
    gen_len = torch.randint(64, 257, (batch,), generator=gen)
    return np.array([PROMPT_CHOICES[int(i)] + int(g) for i, g in zip(prompt_idx, gen_len)],
                    np.int64)


def qwen15_mixed(seed: int = 0, batch: int = 32, num_pages: int = 1024) -> Workload:
    gen = torch.Generator("cpu").manual_seed(seed)
    lens = qwen15_mixed_lens(gen, batch)
    # the lengths are drawn from their own stream; the rest of the workload uses seed+1
    return custom("qwen15_mixed", lens, 256, 12, 2, 128, "fp16", num_pages, seed=seed + 1,
                  description=f"{batch} requests, prompt in {{16,64,256,1024,4096}} + gen "
                              f"U[64,256], page 256, Hq12/Hkv2/d128, fp16, pool {num_pages}")


def long_context(seed: int = 0, batch: int = 1, kv_len: int = 32768,
                 num_pages: int = 1024) -> Workload:
    return custom(f"long_context_b{batch}", [kv_len] * batch, 256, 12, 2, 128, "bf16",
                  num_pages, seed=seed,
                  description=f"batch {batch} x kv_len {kv_len}, page 256, Hq12/Hkv2/d128, "
                              f"bf16, pool {num_pages}")


def ragged(seed: int = 0, n_decode: int = 127, chunk: int = 512, cached: int = 1024,
           num_pages: int = 8192) -> Workload:
    gen = torch.Generator("cpu").manual_seed(seed)
    dec = torch.randint(16, 4097, (n_decode,), generator=gen).numpy().astype(np.int64)
    lens = np.concatenate([[cached + chunk], dec])
    qo = [chunk] + [1] * n_decode
    return custom("ragged_prefill_decode", lens, 64, 14, 2, 64, "bf16", num_pages,
                  seed=seed + 1, qo_lens=qo, causal=True,
                  description=f"1 prefill segment of {chunk} rows over {cached}+{chunk} keys "
                              f"(causal) + {n_decode} decode rows kv_len U[16,4096], page 64, "
                              f"Hq14/Hkv2/d64, bf16, pool {num_pages}")


def wide_group(seed: int = 0, batch: int = 64, cached: int = 2048, num_pages: int = 8400) -> Workload:
    """A 16-wide query group (32 query heads over 2 kv heads, head_dim 128): the
    decode tile's two-n-tile form."""
    return custom(f"wide_group_{batch}x{cached}", [cached + 1] * batch, 16, 32, 2, 128, "bf16",
                  num_pages, seed=seed, append_last=True,
                  description=f"{batch} requests x {cached} cached tokens + 1 appended, page 16, "
                              f"Hq32/Hkv2/d128 (group 16), bf16, pool {num_pages} pages")


def prefill_chunk(seed: int = 0, chunk: int = 512, cached: int = 1024, num_pages: int = 8192) -> Workload:
    """The ragged workload's prompt chunk alone: one request of `chunk` causal query
    rows over its cached + own keys."""
    return custom(f"prefill_chunk_{chunk}x{cached + chunk}", [cached + chunk], 64, 14, 2, 64, "bf16", num_pages,
                  seed=seed + 3, qo_lens=[chunk], causal=True,
                  description=f"1 prefill segment of {chunk} rows over {cached}+{chunk} keys (causal), page 64, "
                              f"Hq14/Hkv2/d64, bf16, pool {num_pages}")


WORKLOADS = {
    "tiny": tiny,
    "qwen05_decode": qwen05_decode,
    "qwen15_mixed": qwen15_mixed,
    "long_context_b1": lambda seed=0: long_context(seed, batch=1),
    "long_context_b4": lambda seed=0: long_context(seed, batch=4),
    "ragged": ragged,
    "wide_group": wide_group,
    "prefill_chunk": prefill_chunk,
}


def make(name: str, seed: int = 0) -> Workload:
    return WORKLOADS[name](seed)


def row_positions(w: Workload) -> np.ndarray:
    """Key position of each query row's own token: the last L positions of a request
    with N keys and L rows are N - L .. N - 1 (int32, one per row)."""
    pos = np.zeros(w.rows, np.int32)
    for b in range(w.batch):
        r0, r1 = (b, b + 1) if w.qo_indptr is None else (int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))
        pos[r0:r1] = int(w.kv_lens[b]) - (r1 - r0) + np.arange(r1 - r0)
    return pos


def algorithmic_flops(w: Workload) -> int:
    """Multiply-adds of the attention counted as 2 flops each: q.k and p.v over every
    admissible (query row, head, key) triple, 4 d flops per triple."""
    triples = 0
    for b in range(w.batch):
        r0, r1 = (b, b + 1) if w.qo_indptr is None else (int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))
        n, L = int(w.kv_lens[b]), r1 - r0
        for i in range(L):
            triples += max(0, min(n, n - L + i + 1)) if w.causal else n
    return triples * w.num_qo_heads * 4 * w.head_dim


def algorithmic_bytes(w: Workload, out_elem_bytes: int = 2) -> dict:
    """Bytes a paged decode call must move at minimum: the K/V rows attended
    (counted once per KV head even though a query group shares them), q, the
    output, and the page table entries read."""
    elem = 2
    kv = int(w.kv_lens.sum()) * 2 * w.num_kv_heads * w.head_dim * elem
    q = w.rows * w.num_qo_heads * w.head_dim * elem
    o = w.rows * w.num_qo_heads * w.head_dim * out_elem_bytes
    pt = 4 * (len(w.kv_indptr) + len(w.kv_indices) + len(w.last_page_len))
    if w.qo_indptr is not None:
        pt += 4 * len(w.qo_indptr)
    pages_touched = int(w.kv_indptr[-1])
    kv_pages = pages_touched * w.page_size * 2 * w.num_kv_heads * w.head_dim * elem
    return {"kv": kv, "q": q, "o": o, "page_table": pt, "total": kv + q + o + pt,
            "kv_whole_pages": kv_pages}
