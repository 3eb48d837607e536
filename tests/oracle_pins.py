"""Pins of the CPU oracle against things other than itself.

Every ``pin_*`` function takes an ``oracle.Oracle`` and raises AssertionError
when the oracle disagrees with:
  * a library routine (torch scaled_dot_product_attention / logsumexp in fp64,
    torch index_copy_, numpy / torch 16-bit float decoding),
  * a closed form (one key, identical keys, zero query, two keys),
  * an invariant of the method (page permutation, unpaged layout, split + LSE
    merge equals the unsplit result, causal rows equal decode over a prefix).

They run on the real oracle in test_oracle_pins.py and on deliberately broken
copies of it in test_oracle_mutants.py, which checks that every planted mistake
fails at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from paged_kv_gqa_05_gb300 import workloads as W

TOL = 1e-12


def _f64(t: torch.Tensor) -> torch.Tensor:
    return t.to(torch.float64)


def dense_kv(w: W.Workload, b: int):
    """The request's pages concatenated in table order, first kv_len rows: [N, Hkv, d]."""
    pages = torch.from_numpy(w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]].astype(np.int64))
    n = int(w.kv_lens[b])
    k = w.k_pool[pages].reshape(-1, w.num_kv_heads, w.head_dim)[:n]
    v = w.v_pool[pages].reshape(-1, w.num_kv_heads, w.head_dim)[:n]
    return k, v


def run(orc, w: W.Workload, scale: float = 0.0, causal=None, nthreads: int = 1):
    return orc.paged_attention(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                               w.kv_indptr, w.kv_indices, w.last_page_len, w.dtype,
                               qo_indptr=w.qo_indptr,
                               causal=w.causal if causal is None else causal,
                               scale=scale, nthreads=nthreads)


def _rows(w: W.Workload, b: int):
    if w.qo_indptr is None:
        return b, b + 1
    return int(w.qo_indptr[b]), int(w.qo_indptr[b + 1])


def sdpa_reference(w: W.Workload, scale: float | None = None):
    """torch fp64 SDPA per request on the gathered K/V, heads grouped with
    repeat_interleave (query head h reads kv head h // g).  Decode rows only,
    or causal segments whose query count equals the key count (where torch's
    top-left causal alignment coincides with the bottom-right one)."""
    g = w.group
    outs = np.zeros((w.rows, w.num_qo_heads, w.head_dim))
    lses = np.zeros((w.rows, w.num_qo_heads))
    sc = 1.0 / math.sqrt(w.head_dim) if scale is None else scale
    for b in range(w.batch):
        r0, r1 = _rows(w, b)
        k, v = dense_kv(w, b)
        q = _f64(w.q[r0:r1]).permute(1, 0, 2).unsqueeze(0)            # [1, Hq, L, d]
        kk = _f64(k).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
        vv = _f64(v).permute(1, 0, 2).repeat_interleave(g, dim=0).unsqueeze(0)
        L, n = r1 - r0, k.shape[0]
        is_causal = bool(w.causal) and L > 1
        if is_causal:
            assert L == n, "library causal pin needs query count == key count"
        o = F.scaled_dot_product_attention(q, kk, vv, scale=sc, is_causal=is_causal)
        s = (q @ kk.transpose(-1, -2)) * sc
        if is_causal:
            s = s.masked_fill(torch.ones(L, n, dtype=torch.bool).triu(1), float("-inf"))
        lse = torch.logsumexp(s, dim=-1)
        outs[r0:r1] = o[0].permute(1, 0, 2).numpy()
        lses[r0:r1] = lse[0].permute(1, 0).numpy()
    return outs, lses


def _close(a, b, tol=TOL, what=""):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    assert not np.isnan(a).any(), f"{what}: NaN in oracle output"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    assert err <= tol, f"{what}: max abs diff {err:.3e} > {tol:.1e}"


# ---------------------------------------------------------------------------
# 16-bit decoding
# ---------------------------------------------------------------------------

def pin_widen_bf16(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = orc.widen(bits, "bf16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "bf16 NaN patterns"
    assert np.array_equal(got[~nan], ref[~nan]), "bf16 widening differs from torch"


def pin_widen_fp16(orc):
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = orc.widen(bits, "fp16")
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan), "fp16 NaN patterns"
    assert np.array_equal(got[~nan], ref[~nan]), "fp16 widening differs from numpy"


# ---------------------------------------------------------------------------
# attention against library routines
# ---------------------------------------------------------------------------

def _small(seed=0, dtype="bf16", Hq=6, Hkv=2, d=16, ps=4, lens=(1, 5, 8, 13), pages=32):
    return W.custom("pin", list(lens), ps, Hq, Hkv, d, dtype, pages, seed=seed)


def pin_sdpa_gqa_bf16(orc):
    w = _small(seed=1, dtype="bf16", Hq=6, Hkv=2, d=16, ps=4, lens=(1, 5, 8, 13, 30))
    o, lse = run(orc, w)
    ro, rl = sdpa_reference(w)
    _close(o, ro, what="out vs torch SDPA (bf16, g=3)")
    _close(lse, rl, what="lse vs torch logsumexp (bf16, g=3)")


def pin_sdpa_gqa_fp16(orc):
    w = _small(seed=2, dtype="fp16", Hq=8, Hkv=4, d=8, ps=8, lens=(3, 9, 16, 17))
    o, lse = run(orc, w)
    ro, rl = sdpa_reference(w)
    _close(o, ro, what="out vs torch SDPA (fp16, g=2)")
    _close(lse, rl, what="lse vs torch logsumexp (fp16, g=2)")


def pin_sdpa_mha(orc):
    w = _small(seed=3, dtype="bf16", Hq=3, Hkv=3, d=8, ps=2, lens=(2, 7))
    o, lse = run(orc, w)
    ro, rl = sdpa_reference(w)
    _close(o, ro, what="out vs torch SDPA (g=1)")
    _close(lse, rl, what="lse (g=1)")


def pin_sdpa_explicit_scale(orc):
    w = _small(seed=4, dtype="bf16", Hq=4, Hkv=1, d=16, ps=4, lens=(6, 11))
    o, lse = run(orc, w, scale=0.37)
    ro, rl = sdpa_reference(w, scale=0.37)
    _close(o, ro, what="out with explicit scale")
    _close(lse, rl, what="lse with explicit scale")


def pin_sdpa_causal_full_chunk(orc):
    """A causal segment that is the request's whole history (L == N): bottom-right
    and top-left alignment coincide, so torch's is_causal is the library pin."""
    w = W.custom("pin", [7, 1, 12], 4, 4, 2, 8, "bf16", 16, seed=5, qo_lens=[7, 1, 12],
                 causal=True)
    o, lse = run(orc, w)
    ro, rl = sdpa_reference(w)
    _close(o, ro, what="causal segment vs torch SDPA is_causal")
    _close(lse, rl, what="causal lse")


# ---------------------------------------------------------------------------
# closed forms
# ---------------------------------------------------------------------------

def pin_kv_len_one(orc):
    """One key: the softmax weight is exactly 1, so the output is that key's V row."""
    w = _small(seed=6, Hq=4, Hkv=2, d=16, ps=4, lens=(1, 1, 1))
    o, lse = run(orc, w)
    for b in range(w.batch):
        k, v = dense_kv(w, b)
        for h in range(w.num_qo_heads):
            kvh = h // w.group
            assert np.array_equal(o[b, h], _f64(v[0, kvh]).numpy()), "kv_len=1 must return V"
            s = float(np.dot(_f64(w.q[b, h]).numpy(), _f64(k[0, kvh]).numpy())) / 4.0
            assert abs(lse[b, h] - s) <= TOL, "kv_len=1 lse must be the scaled score"


def pin_identical_keys(orc):
    """All keys equal: uniform weights, output = mean of V, lse = s + log N."""
    w = _small(seed=7, Hq=4, Hkv=2, d=16, ps=4, lens=(5, 9))
    for b in range(w.batch):
        pages = w.kv_indices[w.kv_indptr[b]:w.kv_indptr[b + 1]]
        for p in pages:
            w.k_pool[int(p)] = w.k_pool[int(pages[0]), 0]
    o, lse = run(orc, w)
    for b in range(w.batch):
        k, v = dense_kv(w, b)
        n = k.shape[0]
        for h in range(w.num_qo_heads):
            kvh = h // w.group
            _close(o[b, h], _f64(v[:, kvh]).numpy().mean(axis=0), what="identical keys -> mean V")
            s = float(np.dot(_f64(w.q[b, h]).numpy(), _f64(k[0, kvh]).numpy())) / 4.0
            assert abs(lse[b, h] - (s + math.log(n))) <= TOL, "identical keys lse"


def pin_zero_query(orc):
    w = _small(seed=8, Hq=2, Hkv=1, d=8, ps=4, lens=(3, 10))
    w.q.zero_()
    o, lse = run(orc, w)
    for b in range(w.batch):
        _, v = dense_kv(w, b)
        for h in range(2):
            _close(o[b, h], _f64(v[:, 0]).numpy().mean(axis=0), what="q=0 -> mean V")
            assert abs(lse[b, h] - math.log(v.shape[0])) <= TOL, "q=0 lse = log N"


def pin_two_keys(orc):
    """Two keys: the weights are the logistic function of the score gap."""
    w = _small(seed=9, Hq=2, Hkv=1, d=8, ps=4, lens=(2,))
    o, lse = run(orc, w)
    k, v = dense_kv(w, 0)
    for h in range(2):
        qv = _f64(w.q[0, h]).numpy()
        s1 = float(np.dot(qv, _f64(k[0, 0]).numpy())) / math.sqrt(8)
        s2 = float(np.dot(qv, _f64(k[1, 0]).numpy())) / math.sqrt(8)
        a = 1.0 / (1.0 + math.exp(s2 - s1))
        ref = a * _f64(v[0, 0]).numpy() + (1.0 - a) * _f64(v[1, 0]).numpy()
        _close(o[0, h], ref, what="two-key logistic closed form")
        big = max(s1, s2)
        assert abs(lse[0, h] - (big + math.log1p(math.exp(min(s1, s2) - big)))) <= TOL


def pin_group_sharing(orc):
    """Heads of one group with the same q give the same output; the other group differs."""
    w = _small(seed=10, Hq=6, Hkv=2, d=16, ps=4, lens=(9,))
    w.q[0, 1] = w.q[0, 0]
    w.q[0, 2] = w.q[0, 0]
    w.q[0, 3] = w.q[0, 0]
    o, _ = run(orc, w)
    assert np.array_equal(o[0, 0], o[0, 1]) and np.array_equal(o[0, 0], o[0, 2])
    assert not np.allclose(o[0, 0], o[0, 3]), "a head of the next group must read the next kv head"


# ---------------------------------------------------------------------------
# invariants of the paged layout and of split-KV
# ---------------------------------------------------------------------------

def pin_page_permutation(orc):
    """Moving pages to other pool slots and remapping the table changes nothing."""
    w = _small(seed=11, Hq=4, Hkv=2, d=16, ps=4, lens=(3, 8, 13, 1), pages=24)
    o, lse = run(orc, w)
    perm = torch.randperm(w.num_pages, generator=torch.Generator().manual_seed(99))
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(w.num_pages)
    w2 = W.Workload(**{**w.__dict__})
    w2.k_pool = w.k_pool[perm].clone()
    w2.v_pool = w.v_pool[perm].clone()
    w2.kv_indices = inv.numpy()[w.kv_indices].astype(np.int32)
    o2, lse2 = run(orc, w2)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2), "page permutation changed the result"


def pin_unpaged_layout(orc):
    """The same keys stored contiguously (one page per request) give the same result."""
    w = _small(seed=12, Hq=4, Hkv=2, d=16, ps=4, lens=(3, 8, 13))
    o, lse = run(orc, w)
    maxn = int(w.kv_lens.max())
    kp = torch.full((w.batch, maxn, 2, 16), float("nan"), dtype=w.k_pool.dtype)
    vp = kp.clone()
    for b in range(w.batch):
        k, v = dense_kv(w, b)
        kp[b, :k.shape[0]] = k
        vp[b, :v.shape[0]] = v
    w2 = W.Workload(**{**w.__dict__})
    w2.k_pool, w2.v_pool, w2.page_size, w2.num_pages = kp, vp, maxn, w.batch
    w2.kv_indptr = np.arange(w.batch + 1, dtype=np.int32)
    w2.kv_indices = np.arange(w.batch, dtype=np.int32)
    w2.last_page_len = w.kv_lens.astype(np.int32)
    o2, lse2 = run(orc, w2)
    assert np.array_equal(o, o2) and np.array_equal(lse, lse2), "paged != unpaged"


def pin_split_merge(orc):
    """Partials over any cut of the keys (empty slices included), merged by
    log-sum-exp, equal the unsplit result."""
    w = _small(seed=13, Hq=4, Hkv=2, d=16, ps=4, lens=(1, 6, 19, 40))
    o, lse = run(orc, w)
    rng = np.random.default_rng(0)
    for b in range(w.batch):
        n = int(w.kv_lens[b])
        for h in range(w.num_qo_heads):
            cuts = np.sort(rng.integers(0, n + 1, size=3))
            bounds = [0, *cuts.tolist(), n, n]          # includes empty slices
            parts_o, parts_l = [], []
            for j0, j1 in zip(bounds[:-1], bounds[1:]):
                po, pl = orc.attention_partial(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                                               w.kv_indptr, w.kv_indices, w.last_page_len,
                                               w.dtype, b, b, h, j0, j1)
                parts_o.append(po)
                parts_l.append(pl)
            mo, ml = orc.lse_merge(np.stack(parts_o), np.array(parts_l))
            _close(mo, o[b, h], what="merge of split partials")
            assert abs(ml - lse[b, h]) <= TOL, "merged lse"
    # a single slice is the whole problem, and an all-empty merge is (0, -inf)
    mo, ml = orc.lse_merge(np.zeros((2, 16)), np.array([-np.inf, -np.inf]))
    assert ml == -np.inf and not mo.any()


def pin_causal_rows_are_prefix_decodes(orc):
    """Bottom-right causal: row i of an L-row segment over N keys equals a decode
    row over the first N - L + i + 1 keys, and the last row equals a full decode."""
    L, n = 5, 12
    w = W.custom("pin", [n, 4], 4, 4, 2, 8, "bf16", 16, seed=14, qo_lens=[L, 1], causal=True)
    o, lse = run(orc, w)
    for i in range(L):
        m = n - L + i + 1
        npg = (m + 3) // 4
        w2 = W.Workload(**{**w.__dict__})
        w2.kv_indptr = np.array([0, npg], np.int32)
        w2.kv_indices = w.kv_indices[:npg].copy()
        w2.last_page_len = np.array([m - (npg - 1) * 4], np.int32)
        w2.kv_lens = np.array([m])
        w2.qo_indptr = None
        w2.q = w.q[i:i + 1].clone()
        w2.causal = False
        w2.k_pool = w.k_pool.clone()
        w2.v_pool = w.v_pool.clone()
        o2, lse2 = run(orc, w2)
        assert np.array_equal(o[i], o2[0]) and np.array_equal(lse[i], lse2[0]), f"row {i}"
    # decode rows are unaffected by the causal flag
    o_nc, _ = run(orc, w, causal=False)
    assert np.array_equal(o[L], o_nc[L])


def pin_nan_poison_unread(orc):
    """The seeded pools hold NaN outside the page table; the oracle never reads it."""
    w = W.tiny()
    o, lse = run(orc, w)
    assert not np.isnan(o).any() and not np.isnan(lse).any()


def pin_kv_append(orc):
    """The append equals torch's index_copy_ of the rows into the flat slots."""
    w = _small(seed=15, Hq=4, Hkv=2, d=16, ps=4, lens=(5, 9))
    gen = torch.Generator().manual_seed(3)
    T = 6
    k = torch.randn(T, 2, 16, generator=gen).to(torch.bfloat16)
    v = torch.randn(T, 2, 16, generator=gen).to(torch.bfloat16)
    slots = torch.tensor([5, 0, 77, -1, 40, 127], dtype=torch.int64)
    kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
    orc.kv_append(kp, vp, W.raw16(k), W.raw16(v), slots.numpy())
    keep = slots >= 0
    rk = w.k_pool.reshape(-1, 2, 16).clone().index_copy_(0, slots[keep], k[keep])
    rv = w.v_pool.reshape(-1, 2, 16).clone().index_copy_(0, slots[keep], v[keep])
    assert np.array_equal(kp.reshape(-1), W.raw16(rk).reshape(-1)), "append K"
    assert np.array_equal(vp.reshape(-1), W.raw16(rv).reshape(-1)), "append V"


def pin_page_table_checks(orc):
    ok = orc.check_page_table([0, 2, 3], [0, 5, 1], [4, 1], 8, 4)
    assert ok == 0
    assert orc.check_page_table([0, 2, 3], [0, 8, 1], [4, 1], 8, 4) != 0, "index >= pool"
    assert orc.check_page_table([0, 2, 3], [0, 5, 1], [5, 1], 8, 4) != 0, "last_page_len > ps"
    assert orc.check_page_table([0, 2, 3], [0, 5, 1], [0, 1], 8, 4) != 0, "last_page_len 0"
    assert orc.check_page_table([0, 2, 1], [0, 5, 1], [4, 1], 8, 4) != 0, "indptr not monotone"
    assert orc.check_page_table([0, 0, 1], [3], [0, 2], 8, 4) == 0, "empty request"
    assert orc.check_page_table([0, 0, 1], [3], [1, 2], 8, 4) != 0, "no pages but last_page_len 1"
    assert orc.check_page_table([0, 2, 3], [0, -1, 1], [4, 1], 8, 4) != 0, "negative index"
    assert orc.check_page_table([0, 2, 3], [0, 7, 1], [4, 1], 8, 4) == 0, "last page of the pool"


def pin_empty_request(orc):
    """A request with no pages attends over nothing: o = 0, lse = -inf."""
    w = W.custom("pin", [0, 3], 4, 2, 1, 8, "bf16", 8, seed=16)
    o, lse = run(orc, w)
    assert not o[0].any() and np.all(lse[0] == -np.inf)
    assert np.isfinite(lse[1]).all()


# ---------------------------------------------------------------------------
# rounding to the 16-bit types (used by the rotary embedding)
# ---------------------------------------------------------------------------

def _grid(dtype):
    """Every finite non-negative 16-bit value (decoded by torch / numpy) with its pattern, ascending."""
    bits = np.arange(0x8000, dtype=np.uint16)  # sign bit clear
    if dtype == "bf16":
        vals = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    else:
        vals = bits.view(np.float16).astype(np.float64)
    keep = np.isfinite(vals)
    return vals[keep], bits[keep]


def nearest_even(x: np.ndarray, dtype: str) -> np.ndarray:
    """Brute-force round to nearest, ties to the even pattern, over the whole grid of
    finite values; |x| at or past the largest value plus half its spacing is infinity."""
    vals, bits = _grid(dtype)
    top, gap = vals[-1], vals[-1] - vals[-2]
    inf = np.uint16(0x7F80 if dtype == "bf16" else 0x7C00)
    out = np.empty(x.shape, np.uint16)
    for k, xv in enumerate(np.asarray(x, np.float64).ravel()):
        a = abs(xv)
        sign = np.uint16(0x8000) if np.signbit(xv) else np.uint16(0)
        if a >= top + gap / 2:
            out.flat[k] = sign | inf
            continue
        j = int(np.searchsorted(vals, a))
        cands = [c for c in (j - 1, j) if 0 <= c < len(vals)]
        dist = [abs(vals[c] - a) for c in cands]
        best = [c for c, dd in zip(cands, dist) if dd == min(dist)]
        pick = best[0] if len(best) == 1 else next(c for c in best if bits[c] % 2 == 0)
        out.flat[k] = sign | bits[pick]
    return out


def _narrow_cases(dtype, seed):
    """Random magnitudes over the whole range (subnormals and overflow included), exact
    ties between neighbours, and values just past a tie that binary32 would round onto
    the tie (a two-step rounding through binary32 lands on the wrong side)."""
    rng = np.random.default_rng(seed)
    vals, _ = _grid(dtype)
    lo, hi = (-136, 129) if dtype == "bf16" else (-26, 17)
    rand = np.ldexp(1.0 + rng.random(400), rng.integers(lo, hi, 400)) * rng.choice([-1.0, 1.0], 400)
    k = rng.integers(0, len(vals) - 1, 300)
    ties = (vals[k] + vals[k + 1]) / 2
    k2 = rng.integers(1, len(vals) - 1, 300)
    mids = (vals[k2] + vals[k2 + 1]) / 2
    traps = np.concatenate([mids * (1 + 2.0 ** -33), mids * (1 - 2.0 ** -33)])
    top, gap = vals[-1], vals[-1] - vals[-2]
    edges = np.array([0.0, -0.0, top, top + gap / 2, top + gap / 2 * (1 - 2.0 ** -40), vals[1] / 2,
                      vals[1] / 2 * (1 + 2.0 ** -30), vals[1] * 0.75, 1.0, -1.0, np.inf, -np.inf])
    return np.concatenate([rand, ties, -ties, traps, edges])


def pin_narrow_bf16(orc):
    x = _narrow_cases("bf16", 1)
    assert np.array_equal(orc.narrow(x, "bf16"), nearest_even(x, "bf16")), "bf16 rounding"


def pin_narrow_fp16(orc):
    x = _narrow_cases("fp16", 2)
    got = orc.narrow(x, "fp16")
    assert np.array_equal(got, nearest_even(x, "fp16")), "fp16 rounding (brute force)"
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, ref), "fp16 rounding (numpy)"


# ---------------------------------------------------------------------------
# rotary position embedding
# ---------------------------------------------------------------------------

def _rand16(shape, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    t = torch.randn(*shape, generator=gen).to(W.TORCH_DTYPES[dtype])
    return W.raw16(t).reshape(shape)


def pin_rope_position_zero(orc):
    """At position 0 every angle is 0: the rotation is the identity, bit for bit."""
    for dt in ("bf16", "fp16"):
        x = _rand16((5, 3, 64), dt, 4)
        out16, _ = orc.rope(x, np.zeros(5, np.int32), 1.0e6, dt)
        assert np.array_equal(out16, x), dt


def pin_rope_unit_vectors(orc):
    """Unit vector e_i (i < d/2) at position p turns into cos(phi) e_i + sin(phi) e_(i+d/2),
    and e_(i+d/2) into cos(phi) e_(i+d/2) - sin(phi) e_i, phi = p * theta^(-2i/d): which
    channels pair, which way they turn and how fast each pair turns."""
    d, theta = 16, 1.0e4
    pos = np.array([1, 7, 300, 40001], np.int32)
    for i in range(d // 2):
        for second in (False, True):
            x = np.zeros((len(pos), 1, d))
            x[:, 0, i + (d // 2 if second else 0)] = 1.0
            y = orc.rope_f64(x, pos, theta)
            phi = pos.astype(np.float64) * np.power(theta, -2.0 * i / d)
            ref = np.zeros_like(x)
            if second:
                ref[:, 0, i], ref[:, 0, i + d // 2] = -np.sin(phi), np.cos(phi)
            else:
                ref[:, 0, i], ref[:, 0, i + d // 2] = np.cos(phi), np.sin(phi)
            _close(y, ref, 1e-9, f"unit vector {i} second={second}")


def pin_rope_relative_position(orc):
    """The defining property: q.k after rotating q to m and k to n depends on m - n only."""
    rng = np.random.default_rng(5)
    q, k = rng.standard_normal((1, 4, 64)), rng.standard_normal((1, 4, 64))
    def dot(m, n):
        return np.sum(orc.rope_f64(q, np.array([m], np.int32), 1.0e6) *
                      orc.rope_f64(k, np.array([n], np.int32), 1.0e6), axis=-1)
    base = dot(40, 13)
    for t in (1, 977, 30000):
        _close(dot(40 + t, 13 + t), base, 1e-9, f"shift {t}")
    _close(dot(77, 77), np.sum(q * k, axis=-1), 1e-9, "equal positions")


def pin_rope_composition(orc):
    """Rotating to p1 and then by p2 equals rotating to p1 + p2."""
    rng = np.random.default_rng(6)
    x = rng.standard_normal((3, 2, 32))
    p1, p2 = np.array([5, 1000, 31], np.int32), np.array([2, 65, 12345], np.int32)
    two = orc.rope_f64(orc.rope_f64(x, p1, 1.0e6), p2, 1.0e6)
    _close(two, orc.rope_f64(x, p1 + p2, 1.0e6), 1e-9, "composition")


def pin_rope_pair_norms(orc):
    """Each (i, i + d/2) pair keeps its length."""
    rng = np.random.default_rng(7)
    x = rng.standard_normal((6, 3, 128))
    y = orc.rope_f64(x, np.array([0, 1, 9, 500, 8191, 32767], np.int32), 1.0e6)
    h = 64
    _close(np.hypot(y[..., :h], y[..., h:]), np.hypot(x[..., :h], x[..., h:]), 1e-12, "pair norms")


def pin_rope_rounding(orc):
    """The 16-bit result is the fp64 rotation rounded once, to nearest even."""
    for dt in ("bf16", "fp16"):
        x = _rand16((4, 2, 64), dt, 8)
        out16, out64 = orc.rope(x, np.array([3, 100, 4096, 30001], np.int32), 1.0e6, dt)
        assert np.array_equal(out16, nearest_even(out64, dt)), dt
        _close(out64, orc.rope_f64(orc.widen(x, dt), np.array([3, 100, 4096, 30001], np.int32), 1.0e6),
               0.0, f"{dt} widen-then-rotate")


PINS = {name: fn for name, fn in globals().items() if name.startswith("pin_")}
