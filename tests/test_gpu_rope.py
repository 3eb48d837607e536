"""GPU: the rotary position embedding on the append path -- pgqa_kv_append_rope, and
pgqa_append_run / pgqa_run with a RoPE plan -- against the CPU oracle's fp64
rotation, rounded once to the 16-bit type, followed by its append and attention.

Rotated 16-bit values are checked against the rounding bound of the fp32 rotation:
the kernels compute a*cos - b*sin (and b*cos + a*sin) in fp32 with cos/sin rounded
to fp32, within eps = 2^-22 (|a| + |b|) of the exact value v, so each stored value
must lie between RNE(v - eps) and RNE(v + eps) (round to nearest even is monotone);
it equals RNE(v) except where v sits within eps of a rounding midpoint.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_05_gb300 as pg
from paged_kv_gqa_05_gb300 import workloads as W
import gpu_helpers as H

pytestmark = pytest.mark.gpu

THETA = 1.0e6
MAX_POS = 32768


def query_positions(w: W.Workload) -> np.ndarray:
    """Row r of a request with n keys and L rows sits at key position n - L + i."""
    pos = np.zeros(w.rows, np.int32)
    for b in range(w.batch):
        r0, r1 = (b, b + 1) if w.qo_indptr is None else (int(w.qo_indptr[b]), int(w.qo_indptr[b + 1]))
        n = int(w.kv_lens[b])
        pos[r0:r1] = n - (r1 - r0) + np.arange(r1 - r0)
    return pos


def rope_oracle(w: W.Workload, theta: float = THETA):
    """Oracle out/lse with q and the new K rows rotated at their positions, plus the
    pools after the append and the rotated K rows (16-bit and fp64)."""
    orc = oracle.get()
    pos = query_positions(w)
    q16, _ = orc.rope(W.raw16(w.q), pos, theta, w.dtype)
    k16, k64 = orc.rope(W.raw16(w.k_new), pos, theta, w.dtype)
    kp, vp = W.raw16(w.k_pool).copy(), W.raw16(w.v_pool).copy()
    orc.kv_append(kp, vp, k16, W.raw16(w.v_new), w.slot_mapping)
    out, lse = orc.paged_attention(q16, kp, vp, w.kv_indptr, w.kv_indices, w.last_page_len, w.dtype,
                                   qo_indptr=w.qo_indptr, causal=w.causal, nthreads=H.NTHREADS)
    return out, lse, kp, vp, k16, k64


def check_rotated(got16: np.ndarray, ref16: np.ndarray, ref64: np.ndarray, x16: np.ndarray, dtype: str, what: str):
    """got16, ref16, ref64, x16: [..., d] rotated GPU bits, oracle bits, oracle fp64, input bits."""
    orc = oracle.get()
    d = x16.shape[-1]
    x = orc.widen(x16, dtype)
    mag = np.abs(x) + np.abs(np.concatenate([x[..., d // 2:], x[..., :d // 2]], axis=-1))
    eps = mag * 2.0 ** -22
    diff = np.argwhere(got16 != ref16)
    assert len(diff) <= max(4, got16.size // 200), f"{what}: {len(diff)} of {got16.size} values differ"
    for idx in map(tuple, diff):
        v, e = ref64[idx], eps[idx]
        lo = orc.widen(orc.narrow(np.array([v - e]), dtype), dtype)[0]
        hi = orc.widen(orc.narrow(np.array([v + e]), dtype), dtype)[0]
        g = orc.widen(np.array([got16[idx]], np.uint16), dtype)[0]
        assert lo <= g <= hi, f"{what}: element {idx}: {g!r} outside [{lo!r}, {hi!r}] (exact {v!r})"


def slot_rows(pool16: np.ndarray, slots: np.ndarray) -> np.ndarray:
    P, ps, Hkv, d = pool16.shape
    return pool16.reshape(P * ps, Hkv, d)[slots]


def rope_plan(w: W.Workload, **opts) -> pg.Plan:
    dt = W.TORCH_DTYPES[w.dtype]
    return pg.Plan(w.num_qo_heads, w.num_kv_heads, w.head_dim, w.page_size, dt, max_batch=max(1, w.batch),
                   max_q_rows=max(1, w.rows), rope_theta=THETA, rope_max_position=MAX_POS, **opts)


def fused_rope(w: W.Workload, pool_stable: bool = False, **opts):
    dev = H.to_device(w)
    plan = rope_plan(w, **opts)
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                causal=w.causal, kv_indices_host=w.kv_indices)
    out = torch.empty(dev["q"].shape, dtype=torch.float32, device="cuda")
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    plan.append_run(dev["k_new"], dev["v_new"], dev["q"], dev["k_pool"], dev["v_pool"], out=out, lse=lse,
                    pool_stable=pool_stable)
    torch.cuda.synchronize()
    plan.close()
    assert pg.read_device_flags() == 0
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), dev


def check_fused(w: W.Workload, what: str, **opts):
    ro, rl, kp, vp, k16, k64 = rope_oracle(w)
    out, lse, dev = fused_rope(w, **opts)
    H.compare(out, lse, ro, rl, what)
    gk, gv = W.raw16(dev["k_pool"]), W.raw16(dev["v_pool"])
    check_rotated(slot_rows(gk, w.slot_mapping), k16, k64, W.raw16(w.k_new), w.dtype, what + " K rows")
    assert np.array_equal(slot_rows(gv, w.slot_mapping), W.raw16(w.v_new)), what + ": V rows are not rotated"
    untouched = np.ones(gk.shape[0] * gk.shape[1], bool)
    untouched[w.slot_mapping] = False
    P, ps, Hkv, d = gk.shape
    same = lambda a, b: np.array_equal(a.reshape(P * ps, Hkv, d)[untouched].view(np.uint16),
                                       b.reshape(P * ps, Hkv, d)[untouched].view(np.uint16))
    assert same(gk, kp) and same(gv, vp), what + ": rows other than the new ones changed"


@pytest.mark.parametrize("opts", [{}, {"split_tokens": 64}, {"pipeline_stages": 3}])
@pytest.mark.parametrize("pool_stable", [False, True])
def test_rope_decode_step(opts, pool_stable):
    """The 128 x 300-style decode step (smaller batch) with RoPE; forced splits put the
    new row in the last slice of several; the 3-stage ring form as well as the plan's choice."""
    w = W.qwen05_decode(batch=32, cached=300, num_pages=1024)
    check_fused(w, f"rope decode {opts} stable={pool_stable}", pool_stable=pool_stable, **opts)


@pytest.mark.parametrize("head_dim,page_size,dtype,hq,hkv", [
    (64, 16, "bf16", 14, 2), (128, 256, "fp16", 12, 2), (128, 32, "bf16", 32, 2), (64, 64, "fp16", 2, 2),
    (128, 16, "bf16", 16, 1)])
def test_rope_shapes(head_dim, page_size, dtype, hq, hkv):
    """Both head dims and types, groups 1..16, positions from 0 (identity) to past 30000."""
    lens = [1, 2, 17, 300, 1025, 30001]
    pages = sum(-(-n // page_size) for n in lens) + 8
    w = W.custom("rope", lens, page_size, hq, hkv, head_dim, dtype, pages, seed=head_dim + hq + page_size)
    H.new_rows_for_query_rows(w)
    check_fused(w, f"rope d{head_dim} ps{page_size} {dtype} {hq}/{hkv}", split_tokens=256)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("head_dim,group", [(64, 7), (128, 6), (128, 16)])
@pytest.mark.parametrize("prefill_kernel", ["tcgen05", "mma_sync"])
def test_rope_prefill_segments(causal, head_dim, group, prefill_kernel):
    """Multi-row requests (prefill tiles): each query row and each new K row turns at its
    own position."""
    lens, qo = [300, 5, 1030, 77, 3], [70, 1, 200, 77, 3]
    w = W.custom("ropepf", lens, 64, group * 2, 2, head_dim, "bf16", 64, seed=group + head_dim,
                 qo_lens=qo, causal=causal)
    H.new_rows_for_query_rows(w)
    check_fused(w, f"rope prefill g{group} d{head_dim} causal={causal} {prefill_kernel}",
                prefill_kernel=prefill_kernel)


def test_two_step_equals_fused():
    """pgqa_kv_append_rope followed by pgqa_run (q rotated by run) gives the fused
    call's output bit for bit, and the oracle's within tolerance."""
    w = W.custom("rope2", [5, 64, 300, 999], 16, 14, 2, 64, "bf16", 96, seed=31, qo_lens=[1, 3, 1, 12],
                 causal=True)
    H.new_rows_for_query_rows(w)
    ro, rl, *_ = rope_oracle(w)
    fo, fl, _ = fused_rope(w)
    dev = H.to_device(w)
    plan = rope_plan(w)
    plan.kv_append_rope(dev["k_pool"], dev["v_pool"], dev["k_new"], dev["v_new"], dev["slot_mapping"],
                        torch.from_numpy(query_positions(w)).cuda())
    plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                causal=True, kv_indices_host=w.kv_indices)
    lse = torch.empty(dev["q"].shape[:2], dtype=torch.float32, device="cuda")
    out = plan.run(dev["q"], dev["k_pool"], dev["v_pool"], out_dtype=torch.float32, lse=lse)
    torch.cuda.synchronize()
    plan.close()
    assert pg.read_device_flags() == 0
    o2, l2 = out.double().cpu().numpy(), lse.double().cpu().numpy()
    H.compare(o2, l2, ro, rl, "two-step rope")
    assert np.array_equal(o2, fo) and np.array_equal(l2, fl), "two-step and fused results differ"


@pytest.mark.parametrize("head_dim,dtype", [(64, "bf16"), (128, "fp16")])
def test_kv_append_rope(head_dim, dtype):
    """The standalone append: K rotated at each token's position, V copied; a row with a
    position outside the table is skipped (K and V) and flagged."""
    gen = torch.Generator().manual_seed(head_dim)
    T, Hkv, P, ps = 300, 2, 64, 16
    dt = W.TORCH_DTYPES[dtype]
    k = torch.randn(T, Hkv, head_dim, generator=gen).to(dt)
    v = torch.randn(T, Hkv, head_dim, generator=gen).to(dt)
    slots = torch.randperm(P * ps, generator=gen)[:T].to(torch.int64)
    pos = torch.randint(0, MAX_POS, (T,), generator=gen, dtype=torch.int32)
    pos[:4] = torch.tensor([0, 1, MAX_POS - 1, 12345], dtype=torch.int32)
    pos[7] = MAX_POS       # past the table: skipped
    pos[9] = -1            # negative: skipped
    kp = torch.zeros(P, ps, Hkv, head_dim, dtype=dt)
    vp = torch.zeros(P, ps, Hkv, head_dim, dtype=dt)
    plan = pg.Plan(Hkv, Hkv, head_dim, ps, dt, 1, 1, rope_theta=THETA, rope_max_position=MAX_POS)
    dkp, dvp = kp.cuda(), vp.cuda()
    plan.kv_append_rope(dkp, dvp, k.cuda(), v.cuda(), slots.cuda(), pos.cuda())
    torch.cuda.synchronize()
    plan.close()
    assert pg.read_device_flags(clear=True) == pg.binding.FLAG_ROPE_POSITION
    ok = np.ones(T, bool)
    ok[[7, 9]] = False
    k16, k64 = oracle.get().rope(W.raw16(k)[ok], pos.numpy()[ok], THETA, dtype)
    gk, gv = W.raw16(dkp.cpu()), W.raw16(dvp.cpu())
    s = slots.numpy()
    check_rotated(slot_rows(gk, s[ok]), k16, k64, W.raw16(k)[ok], dtype, "kv_append_rope")
    assert np.array_equal(slot_rows(gk, s[ok])[0], W.raw16(k)[ok][0]), "position 0 is the identity"
    assert np.array_equal(slot_rows(gv, s[ok]), W.raw16(v)[ok])
    assert not slot_rows(gk, s[~ok]).any() and not slot_rows(gv, s[~ok]).any(), "skipped rows were written"


def test_rope_rejections():
    w = W.custom("rej", [2, 40], 16, 4, 2, 64, "bf16", 8, seed=1, qo_lens=[3, 1], causal=True)
    dev = H.to_device(w)
    plan = rope_plan(w)
    with pytest.raises(pg.PagedGQAError) as e:  # 3 query rows over 2 keys: no positions
        plan.update(w.kv_indptr, w.last_page_len, dev["kv_indices"], w.num_pages, qo_indptr=w.qo_indptr,
                    causal=True)
    assert e.value.name == "PGQA_ERR_INVALID_ARG"
    plan.close()
    w2 = W.custom("rej2", [50], 16, 4, 2, 64, "bf16", 8, seed=2)
    d2 = H.to_device(w2)
    p2 = pg.Plan(4, 2, 64, 16, torch.bfloat16, 1, 1, rope_theta=THETA, rope_max_position=49)
    with pytest.raises(pg.PagedGQAError) as e:  # key positions up to 49 with a 49-row table
        p2.update(w2.kv_indptr, w2.last_page_len, d2["kv_indices"], w2.num_pages)
    assert e.value.name == "PGQA_ERR_INVALID_ARG"
    p2.close()
    with pytest.raises(pg.PagedGQAError) as e:
        pg.Plan(4, 2, 64, 16, torch.bfloat16, 1, 1, decode_kernel="cuda_core", rope_theta=THETA,
                rope_max_position=64)
    assert e.value.name == "PGQA_ERR_UNSUPPORTED"
    p3 = pg.Plan(4, 2, 64, 16, torch.bfloat16, 1, 1)
    z = torch.zeros(1, 2, 64, dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros(8, 16, 2, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pg.PagedGQAError) as e:
        p3.kv_append_rope(pool, pool.clone(), z, z, torch.zeros(1, dtype=torch.int64, device="cuda"),
                          torch.zeros(1, dtype=torch.int32, device="cuda"))
    assert e.value.name == "PGQA_ERR_INVALID_ARG"
    p3.close()
