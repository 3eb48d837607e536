"""Regression guard: the oracle and the input generator still reproduce the
stored tiny-workload fixture (written by tests/golden/make_golden.py)."""
import json
import os

import numpy as np

import oracle
from paged_kv_gqa_05_gb300 import workloads as W
from golden.make_golden import input_digest

HERE = os.path.dirname(os.path.abspath(__file__))


def test_tiny_fixture():
    rec = json.load(open(os.path.join(HERE, "golden", "tiny_decode.json")))
    w = W.tiny(seed=0)
    assert input_digest(w) == rec["input_sha256"], "seeded input generator changed"
    out, lse = oracle.get().paged_attention(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                                            w.kv_indptr, w.kv_indices, w.last_page_len, "bf16")
    assert np.allclose(lse, rec["lse"], rtol=0, atol=1e-12)
    assert np.allclose(out.sum(axis=2), rec["out_row_head_sums"], rtol=0, atol=1e-12)
    assert np.allclose(out[:, :, :4].reshape(4, -1), rec["out_first_channels"], rtol=0, atol=1e-12)
