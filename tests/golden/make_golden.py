"""Writes tests/golden/tiny_decode.json from the CPU oracle alone.

No page prints a worked numeric example for paged GQA decode, so this fixture
is a regression guard, not an independent pin: it stores the oracle's fp64
output for the seeded tiny workload (batch 4, kv_len {1,17,64,200}, page 16,
Hq 14 / Hkv 2 / d 64, bf16 -- the first workload of the "flashlet" README's
shape family) together with a digest of the generated inputs, so that a
silent change to the input generator or to the oracle shows up as a diff.

Run:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from paged_kv_gqa_05_gb300 import workloads as W  # noqa: E402


def input_digest(w):
    h = hashlib.sha256()
    for a in (W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool), w.kv_indptr, w.kv_indices,
              w.last_page_len):
        h.update(a.tobytes())
    return h.hexdigest()


def main():
    w = W.tiny(seed=0)
    out, lse = oracle.get().paged_attention(W.raw16(w.q), W.raw16(w.k_pool), W.raw16(w.v_pool),
                                            w.kv_indptr, w.kv_indices, w.last_page_len, "bf16")
    rec = {
        "source": "CPU fp64 oracle (oracle/pgqa_oracle.c) on workloads.tiny(seed=0)",
        "input_sha256": input_digest(w),
        "kv_indptr": w.kv_indptr.tolist(),
        "last_page_len": w.last_page_len.tolist(),
        "lse": [[float(x) for x in row] for row in lse],
        "out_row_head_sums": [[float(x) for x in row] for row in out.sum(axis=2)],
        "out_first_channels": [[float(x) for x in row] for row in out[:, :, :4].reshape(4, -1)],
    }
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_decode.json")
    with open(path, "w") as f:
        json.dump(rec, f, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
