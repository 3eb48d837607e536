"""The boundary is a plain C ABI: a C11 program that includes include/pagedgqa.h
(compiled as C, warnings as errors) and links libpagedgqa.so asks for a schedule
through pgqa_plan_schedule and gets the same work list as the Python binding, and a
malformed table's status and message (no GPU needed)."""
import shutil
import subprocess

import numpy as np
import pytest
import torch

from paged_kv_gqa_05_gb300 import binding as B
from paged_kv_gqa_05_gb300 import build

ROOT = build.ROOT

CLIENT = r"""
#include <stdio.h>
#include <string.h>

#include "pagedgqa.h"

int main(void) {
    if (pgqa_abi_version() != PGQA_ABI_VERSION) return 10;
    pgqa_plan_config cfg;
    memset(&cfg, 0, sizeof cfg);
    cfg.num_qo_heads = 14;
    cfg.num_kv_heads = 2;
    cfg.head_dim = 64;
    cfg.page_size = 16;
    cfg.dtype = PGQA_BF16;
    cfg.max_batch = 3;
    cfg.max_q_rows = 3;
    cfg.split_tokens = 64;
    /* three requests of 40, 0 and 300 keys */
    const int32_t indptr[4] = {0, 3, 3, 22};
    const int32_t last[3] = {8, 0, 12};
    int32_t idx[22];
    for (int i = 0; i < 22; ++i) idx[i] = (i * 7) % 24;
    pgqa_schedule_info info;
    pgqa_status st = pgqa_plan_schedule(&cfg, 152, indptr, last, NULL, 3, idx, 24, 0, NULL, 0, NULL, 0, NULL, 0,
                                        &info);
    if (st != PGQA_OK) {
        fprintf(stderr, "%s: %s\n", pgqa_status_string(st), pgqa_last_error());
        return 11;
    }
    pgqa_slice slices[64];
    pgqa_merge merges[16];
    if (info.num_items > 64 || info.num_merge_tasks > 16) return 12;
    st = pgqa_plan_schedule(&cfg, 152, indptr, last, NULL, 3, idx, 24, 0, slices, 64, merges, 16, NULL, 0, &info);
    if (st != PGQA_OK) return 13;
    printf("info %d %d %d %d\n", info.num_items, info.num_merge_tasks, info.split_tokens, info.pipeline_stages);
    for (int i = 0; i < info.num_items; ++i)
        printf("slice %d %d %d %d %d\n", slices[i].q_row, slices[i].kv_head, slices[i].key_begin,
               slices[i].key_end, slices[i].partial_slot);
    for (int i = 0; i < info.num_merge_tasks; ++i)
        printf("merge %d %d %d %d\n", merges[i].q_row, merges[i].kv_head, merges[i].slot_base, merges[i].num_splits);
    /* a page index outside the pool */
    idx[5] = 24;
    st = pgqa_plan_schedule(&cfg, 152, indptr, last, NULL, 3, idx, 24, 0, NULL, 0, NULL, 0, NULL, 0, &info);
    printf("bad %s | %s\n", pgqa_status_string(st), pgqa_last_error());
    return 0;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs a C compiler")
def test_c_program_gets_the_binding_schedule(tmp_path):
    lib = build.build()
    src = tmp_path / "client.c"
    src.write_text(CLIENT)
    exe = tmp_path / "client"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{ROOT / 'include'}",
                    str(src), "-o", str(exe), f"-L{lib.parent}", "-lpagedgqa", f"-Wl,-rpath,{lib.parent}"],
                   check=True)
    lines = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.splitlines()

    idx = np.array([(i * 7) % 24 for i in range(22)], np.int32)
    py = B.plan_schedule(14, 2, 64, 16, torch.bfloat16, [0, 3, 3, 22], [8, 0, 12], idx, 24, max_batch=3,
                         max_q_rows=3, split_tokens=64)
    info = py["info"]
    assert lines[0] == (f"info {info['num_items']} {info['num_merge_tasks']} {info['split_tokens']} "
                        f"{info['pipeline_stages']}")
    want = [f"slice {s['q_row']} {s['kv_head']} {s['key_begin']} {s['key_end']} {s['partial_slot']}"
            for s in py["slices"]]
    want += [f"merge {m['q_row']} {m['kv_head']} {m['slot_base']} {m['num_splits']}" for m in py["merges"]]
    assert lines[1:-1] == want
    assert info["num_merge_tasks"] == 2  # the 300-key request is split for both kv heads
    assert lines[-1].startswith("bad malformed page table | kv_indices[5] = 24 outside [0, 24)")


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a C++ compiler")
def test_header_compiles_as_cpp(tmp_path):
    """The same client builds as C++11 (the header's extern "C" block), warnings as errors."""
    lib = build.build()
    src = tmp_path / "client.cpp"
    src.write_text(CLIENT)
    exe = tmp_path / "client_cpp"
    subprocess.run(["g++", "-std=c++11", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{ROOT / 'include'}",
                    str(src), "-o", str(exe), f"-L{lib.parent}", "-lpagedgqa", f"-Wl,-rpath,{lib.parent}"],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    assert out.startswith("info ") and "bad malformed page table" in out

