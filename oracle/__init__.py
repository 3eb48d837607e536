"""TEST INFRASTRUCTURE: ctypes front end of the CPU fp64 oracle (pgqa_oracle.c).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
use this package.  It never imports the CUDA library and the library never
imports it.  Inputs are raw 16-bit patterns (numpy ``uint16``) so that the
oracle widens exactly the values the GPU sees; outputs are fp64.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "pgqa_oracle.c"
BUILD_DIR = HERE / "_build"
LIBRARY = BUILD_DIR / "liboracle.so"

DTYPE_CODES = {"bf16": 0, "fp16": 1}

_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)


def build(source: Path = SOURCE, output: Path = LIBRARY, force: bool = False) -> Path:
    """Compile the oracle with plain gcc (no fast-math: IEEE exp/log)."""
    source, output = Path(source), Path(output)
    if output.exists() and not force and output.stat().st_mtime >= source.stat().st_mtime:
        return output
    output.parent.mkdir(parents=True, exist_ok=True)
    tmp = output.with_suffix(f".{os.getpid()}.tmp.so")
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-Wall", "-Wextra",
           "-o", str(tmp), str(source), "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, output)
    return output


def _ptr(a: np.ndarray | None, typ):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(typ)


class Oracle:
    """Bound oracle library (the real one, or a test-built variant of it)."""

    def __init__(self, path: Path | str | None = None):
        self.path = Path(path) if path is not None else build()
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_widen.restype = ctypes.c_double
        lib.oracle_widen.argtypes = [ctypes.c_uint16, ctypes.c_int]
        lib.oracle_check_page_table.restype = ctypes.c_int
        lib.oracle_check_page_table.argtypes = [_i32p, _i32p, _i32p, ctypes.c_int,
                                                ctypes.c_int64, ctypes.c_int]
        lib.oracle_kv_append.restype = ctypes.c_int
        lib.oracle_kv_append.argtypes = [_u8p, _u8p, ctypes.c_int64, ctypes.c_int64,
                                         _u8p, _u8p, _i64p, ctypes.c_int64]
        lib.oracle_lse_merge.restype = None
        lib.oracle_lse_merge.argtypes = [ctypes.c_int, ctypes.c_int, _f64p, _f64p, _f64p, _f64p]
        lib.oracle_paged_attention.restype = ctypes.c_int
        lib.oracle_paged_attention.argtypes = [
            _u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, ctypes.c_int, _i32p, _i32p, _i32p, _i32p, ctypes.c_int,
            ctypes.c_int, ctypes.c_double, _f64p, _f64p, ctypes.c_int]
        lib.oracle_attention_partial.restype = ctypes.c_int
        lib.oracle_attention_partial.argtypes = [
            _u16p, _u16p, _u16p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, _i32p, _i32p, _i32p, _i32p, ctypes.c_int, ctypes.c_int64,
            ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, ctypes.c_double,
            _f64p, _f64p]
        lib.oracle_narrow.restype = ctypes.c_uint16
        lib.oracle_narrow.argtypes = [ctypes.c_double, ctypes.c_int]
        lib.oracle_rope_f64.restype = ctypes.c_int
        lib.oracle_rope_f64.argtypes = [_f64p, _f64p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i32p,
                                        ctypes.c_double]
        lib.oracle_rope.restype = ctypes.c_int
        lib.oracle_rope.argtypes = [_u16p, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _i32p, ctypes.c_double,
                                    ctypes.c_int, _f64p, _u16p]
        self.lib = lib

    # -- scalar helpers ---------------------------------------------------
    def widen(self, bits: np.ndarray, dtype: str) -> np.ndarray:
        code = DTYPE_CODES[dtype]
        flat = np.ascontiguousarray(bits, dtype=np.uint16).ravel()
        return np.array([self.lib.oracle_widen(int(b), code) for b in flat]).reshape(np.shape(bits))

    def narrow(self, values: np.ndarray, dtype: str) -> np.ndarray:
        """fp64 values -> 16-bit patterns, rounded once to nearest, ties to even."""
        code = DTYPE_CODES[dtype]
        flat = np.ascontiguousarray(values, dtype=np.float64).ravel()
        return np.array([self.lib.oracle_narrow(float(v), code) for v in flat],
                        dtype=np.uint16).reshape(np.shape(values))

    # -- rotary position embedding ----------------------------------------
    def rope_f64(self, x: np.ndarray, positions, theta: float) -> np.ndarray:
        """x [rows, heads, d] fp64 -> rotated fp64 (positions [rows])."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        positions = np.ascontiguousarray(positions, dtype=np.int32)
        rows, heads, d = x.shape
        assert positions.shape == (rows,)
        y = np.empty_like(x)
        rc = self.lib.oracle_rope_f64(_ptr(x, _f64p), _ptr(y, _f64p), rows, heads, d,
                                      _ptr(positions, _i32p), float(theta))
        if rc != 0:
            raise ValueError(f"oracle_rope_f64 failed (code {rc})")
        return y

    def rope(self, x: np.ndarray, positions, theta: float, dtype: str):
        """x [rows, heads, d] uint16 -> (rotated uint16, rotated fp64 before rounding)."""
        x = np.ascontiguousarray(x, dtype=np.uint16)
        positions = np.ascontiguousarray(positions, dtype=np.int32)
        rows, heads, d = x.shape
        assert positions.shape == (rows,)
        out64 = np.empty(x.shape, np.float64)
        out16 = np.empty(x.shape, np.uint16)
        if rows == 0:
            return out16, out64
        rc = self.lib.oracle_rope(_ptr(x, _u16p), rows, heads, d, _ptr(positions, _i32p), float(theta),
                                  DTYPE_CODES[dtype], _ptr(out64, _f64p), _ptr(out16, _u16p))
        if rc != 0:
            raise ValueError(f"oracle_rope failed (code {rc})")
        return out16, out64

    def check_page_table(self, kv_indptr, kv_indices, last_page_len, num_pages, page_size) -> int:
        kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
        kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        if kv_indices.size == 0:
            kv_indices = np.zeros(1, np.int32)
        return self.lib.oracle_check_page_table(
            _ptr(kv_indptr, _i32p), _ptr(kv_indices, _i32p), _ptr(last_page_len, _i32p),
            len(kv_indptr) - 1, int(num_pages), int(page_size))

    # -- append -----------------------------------------------------------
    def kv_append(self, k_pool: np.ndarray, v_pool: np.ndarray, k: np.ndarray, v: np.ndarray,
                  slot_mapping: np.ndarray) -> None:
        """In place on k_pool / v_pool (any C-contiguous arrays [P, ps, Hkv, d])."""
        num_slots = k_pool.shape[0] * k_pool.shape[1]
        row_bytes = k_pool.itemsize * k_pool.shape[2] * k_pool.shape[3]
        slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
        k = np.ascontiguousarray(k)
        v = np.ascontiguousarray(v)
        rc = self.lib.oracle_kv_append(
            k_pool.ctypes.data_as(_u8p), v_pool.ctypes.data_as(_u8p), num_slots, row_bytes,
            k.ctypes.data_as(_u8p), v.ctypes.data_as(_u8p), _ptr(slot_mapping, _i64p),
            len(slot_mapping))
        if rc != 0:
            raise ValueError(f"oracle_kv_append rejected the slots (code {rc})")

    # -- attention --------------------------------------------------------
    def paged_attention(self, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                        dtype: str, qo_indptr=None, causal: bool = False,
                        scale: float = 0.0, nthreads: int = 1):
        """q [rows, Hq, d] uint16, pools [P, ps, Hkv, d] uint16 -> (out fp64, lse fp64)."""
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
        kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
        if kv_indices.size == 0:
            kv_indices = np.zeros(1, np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        qo = None if qo_indptr is None else np.ascontiguousarray(qo_indptr, dtype=np.int32)
        rows, Hq, d = q.shape
        P, ps, Hkv, d2 = k_pool.shape
        assert d == d2
        out = np.zeros((rows, Hq, d), np.float64)
        lse = np.zeros((rows, Hq), np.float64)
        rc = self.lib.oracle_paged_attention(
            _ptr(q, _u16p), _ptr(k_pool, _u16p), _ptr(v_pool, _u16p), DTYPE_CODES[dtype],
            P, ps, Hq, Hkv, d, _ptr(kv_indptr, _i32p), _ptr(kv_indices, _i32p),
            _ptr(last_page_len, _i32p), _ptr(qo, _i32p), len(kv_indptr) - 1,
            int(bool(causal)), float(scale), _ptr(out, _f64p), _ptr(lse, _f64p), int(nthreads))
        if rc != 0:
            raise ValueError(f"oracle_paged_attention rejected the input (code {rc})")
        return out, lse

    def attention_partial(self, q, k_pool, v_pool, kv_indptr, kv_indices, last_page_len,
                          dtype: str, b: int, r: int, h: int, j0: int, j1: int,
                          qo_indptr=None, causal: bool = False, scale: float = 0.0):
        q = np.ascontiguousarray(q, dtype=np.uint16)
        k_pool = np.ascontiguousarray(k_pool, dtype=np.uint16)
        v_pool = np.ascontiguousarray(v_pool, dtype=np.uint16)
        kv_indptr = np.ascontiguousarray(kv_indptr, dtype=np.int32)
        kv_indices = np.ascontiguousarray(kv_indices, dtype=np.int32)
        if kv_indices.size == 0:
            kv_indices = np.zeros(1, np.int32)
        last_page_len = np.ascontiguousarray(last_page_len, dtype=np.int32)
        qo = None if qo_indptr is None else np.ascontiguousarray(qo_indptr, dtype=np.int32)
        _, Hq, d = q.shape
        _, ps, Hkv, _ = k_pool.shape
        o = np.zeros(d, np.float64)
        lse = np.zeros(1, np.float64)
        rc = self.lib.oracle_attention_partial(
            _ptr(q, _u16p), _ptr(k_pool, _u16p), _ptr(v_pool, _u16p), DTYPE_CODES[dtype],
            ps, Hq, Hkv, d, _ptr(kv_indptr, _i32p), _ptr(kv_indices, _i32p),
            _ptr(last_page_len, _i32p), _ptr(qo, _i32p), int(b), int(r), int(h), int(j0),
            int(j1), int(bool(causal)), float(scale), _ptr(o, _f64p), _ptr(lse, _f64p))
        if rc != 0:
            raise ValueError(f"oracle_attention_partial failed (code {rc})")
        return o, float(lse[0])

    def lse_merge(self, o_parts: np.ndarray, lse_parts: np.ndarray):
        o_parts = np.ascontiguousarray(o_parts, dtype=np.float64)
        lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
        n, d = o_parts.shape
        o = np.zeros(d, np.float64)
        lse = np.zeros(1, np.float64)
        self.lib.oracle_lse_merge(n, d, _ptr(o_parts, _f64p), _ptr(lse_parts, _f64p),
                                  _ptr(o, _f64p), _ptr(lse, _f64p))
        return o, float(lse[0])


_default: Oracle | None = None


def get() -> Oracle:
    """The oracle built from this directory's source (compiled on first use)."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
