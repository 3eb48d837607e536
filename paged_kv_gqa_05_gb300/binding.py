"""Thin ctypes binding of libpagedgqa.so (argument marshalling and size checks only).

The functions carry the C ABI's names without the ``pgqa_`` prefix:
``kv_append``, ``plan_create``, ``plan_update``, ``run``, ``plan_destroy``,
``plan_get_info``, ``plan_schedule``, ``read_device_flags``.  Every step of the computation runs in
the library's CUDA kernels; torch only supplies device memory and the stream.
There is no fallback: if the shared library is missing or fails to load, every
call raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path
from typing import Optional

import numpy as np
import torch

LIBRARY = Path(__file__).resolve().parent / "_build" / "libpagedgqa.so"

BF16, FP16, FP32 = 0, 1, 2
TORCH_TO_CODE = {torch.bfloat16: BF16, torch.float16: FP16, torch.float32: FP32}
CODE_TO_TORCH = {v: k for k, v in TORCH_TO_CODE.items()}

STATUS_NAMES = {0: "PGQA_OK", 1: "PGQA_ERR_INVALID_ARG", 2: "PGQA_ERR_UNSUPPORTED",
                3: "PGQA_ERR_BAD_PAGE_TABLE", 4: "PGQA_ERR_CUDA", 5: "PGQA_ERR_CAPACITY",
                6: "PGQA_ERR_DEVICE_CHECK"}

# Every entry point include/pagedgqa.h declares.
EXPORTS = ("pgqa_abi_version", "pgqa_status_string", "pgqa_last_error", "pgqa_read_device_flags",
           "pgqa_kv_append", "pgqa_plan_create", "pgqa_plan_update", "pgqa_run",
           "pgqa_plan_destroy", "pgqa_plan_get_info", "pgqa_append_run", "pgqa_decode_static_scratch",
           "pgqa_kv_append_rope", "pgqa_plan_schedule")


class PagedGQAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))


class PlanConfig(ctypes.Structure):
    _fields_ = [("num_qo_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("page_size", ctypes.c_int), ("dtype", ctypes.c_int),
                ("max_batch", ctypes.c_int), ("max_q_rows", ctypes.c_int64),
                ("max_splits", ctypes.c_int), ("split_tokens", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("decode_kernel", ctypes.c_int),
                ("pipeline_stages", ctypes.c_int), ("prefill_splits", ctypes.c_int),
                ("rope_max_position", ctypes.c_int),
                ("rope_theta", ctypes.c_double), ("prefill_kernel", ctypes.c_int),
                ("test_stall_wait_us", ctypes.c_int)]


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_items", ctypes.c_int), ("num_merge_tasks", ctypes.c_int),
                ("split_tokens", ctypes.c_int), ("max_splits_used", ctypes.c_int),
                ("total_q_rows", ctypes.c_int), ("num_sms", ctypes.c_int),
                ("kv_tokens", ctypes.c_int64), ("num_prefill_tiles", ctypes.c_int)]


class ScheduleInfo(ctypes.Structure):
    _fields_ = [("num_items", ctypes.c_int), ("num_merge_tasks", ctypes.c_int),
                ("num_prefill_tiles", ctypes.c_int), ("split_tokens", ctypes.c_int),
                ("max_splits_used", ctypes.c_int), ("pipeline_stages", ctypes.c_int),
                ("total_q_rows", ctypes.c_int), ("kv_tokens", ctypes.c_int64)]


# Rows of pgqa_plan_schedule's output arrays (pgqa_slice, pgqa_merge, pgqa_prefill_tile): int32 fields.
SLICE_DTYPE = np.dtype([(f, np.int32) for f in ("q_row", "kv_head", "key_begin", "key_end", "partial_slot",
                                                 "append_pos")])
MERGE_DTYPE = np.dtype([(f, np.int32) for f in ("q_row", "kv_head", "slot_base", "num_splits")])
TILE_DTYPE = np.dtype([(f, np.int32) for f in ("q_row0", "rows", "n_keys", "kv_head", "pair0", "pairs", "key_begin",
                                                "key_end", "partial_base", "split", "num_splits")])

_lib: Optional[ctypes.CDLL] = None
_i32p = ctypes.POINTER(ctypes.c_int32)
_vp = ctypes.c_void_p


def load(path: Path | str | None = None) -> ctypes.CDLL:
    """Loads the library (once).  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = Path(path) if path else LIBRARY
    if not path.exists():
        raise RuntimeError(f"{path} is missing: build it with `python -m paged_kv_gqa_05_gb300.build` "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(str(path))
    lib.pgqa_abi_version.restype = ctypes.c_int
    lib.pgqa_status_string.restype = ctypes.c_char_p
    lib.pgqa_status_string.argtypes = [ctypes.c_int]
    lib.pgqa_last_error.restype = ctypes.c_char_p
    lib.pgqa_read_device_flags.restype = ctypes.c_int
    lib.pgqa_read_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), ctypes.c_int]
    lib.pgqa_kv_append.restype = ctypes.c_int
    lib.pgqa_kv_append.argtypes = [_vp, _vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                   ctypes.c_int, _vp, _vp, _vp, ctypes.c_int64, _vp]
    lib.pgqa_plan_create.restype = ctypes.c_int
    lib.pgqa_plan_create.argtypes = [ctypes.POINTER(_vp), ctypes.POINTER(PlanConfig)]
    lib.pgqa_plan_update.restype = ctypes.c_int
    lib.pgqa_plan_update.argtypes = [_vp, _i32p, _i32p, _i32p, ctypes.c_int, _vp, _i32p,
                                     ctypes.c_int64, ctypes.c_int, _vp]
    lib.pgqa_run.restype = ctypes.c_int
    lib.pgqa_run.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_float, _vp]
    lib.pgqa_append_run.restype = ctypes.c_int
    lib.pgqa_append_run.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int, _vp, ctypes.c_float,
                                    ctypes.c_int, _vp]
    lib.pgqa_decode_static_scratch.restype = ctypes.c_int
    lib.pgqa_decode_static_scratch.argtypes = [_vp, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp, ctypes.c_int,
                                               ctypes.c_int64,
                                               ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                               ctypes.c_int, ctypes.c_int, _vp, ctypes.c_int, _vp,
                                               ctypes.c_float, _vp]
    lib.pgqa_kv_append_rope.restype = ctypes.c_int
    lib.pgqa_kv_append_rope.argtypes = [_vp, _vp, _vp, ctypes.c_int64, _vp, _vp, _vp, _vp, ctypes.c_int64, _vp]
    lib.pgqa_plan_destroy.restype = ctypes.c_int
    lib.pgqa_plan_destroy.argtypes = [_vp]
    lib.pgqa_plan_get_info.restype = ctypes.c_int
    lib.pgqa_plan_get_info.argtypes = [_vp, ctypes.POINTER(PlanInfo)]
    lib.pgqa_plan_schedule.restype = ctypes.c_int
    lib.pgqa_plan_schedule.argtypes = [ctypes.POINTER(PlanConfig), ctypes.c_int, _i32p, _i32p, _i32p, ctypes.c_int,
                                       _i32p, ctypes.c_int64, ctypes.c_int, _vp, ctypes.c_int, _vp, ctypes.c_int,
                                       _vp, ctypes.c_int, ctypes.POINTER(ScheduleInfo)]
    if lib.pgqa_abi_version() != 5:
        raise RuntimeError("libpagedgqa.so ABI version mismatch")
    _lib = lib
    return lib


def _check(status: int) -> None:
    if status != 0:
        raise PagedGQAError(status, load().pgqa_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor, name: str) -> int:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _host_i32(a, name: str) -> Optional[np.ndarray]:
    """A host int32 copy (or view) of an integer array; values that int32 cannot hold
    and non-integer arrays raise instead of being truncated."""
    if a is None:
        return None
    if isinstance(a, torch.Tensor):
        if a.is_cuda:
            raise ValueError(f"{name} must be a host array")
        a = a.numpy()
    arr = np.asarray(a)
    if arr.size:
        if arr.dtype.kind not in "iu":
            raise ValueError(f"{name} must hold integers, not {arr.dtype}")
        if arr.dtype.itemsize > 4 or arr.dtype == np.uint32:
            lo, hi = int(arr.min()), int(arr.max())
            if lo < -(1 << 31) or hi >= (1 << 31):
                raise ValueError(f"{name} holds values outside int32 ({lo} .. {hi})")
    return np.ascontiguousarray(arr, dtype=np.int32)


def _i32ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_i32p)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------

def kv_append(k_pool: torch.Tensor, v_pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
              slot_mapping: torch.Tensor, stream=None) -> None:
    """pgqa_kv_append: rows k[t], v[t] -> flat slot slot_mapping[t] of the pools."""
    P, ps, Hkv, D = k_pool.shape
    if v_pool.shape != k_pool.shape or k.shape != v.shape or k.shape[1:] != (Hkv, D):
        raise ValueError("shape mismatch between pools and rows")
    if k_pool.dtype != k.dtype or v_pool.dtype != k.dtype or v.dtype != k.dtype:
        raise ValueError("pools and rows must share one dtype")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    if slot_mapping.numel() < k.shape[0]:
        raise ValueError("slot_mapping needs one slot per row")
    lib = load()
    _check(lib.pgqa_kv_append(_dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), P, ps, Hkv, D,
                              TORCH_TO_CODE[k.dtype], _dev(k, "k"), _dev(v, "v"),
                              _dev(slot_mapping, "slot_mapping"), k.shape[0], _stream(stream)))


def kv_append_rope(plan: int, k_pool: torch.Tensor, v_pool: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                   slot_mapping: torch.Tensor, positions: torch.Tensor, stream=None) -> None:
    """pgqa_kv_append_rope: k[t] rotated at positions[t] and v[t] -> flat slot slot_mapping[t]."""
    P, ps, Hkv, D = k_pool.shape
    if v_pool.shape != k_pool.shape or k.shape != v.shape or k.shape[1:] != (Hkv, D):
        raise ValueError("shape mismatch between pools and rows")
    if k_pool.dtype != k.dtype or v_pool.dtype != k.dtype or v.dtype != k.dtype:
        raise ValueError("pools and rows must share one dtype")
    if slot_mapping.dtype != torch.int64 or positions.dtype != torch.int32:
        raise ValueError("slot_mapping must be int64 and positions int32")
    if slot_mapping.shape != (k.shape[0],) or positions.shape != (k.shape[0],):
        raise ValueError("one slot and one position per row")
    _check(load().pgqa_kv_append_rope(plan, _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), P, _dev(k, "k"),
                                      _dev(v, "v"), _dev(slot_mapping, "slot_mapping"),
                                      _dev(positions, "positions"), k.shape[0], _stream(stream)))


def _config(num_qo_heads, num_kv_heads, head_dim, page_size, dtype, max_batch, max_q_rows, max_splits=0,
            split_tokens=0, ctas_per_sm=0, decode_kernel="auto", pipeline_stages=0, prefill_splits=0,
            rope_theta=0.0, rope_max_position=0, prefill_kernel="auto",
            test_stall_wait_us=0) -> PlanConfig:
    kinds = {"auto": 0, "tensor_core": 1, "cuda_core": 2}
    pf_kinds = {"auto": 0, "tcgen05": 1, "mma_sync": 2}
    return PlanConfig(num_qo_heads, num_kv_heads, head_dim, page_size, TORCH_TO_CODE[dtype],
                      max_batch, max_q_rows, max_splits, split_tokens, ctas_per_sm, kinds[decode_kernel],
                      pipeline_stages, prefill_splits, rope_max_position, float(rope_theta),
                      pf_kinds[prefill_kernel], int(test_stall_wait_us))


def plan_create(num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                dtype: torch.dtype, max_batch: int, max_q_rows: int, max_splits: int = 0,
                split_tokens: int = 0, ctas_per_sm: int = 0, decode_kernel: str = "auto",
                pipeline_stages: int = 0, prefill_splits: int = 0,
                rope_theta: float = 0.0, rope_max_position: int = 0, prefill_kernel: str = "auto",
                test_stall_wait_us: int = 0) -> int:
    """pgqa_plan_create on the current CUDA device; returns the plan handle.
    decode_kernel: "auto" | "tensor_core" | "cuda_core"; rope_theta > 0 turns on the
    rotary embedding of q and the appended K rows (positions < rope_max_position);
    prefill_kernel: "auto" | "tcgen05" | "mma_sync"; test_stall_wait_us > 0 only in
    the test of the bounded-wait failure path (see pgqa_plan_config)."""
    cfg = _config(num_qo_heads, num_kv_heads, head_dim, page_size, dtype, max_batch, max_q_rows, max_splits,
                  split_tokens, ctas_per_sm, decode_kernel, pipeline_stages, prefill_splits,
                  rope_theta, rope_max_position, prefill_kernel, test_stall_wait_us)
    h = _vp()
    _check(load().pgqa_plan_create(ctypes.byref(h), ctypes.byref(cfg)))
    return h.value


def plan_update(plan: int, kv_indptr, last_page_len, kv_indices: torch.Tensor, num_pages: int,
                qo_indptr=None, kv_indices_host=None, causal: bool = False, stream=None) -> None:
    """pgqa_plan_update; kv_indptr / last_page_len / qo_indptr / kv_indices_host are host arrays."""
    indptr = _host_i32(kv_indptr, "kv_indptr")
    last = _host_i32(last_page_len, "last_page_len")
    qo = _host_i32(qo_indptr, "qo_indptr")
    mirror = _host_i32(kv_indices_host, "kv_indices_host")
    if kv_indices.dtype != torch.int32:
        raise ValueError("kv_indices must be int32")
    batch = len(indptr) - 1
    dptr = _dev(kv_indices, "kv_indices") if kv_indices.numel() else None
    _check(load().pgqa_plan_update(plan, _i32ptr(indptr), _i32ptr(last), _i32ptr(qo), batch, dptr,
                                   _i32ptr(mirror), int(num_pages), int(bool(causal)),
                                   _stream(stream)))


def _check_outputs(q: torch.Tensor, out: torch.Tensor, lse: Optional[torch.Tensor]) -> None:
    """out holds a row for every row of q, and lse a value for every (row, head)."""
    if q.dim() != 3:
        raise ValueError("q must be [rows, num_qo_heads, head_dim]")
    if out.numel() < q.numel():
        raise ValueError(f"out holds {out.numel()} elements, q {q.numel()}")
    if lse is not None and lse.numel() < q.shape[0] * q.shape[1]:
        raise ValueError(f"lse holds {lse.numel()} elements, q has {q.shape[0] * q.shape[1]} (row, head) pairs")


def run(plan: int, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
        out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
        lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0, pool_stable: bool = False,
        stream=None) -> torch.Tensor:
    """pgqa_run; allocates `out` (torch) when it is not given.  pool_stable: the
    PGQA_RUN_POOL_STABLE promise (pgqa_append_run without new rows)."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    _check_outputs(q, out, lse)
    if k_pool.dtype != q.dtype or v_pool.dtype != q.dtype:
        raise ValueError("q and pools must share one dtype")
    if pool_stable:
        _check(load().pgqa_append_run(plan, None, None, _dev(q, "q"), _dev(k_pool, "k_pool"),
                                      _dev(v_pool, "v_pool"), _dev(out, "out"), TORCH_TO_CODE[out.dtype],
                                      None if lse is None else _dev(lse, "lse"), float(sm_scale), POOL_STABLE,
                                      _stream(stream)))
        return out
    _check(load().pgqa_run(plan, _dev(q, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"),
                           _dev(out, "out"), TORCH_TO_CODE[out.dtype],
                           None if lse is None else _dev(lse, "lse"), float(sm_scale),
                           _stream(stream)))
    return out


POOL_STABLE = 1


def append_run(plan: int, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
               v_pool: torch.Tensor, out: Optional[torch.Tensor] = None,
               out_dtype: Optional[torch.dtype] = None, lse: Optional[torch.Tensor] = None,
               sm_scale: float = 0.0, pool_stable: bool = False, stream=None) -> torch.Tensor:
    """pgqa_append_run: the step's new K/V rows (one per query row) are appended and
    attended in one launch."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    if lse is not None and lse.dtype != torch.float32:
        raise ValueError("lse must be float32")
    _check_outputs(q, out, lse)
    for t, name in ((k_pool, "k_pool"), (v_pool, "v_pool"), (k_new, "k_new"), (v_new, "v_new")):
        if t.dtype != q.dtype:
            raise ValueError(f"{name} must have q's dtype")
    if k_new.shape != v_new.shape or k_new.shape[0] != q.shape[0] or k_new.shape[1:] != k_pool.shape[2:]:
        raise ValueError("k_new / v_new must be [q rows, num_kv_heads, head_dim]")
    _check(load().pgqa_append_run(plan, _dev(k_new, "k_new"), _dev(v_new, "v_new"), _dev(q, "q"),
                                  _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), _dev(out, "out"),
                                  TORCH_TO_CODE[out.dtype], None if lse is None else _dev(lse, "lse"),
                                  float(sm_scale), POOL_STABLE if pool_stable else 0, _stream(stream)))
    return out


def decode_static_scratch(q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor,
                          kv_indptr: torch.Tensor, kv_indices: torch.Tensor, last_page_len: torch.Tensor,
                          splits: int, out: Optional[torch.Tensor] = None,
                          out_dtype: Optional[torch.dtype] = None, lse: Optional[torch.Tensor] = None,
                          sm_scale: float = 0.0, stream=None) -> torch.Tensor:
    """pgqa_decode_static_scratch: decode without any device allocation inside the
    library (page table on the device; kv_indices may be empty).  Callers that
    cannot allocate pass a preallocated `out`."""
    if out is None:
        out = torch.empty(q.shape, dtype=out_dtype or q.dtype, device=q.device)
    for t, name in ((kv_indptr, "kv_indptr"), (kv_indices, "kv_indices"), (last_page_len, "last_page_len")):
        if t.dtype != torch.int32:
            raise ValueError(f"{name} must be int32")
    P, ps, Hkv, D = k_pool.shape
    batch, hq = q.shape[0], q.shape[1]
    for t, n, name in ((kv_indptr, batch + 1, "kv_indptr"), (last_page_len, batch, "last_page_len"),
                       (out, q.numel(), "out"), (lse, batch * hq, "lse")):
        if t is not None and t.numel() < n:
            raise ValueError(f"{name} holds {t.numel()} elements; the call reads or writes {n}")
    _check(load().pgqa_decode_static_scratch(
        _dev(q, "q"), _dev(k_pool, "k_pool"), _dev(v_pool, "v_pool"), _dev(kv_indptr, "kv_indptr"),
        _dev(kv_indices, "kv_indices") if kv_indices.numel() else None, kv_indices.numel(),
        _dev(last_page_len, "last_page_len"),
        q.shape[0], P, ps, q.shape[1], Hkv, D, TORCH_TO_CODE[q.dtype], int(splits), _dev(out, "out"),
        TORCH_TO_CODE[out.dtype], None if lse is None else _dev(lse, "lse"), float(sm_scale), _stream(stream)))
    return out


def plan_schedule(num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int, dtype: torch.dtype,
                  kv_indptr, last_page_len, kv_indices, num_pages: int, qo_indptr=None, causal: bool = False,
                  num_sms: int = 152, max_batch: Optional[int] = None, max_q_rows: Optional[int] = None,
                  **options) -> dict:
    """pgqa_plan_schedule: the schedule plan_update would build, on the host alone
    (no GPU needed).  All arrays are host int32; options as for plan_create.
    Returns {"info": {...}, "slices", "merges", "tiles"} with numpy structured arrays
    (SLICE_DTYPE, MERGE_DTYPE, TILE_DTYPE) in launch order."""
    indptr = _host_i32(kv_indptr, "kv_indptr")
    last = _host_i32(last_page_len, "last_page_len")
    qo = _host_i32(qo_indptr, "qo_indptr")
    idx = _host_i32(kv_indices, "kv_indices")
    batch = len(indptr) - 1
    rows = batch if qo is None else (int(qo[-1]) if len(qo) else 0)
    cfg = _config(num_qo_heads, num_kv_heads, head_dim, page_size, dtype,
                  max(1, batch) if max_batch is None else max_batch,
                  max(1, rows) if max_q_rows is None else max_q_rows, **options)
    lib = load()
    info = ScheduleInfo()

    def call(slices, merges, tiles):
        def ptr(a):
            return None if a is None else a.ctypes.data
        _check(lib.pgqa_plan_schedule(ctypes.byref(cfg), int(num_sms), _i32ptr(indptr), _i32ptr(last), _i32ptr(qo),
                                      batch, _i32ptr(idx if idx is not None and idx.size else None), int(num_pages),
                                      int(bool(causal)), ptr(slices), 0 if slices is None else len(slices),
                                      ptr(merges), 0 if merges is None else len(merges), ptr(tiles),
                                      0 if tiles is None else len(tiles), ctypes.byref(info)))

    call(None, None, None)  # counts
    slices = np.zeros(info.num_items, SLICE_DTYPE)
    merges = np.zeros(info.num_merge_tasks, MERGE_DTYPE)
    tiles = np.zeros(info.num_prefill_tiles, TILE_DTYPE)
    call(slices, merges, tiles)
    return {"info": {name: getattr(info, name) for name, _ in ScheduleInfo._fields_},
            "slices": slices, "merges": merges, "tiles": tiles}


def plan_destroy(plan: int) -> None:
    _check(load().pgqa_plan_destroy(plan))


def plan_get_info(plan: int) -> dict:
    info = PlanInfo()
    _check(load().pgqa_plan_get_info(plan, ctypes.byref(info)))
    return {name: getattr(info, name) for name, _ in PlanInfo._fields_}


# Bits of the device flag word (include/pagedgqa.h).
FLAG_PAGE_INDEX, FLAG_SLOT_RANGE, FLAG_WAIT_TIMEOUT, FLAG_SMEM_ALIGN, FLAG_ROPE_POSITION = 1, 2, 4, 8, 16


def read_device_flags(clear: bool = True) -> int:
    """Flag word of the current device (synchronises).  0 when no check fired."""
    v = ctypes.c_uint32(0)
    st = load().pgqa_read_device_flags(ctypes.byref(v), int(clear))
    if st not in (0, 6):
        _check(st)
    return int(v.value)


class Plan:
    """Owns a plan handle; plan()/run() in the style of an attention backend.

    Unlike the module-level calls, which take a bare handle, run() and append_run()
    here check that every tensor holds at least the elements the plan's last
    successful update() reads or writes through it (the C ABI receives pointers
    only and cannot), and raise ValueError before any launch otherwise."""

    def __init__(self, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int,
                 dtype: torch.dtype, max_batch: int, max_q_rows: int, **options):
        self.handle = plan_create(num_qo_heads, num_kv_heads, head_dim, page_size, dtype,
                                  max_batch, max_q_rows, **options)
        self._shape(num_qo_heads, num_kv_heads, head_dim, page_size)

    def _shape(self, num_qo_heads: int, num_kv_heads: int, head_dim: int, page_size: int) -> None:
        self.num_qo_heads, self.num_kv_heads, self.head_dim = num_qo_heads, num_kv_heads, head_dim
        self.page_size = page_size
        self._num_pages = None  # pool pages of the last successful update()
        self._need = None       # elements per tensor that update implies (computed on first use)

    def _check_sizes(self, **tensors) -> None:
        if self._num_pages is None:
            return  # no successful update: the library refuses the call itself
        if self._need is None:
            rows = int(self.info()["total_q_rows"])
            hq, hkv, d = self.num_qo_heads, self.num_kv_heads, self.head_dim
            pool = self._num_pages * self.page_size * hkv * d
            self._rows = rows
            self._need = {"q": rows * hq * d, "out": rows * hq * d, "lse": rows * hq, "k_pool": pool,
                          "v_pool": pool, "k_new": rows * hkv * d, "v_new": rows * hkv * d}
        for name, t in tensors.items():
            if t is not None and t.numel() < self._need[name]:
                raise ValueError(f"{name} holds {t.numel()} elements; the plan reads or writes "
                                 f"{self._need[name]} ({self._rows} query rows, {self._num_pages} pool pages)")

    def update(self, kv_indptr, last_page_len, kv_indices: torch.Tensor, num_pages: int, **kwargs) -> "Plan":
        self._num_pages, self._need = None, None
        plan_update(self.handle, kv_indptr, last_page_len, kv_indices, num_pages, **kwargs)
        self._num_pages = int(num_pages)
        return self

    def run(self, q: torch.Tensor, k_pool: torch.Tensor, v_pool: torch.Tensor, out: Optional[torch.Tensor] = None,
            out_dtype: Optional[torch.dtype] = None, lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0,
            pool_stable: bool = False, stream=None) -> torch.Tensor:
        self._check_sizes(q=q, k_pool=k_pool, v_pool=v_pool, out=out, lse=lse)
        return run(self.handle, q, k_pool, v_pool, out=out, out_dtype=out_dtype, lse=lse, sm_scale=sm_scale,
                   pool_stable=pool_stable, stream=stream)

    def append_run(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor, k_pool: torch.Tensor,
                   v_pool: torch.Tensor, out: Optional[torch.Tensor] = None, out_dtype: Optional[torch.dtype] = None,
                   lse: Optional[torch.Tensor] = None, sm_scale: float = 0.0, pool_stable: bool = False,
                   stream=None) -> torch.Tensor:
        self._check_sizes(k_new=k_new, v_new=v_new, q=q, k_pool=k_pool, v_pool=v_pool, out=out, lse=lse)
        return append_run(self.handle, k_new, v_new, q, k_pool, v_pool, out=out, out_dtype=out_dtype, lse=lse,
                          sm_scale=sm_scale, pool_stable=pool_stable, stream=stream)

    def kv_append_rope(self, *args, **kwargs) -> None:
        kv_append_rope(self.handle, *args, **kwargs)

    def info(self) -> dict:
        return plan_get_info(self.handle)

    def close(self) -> None:
        if self.handle:
            plan_destroy(self.handle)
            self.handle = None

    def __enter__(self) -> "Plan":
        return self

    def __exit__(self, *exc) -> None:
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
