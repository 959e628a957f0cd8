"""Python binding of the GB300 embedding-step library (include/emb_gb300.h).

Argument marshalling only: every function forwards to the C entry point of the
same name in ``_build/libemb_gb300.so``, passing tensor data pointers, sizes
and the current CUDA stream.  All computation happens in the library's
sm_103a kernels; there is no fallback path.  If the library has not been
built, importing succeeds but the first call raises ``LibraryNotBuilt``.
"""
from __future__ import annotations

import ctypes
import os
import re
from typing import Optional, Sequence, Tuple

import numpy as np
import torch

from .build import HEADER, LIB_PATH, build

__all__ = [
    "EmbError", "LibraryNotBuilt", "Table", "lib", "declared_symbols",
    "emb_table_create", "emb_table_create_device", "emb_table_destroy", "emb_table_get_stats", "emb_table_plan",
    "emb_lookup_fwd", "emb_lookup_fwd_record", "emb_lookup_fwd_dedup", "emb_bwd_adagrad_recorded", "emb_bwd_workspace_size", "emb_bwd_adagrad", "emb_bwd_adagrad_noalloc",
    "emb_bwd_ftrl", "emb_bwd_ftrl_recorded", "emb_table_export_z", "emb_table_import_z",
    "emb_debug_fail_device_alloc", "emb_debug_live_device_allocs", "emb_debug_set_probe_bound", "Pipeline",
    "emb_bwd_unique_keys", "emb_bwd_phase_events", "EMB_NOALLOC_SCRATCH_BYTES", "EMB_SORT_DIGIT_BITS", "BWD_PHASES",
    "emb_resolve", "emb_table_export", "emb_table_export_rows", "emb_table_slots", "emb_check_device_flag",
    "emb_status_string", "emb_last_error",
    "EMB_FLAG_PROBE_BOUND", "EMB_FLAG_BAD_OFFSETS", "EMB_FLAG_SLOT_MISMATCH", "EMB_FLAG_BAD_ROW",
]

EMB_OK = 0
STATUS = {0: "EMB_OK", 1: "EMB_ERR_INVALID_ARG", 2: "EMB_ERR_CUDA", 3: "EMB_ERR_OOM", 4: "EMB_ERR_DUP_KEY",
          5: "EMB_ERR_RESERVED_KEY", 6: "EMB_ERR_LOAD_FACTOR", 7: "EMB_ERR_WORKSPACE",
          8: "EMB_ERR_DEVICE_FLAG", 9: "EMB_ERR_UNSUPPORTED"}
EMB_FLAG_PROBE_BOUND, EMB_FLAG_BAD_OFFSETS, EMB_FLAG_SLOT_MISMATCH, EMB_FLAG_BAD_ROW = 1, 2, 4, 8
EMB_NOALLOC_SCRATCH_BYTES = 64 << 20
EMB_SORT_DIGIT_BITS = 7
BWD_PHASES = ("expand", "sort", "reduce", "fixup")
_DTYPE = {"f32": 0, "f16": 1, "f16m": 2}   # f16m: f32 master rows + the f16 copy the forward reads
_POOL = {"sum": 0, "mean": 1}
_OPT = {"adagrad": 0, "ftrl": 1, "rowwise_adagrad": 2}


class LibraryNotBuilt(ImportError):
    pass


class EmbError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS.get(status, status)}: {message}")
        self.status = status
        self.name = STATUS.get(status, str(status))
        self.message = message


class _Desc(ctypes.Structure):
    _fields_ = [("n_slots", ctypes.c_int32), ("slot_dim", ctypes.POINTER(ctypes.c_int32)),
                ("wdtype", ctypes.c_int), ("capacity", ctypes.c_int64), ("acc_init", ctypes.c_float),
                ("optimizer", ctypes.c_int)]


class _Ftrl(ctypes.Structure):
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("lambda1", ctypes.c_float),
                ("lambda2", ctypes.c_float)]


class _Stats(ctypes.Structure):
    _fields_ = [("n_keys", ctypes.c_int64), ("capacity", ctypes.c_int64), ("n_elems", ctypes.c_int64),
                ("n_slots", ctypes.c_int32), ("sum_dims", ctypes.c_int32), ("max_dim", ctypes.c_int32),
                ("wdtype", ctypes.c_int32), ("max_probe", ctypes.c_int64), ("sum_probe", ctypes.c_int64),
                ("max_cluster", ctypes.c_int64), ("probe_bound", ctypes.c_int64),
                ("load_factor", ctypes.c_double), ("device_bytes", ctypes.c_uint64),
                ("max_slot_keys", ctypes.c_int64)]

    def as_dict(self):
        return {f: getattr(self, f) for f, _ in self._fields_}


_lib = None
_vp = ctypes.c_void_p
_i64 = ctypes.c_int64


def lib():
    """The loaded library (ctypes.CDLL); raises LibraryNotBuilt if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise LibraryNotBuilt(f"{LIB_PATH} is missing: run `python -c 'import sparse_ctr_embedding_gb300 as E; E.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "emb_table_create": [ctypes.POINTER(_Desc), _vp, _i64, _vp, _vp, _vp, ctypes.POINTER(_vp)],
            "emb_table_destroy": [_vp],
            "emb_table_create_device": [ctypes.POINTER(_Desc), _vp, _i64, _vp, _vp, _vp, ctypes.POINTER(_vp)],
            "emb_table_get_stats": [_vp, ctypes.POINTER(_Stats)],
            "emb_table_plan": [ctypes.POINTER(_Desc), _vp, _i64, ctypes.POINTER(_Stats), _vp, _vp],
            "emb_lookup_fwd": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, _vp],
            "emb_bwd_workspace_size": [_vp, _i64, _i64, ctypes.POINTER(ctypes.c_size_t)],
            "emb_bwd_adagrad": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, ctypes.c_float, ctypes.c_float,
                                _vp, ctypes.c_size_t, _vp],
            "emb_bwd_unique_keys": [_vp, _vp, ctypes.c_size_t, _vp, _vp, _vp],
            "emb_bwd_phase_events": [_vp, ctypes.POINTER(_vp), ctypes.c_int],
            "emb_lookup_fwd_record": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp],
            "emb_lookup_fwd_dedup": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, _vp, ctypes.c_size_t, _vp],
            "emb_bwd_adagrad_recorded": [_vp, _i64, _i64, ctypes.c_int, _vp, ctypes.c_float, ctypes.c_float, _vp,
                                         ctypes.c_size_t, _vp],
            "emb_bwd_adagrad_noalloc": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, ctypes.c_float,
                                        ctypes.c_float, _vp],
            "emb_bwd_ftrl": [_vp, _vp, _i64, _vp, _i64, ctypes.c_int, _vp, ctypes.POINTER(_Ftrl), _vp,
                             ctypes.c_size_t, _vp],
            "emb_bwd_ftrl_recorded": [_vp, _i64, _i64, ctypes.c_int, _vp, ctypes.POINTER(_Ftrl), _vp,
                                      ctypes.c_size_t, _vp],
            "emb_table_export_z": [_vp, _vp, _vp],
            "emb_debug_fail_device_alloc": [_i64],
            "emb_pipeline_create": [_vp, _i64, _i64, ctypes.c_int, ctypes.c_int, _vp, ctypes.POINTER(_vp)],
            "emb_pipeline_destroy": [_vp],
            "emb_pipeline_submit": [_vp, _vp, _i64, _vp, _i64, _vp, ctypes.POINTER(_i64)],
            "emb_pipeline_forward": [_vp, _i64, ctypes.c_int, _vp, _vp, ctypes.POINTER(_vp)],
            "emb_pipeline_backward_adagrad": [_vp, _i64, _vp, ctypes.c_float, ctypes.c_float],
            "emb_pipeline_backward_ftrl": [_vp, _i64, _vp, ctypes.POINTER(_Ftrl)],
            "emb_pipeline_release": [_vp, _i64],
            "emb_pipeline_wait": [_vp, _i64],
            "emb_debug_set_probe_bound": [_vp, _i64],
            "emb_table_import_z": [_vp, _vp, _vp],
            "emb_resolve": [_vp, _vp, _i64, _vp, _vp, _vp],
            "emb_table_export": [_vp, _vp, _vp, _vp, _vp],
            "emb_table_slots": [_vp, _vp, _vp, _vp],
            "emb_table_export_rows": [_vp, _vp, _i64, _vp, _vp, _vp],
            "emb_check_device_flag": [_vp, _vp, ctypes.POINTER(ctypes.c_uint32)],
        }
        for name, args in sig.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = ctypes.c_int
        L.emb_status_string.argtypes = [ctypes.c_int]
        L.emb_status_string.restype = ctypes.c_char_p
        L.emb_last_error.argtypes = []
        L.emb_last_error.restype = ctypes.c_char_p
        L.emb_debug_live_device_allocs.argtypes = []
        L.emb_debug_live_device_allocs.restype = ctypes.c_int64
        _lib = L
    return _lib


def declared_symbols() -> Sequence[str]:
    """Entry points declared in include/emb_gb300.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^EMB_API [^(]*?\b(emb_\w+)\(", text, flags=re.M)))


def emb_status_string(status: int) -> str:
    return lib().emb_status_string(status).decode()


def emb_last_error() -> str:
    return lib().emb_last_error().decode()


def _check(rc: int):
    if rc != EMB_OK:
        raise EmbError(rc, emb_last_error())


def _stream(stream) -> _vp:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return _vp(stream.cuda_stream)
    return _vp(int(stream))


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _cuda(t: torch.Tensor, dtype, name):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    return _ptr(t, dtype, name)


def _desc(dims, wdtype, capacity, acc_init, optimizer="adagrad"):
    dims_arr = (ctypes.c_int32 * len(dims))(*[int(d) for d in dims])
    d = _Desc(len(dims), dims_arr, _DTYPE[wdtype], int(capacity), float(acc_init), _OPT[optimizer])
    return d, dims_arr


class Table:
    """Owner of one emb_table handle."""

    def __init__(self, handle: int, dims, wdtype: str, optimizer: str = "adagrad"):
        self._h = _vp(handle)
        self.dims = tuple(int(d) for d in dims)
        self.wdtype = wdtype
        self.optimizer = optimizer
        self.stats = emb_table_get_stats(self)

    @property
    def handle(self):
        return self._h

    @property
    def n_slots(self):
        return len(self.dims)

    def close(self):
        if self._h:
            lib().emb_table_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def emb_table_create(dims, wdtype: str, keys: torch.Tensor, values: Optional[torch.Tensor] = None,
                     acc: Optional[torch.Tensor] = None, capacity: int = 0, acc_init: float = 0.0,
                     stream=None, optimizer: str = "adagrad") -> Table:
    """keys: CPU int64; values/acc: CPU or CUDA, ragged rows in keys order.
    optimizer: "adagrad", "ftrl" (acc is then FTRL's n; z starts at 0) or
    "rowwise_adagrad" (acc holds one value per key, in keys order)."""
    if keys.is_cuda:
        raise ValueError("keys must be host memory (the table is prepared on the host)")
    wt = torch.float16 if wdtype == "f16" else torch.float32
    d, _keep = _desc(dims, wdtype, capacity, acc_init, optimizer)
    h = _vp()
    _check(lib().emb_table_create(ctypes.byref(d), _ptr(keys, torch.int64, "keys"), keys.numel(),
                                  _ptr(values, wt, "values"), _ptr(acc, torch.float32, "acc"), _stream(stream),
                                  ctypes.byref(h)))
    return Table(h.value, dims, wdtype, optimizer)


def emb_table_create_device(dims, wdtype: str, keys: torch.Tensor, values: Optional[torch.Tensor] = None,
                            acc: Optional[torch.Tensor] = None, capacity: int = 0, acc_init: float = 0.0,
                            stream=None, optimizer: str = "adagrad") -> Table:
    """The table of emb_table_create, prepared on the GPU: keys is a CUDA int64 tensor."""
    if not keys.is_cuda:
        raise ValueError("keys must be device memory (emb_table_create takes host keys)")
    wt = torch.float16 if wdtype == "f16" else torch.float32
    d, _keep = _desc(dims, wdtype, capacity, acc_init, optimizer)
    h = _vp()
    _check(lib().emb_table_create_device(ctypes.byref(d), _cuda(keys, torch.int64, "keys"), keys.numel(),
                                         _ptr(values, wt, "values"), _ptr(acc, torch.float32, "acc"),
                                         _stream(stream), ctypes.byref(h)))
    return Table(h.value, dims, wdtype, optimizer)


def emb_table_destroy(table: Table):
    table.close()


def emb_table_get_stats(table: Table) -> dict:
    s = _Stats()
    _check(lib().emb_table_get_stats(table.handle, ctypes.byref(s)))
    return s.as_dict()


def emb_table_plan(dims, wdtype: str, keys, capacity: int = 0, layout: bool = False, optimizer: str = "adagrad"):
    """Host-only validation/statistics; with layout=True also the slot layout (numpy)."""
    keys = np.ascontiguousarray(keys, dtype=np.int64)
    d, _keep = _desc(dims, wdtype, capacity, 0.0, optimizer)
    s = _Stats()
    sk = sr = None
    if layout:
        cap = capacity
        if cap == 0:
            cap = 2
            while cap < 2 * keys.size:
                cap <<= 1
        sk = np.empty(cap, dtype=np.int64)
        sr = np.empty(cap, dtype=np.int64)
    _check(lib().emb_table_plan(ctypes.byref(d), keys.ctypes.data, keys.size, ctypes.byref(s),
                                None if sk is None else sk.ctypes.data, None if sr is None else sr.ctypes.data))
    return s.as_dict(), sk, sr


def emb_lookup_fwd(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str,
                   out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    n_bags = offsets.numel() - 1
    if out is None:
        out = torch.empty((n_bags // table.n_slots, sum(table.dims)), dtype=torch.float32, device=offsets.device)
    _check(lib().emb_lookup_fwd(table.handle, _cuda(offsets, torch.int64, "offsets"), n_bags,
                                _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                                _cuda(out, torch.float32, "out"), _stream(stream)))
    return out


def emb_lookup_fwd_record(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str, workspace: torch.Tensor,
                          out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """emb_lookup_fwd that also records the resolved (row, bag) pairs into
    `workspace` for emb_bwd_adagrad_recorded."""
    n_bags = offsets.numel() - 1
    if out is None:
        out = torch.empty((n_bags // table.n_slots, sum(table.dims)), dtype=torch.float32, device=offsets.device)
    _check(lib().emb_lookup_fwd_record(table.handle, _cuda(offsets, torch.int64, "offsets"), n_bags,
                                       _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                                       _cuda(out, torch.float32, "out"), _cuda(workspace, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def emb_lookup_fwd_dedup(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str, workspace: torch.Tensor,
                         out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The forward with a within-batch dedupe: pairs placed and sorted by row,
    each unique row read once; the recorded backward that follows skips its sort."""
    n_bags = offsets.numel() - 1
    if out is None:
        out = torch.empty((n_bags // table.n_slots, sum(table.dims)), dtype=torch.float32, device=offsets.device)
    _check(lib().emb_lookup_fwd_dedup(table.handle, _cuda(offsets, torch.int64, "offsets"), n_bags,
                                      _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                                      _cuda(out, torch.float32, "out"), _cuda(workspace, None, "workspace"),
                                      workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def emb_bwd_adagrad_recorded(table: Table, n_bags: int, nnz: int, pool: str, grad_out: torch.Tensor, lr: float,
                             eps: float, workspace: torch.Tensor, stream=None) -> None:
    _check(lib().emb_bwd_adagrad_recorded(table.handle, n_bags, nnz, _POOL[pool],
                                          _cuda(grad_out, torch.float32, "grad_out"), ctypes.c_float(lr),
                                          ctypes.c_float(eps), _cuda(workspace, None, "workspace"),
                                          workspace.numel() * workspace.element_size(), _stream(stream)))


def emb_bwd_workspace_size(table: Table, n_bags: int, nnz: int) -> int:
    b = ctypes.c_size_t()
    _check(lib().emb_bwd_workspace_size(table.handle, n_bags, nnz, ctypes.byref(b)))
    return b.value


def emb_bwd_adagrad(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str, grad_out: torch.Tensor,
                    lr: float, eps: float, workspace: torch.Tensor, stream=None) -> None:
    _check(lib().emb_bwd_adagrad(table.handle, _cuda(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                 _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                                 _cuda(grad_out, torch.float32, "grad_out"), ctypes.c_float(lr),
                                 ctypes.c_float(eps), _cuda(workspace, None, "workspace"),
                                 workspace.numel() * workspace.element_size(), _stream(stream)))


def emb_bwd_adagrad_noalloc(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str,
                            grad_out: torch.Tensor, lr: float, eps: float, stream=None) -> None:
    """emb_bwd_adagrad without a workspace: for callers that cannot allocate
    device memory, it uses the library's fixed EMB_NOALLOC_SCRATCH_BYTES scratch
    (shared by every call on the device: order overlapping calls)."""
    _check(lib().emb_bwd_adagrad_noalloc(table.handle, _cuda(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                                         _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                                         _cuda(grad_out, torch.float32, "grad_out"), ctypes.c_float(lr),
                                         ctypes.c_float(eps), _stream(stream)))


def _ftrl(alpha, beta, lambda1, lambda2):
    return _Ftrl(float(alpha), float(beta), float(lambda1), float(lambda2))


def emb_bwd_ftrl(table: Table, offsets: torch.Tensor, keys: torch.Tensor, pool: str, grad_out: torch.Tensor,
                 alpha: float, beta: float, lambda1: float, lambda2: float, workspace: torch.Tensor,
                 stream=None) -> None:
    """The backward with the FTRL-Proximal update (tables created with optimizer="ftrl")."""
    p = _ftrl(alpha, beta, lambda1, lambda2)
    _check(lib().emb_bwd_ftrl(table.handle, _cuda(offsets, torch.int64, "offsets"), offsets.numel() - 1,
                              _cuda(keys, torch.int64, "keys"), keys.numel(), _POOL[pool],
                              _cuda(grad_out, torch.float32, "grad_out"), ctypes.byref(p),
                              _cuda(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
                              _stream(stream)))


def emb_bwd_ftrl_recorded(table: Table, n_bags: int, nnz: int, pool: str, grad_out: torch.Tensor, alpha: float,
                          beta: float, lambda1: float, lambda2: float, workspace: torch.Tensor, stream=None) -> None:
    p = _ftrl(alpha, beta, lambda1, lambda2)
    _check(lib().emb_bwd_ftrl_recorded(table.handle, n_bags, nnz, _POOL[pool],
                                       _cuda(grad_out, torch.float32, "grad_out"), ctypes.byref(p),
                                       _cuda(workspace, None, "workspace"),
                                       workspace.numel() * workspace.element_size(), _stream(stream)))


def emb_table_export_z(table: Table, z_out: torch.Tensor, stream=None) -> None:
    _check(lib().emb_table_export_z(table.handle, _ptr(z_out, torch.float32, "z_out"), _stream(stream)))


def emb_table_import_z(table: Table, z_in: torch.Tensor, stream=None) -> None:
    _check(lib().emb_table_import_z(table.handle, _ptr(z_in, torch.float32, "z_in"), _stream(stream)))


def emb_bwd_phase_events(table: Table, events) -> None:
    """Register torch.cuda.Event objects (timing enabled) that each later
    emb_bwd_adagrad records after its expand, sort, reduce and fixup phases."""
    if any(not e.cuda_event for e in events):
        raise ValueError("record each event once (torch creates CUDA events lazily) before registering it")
    arr = (_vp * max(1, len(events)))(*[_vp(e.cuda_event) for e in events])
    _check(lib().emb_bwd_phase_events(table.handle, arr, len(events)))


def emb_bwd_unique_keys(table: Table, workspace: torch.Tensor, keys_out: torch.Tensor, n_unique_out: torch.Tensor,
                        stream=None) -> None:
    _check(lib().emb_bwd_unique_keys(table.handle, _cuda(workspace, None, "workspace"),
                                     workspace.numel() * workspace.element_size(),
                                     _cuda(keys_out, torch.int64, "keys_out"),
                                     _cuda(n_unique_out, torch.int64, "n_unique_out"), _stream(stream)))


def emb_resolve(table: Table, keys: torch.Tensor, slot_out: Optional[torch.Tensor] = None,
                row_out: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    if slot_out is None:
        slot_out = torch.empty_like(keys)
    if row_out is None:
        row_out = torch.empty_like(keys)
    _check(lib().emb_resolve(table.handle, _cuda(keys, torch.int64, "keys"), keys.numel(),
                             _cuda(slot_out, torch.int64, "slot_out"), _cuda(row_out, torch.int64, "row_out"),
                             _stream(stream)))
    return slot_out, row_out


def emb_table_export(table: Table, keys_out: Optional[torch.Tensor], values_out: Optional[torch.Tensor],
                     acc_out: Optional[torch.Tensor], stream=None) -> None:
    wt = torch.float16 if table.wdtype == "f16" else torch.float32
    _check(lib().emb_table_export(table.handle, _ptr(keys_out, torch.int64, "keys_out"),
                                  _ptr(values_out, wt, "values_out"), _ptr(acc_out, torch.float32, "acc_out"),
                                  _stream(stream)))


def emb_table_export_rows(table: Table, rows: torch.Tensor, values_out: Optional[torch.Tensor] = None,
                          acc_out: Optional[torch.Tensor] = None, stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Weights/accumulators of keys-array rows as [n, max_dim] device tensors (zero padded);
    a row-wise Adagrad table's accumulators come as [n]."""
    n, md = rows.numel(), max(table.dims)
    wt = torch.float16 if table.wdtype == "f16" else torch.float32
    if values_out is None:
        values_out = torch.empty((n, md), dtype=wt, device=rows.device)
    if acc_out is None:
        shape = (n,) if table.optimizer == "rowwise_adagrad" else (n, md)
        acc_out = torch.empty(shape, dtype=torch.float32, device=rows.device)
    _check(lib().emb_table_export_rows(table.handle, _cuda(rows, torch.int64, "rows"), n,
                                       _cuda(values_out, wt, "values_out"), _cuda(acc_out, torch.float32, "acc_out"),
                                       _stream(stream)))
    return values_out, acc_out


def emb_table_slots(table: Table, slot_key_out: Optional[torch.Tensor], slot_row_out: Optional[torch.Tensor],
                    stream=None) -> None:
    _check(lib().emb_table_slots(table.handle, _ptr(slot_key_out, torch.int64, "slot_key_out"),
                                 _ptr(slot_row_out, torch.int64, "slot_row_out"), _stream(stream)))


def emb_check_device_flag(table: Table, stream=None) -> int:
    """Synchronise, read and clear the device flag word; returns the flag bits (0 = clean)."""
    f = ctypes.c_uint32()
    rc = lib().emb_check_device_flag(table.handle, _stream(stream), ctypes.byref(f))
    if rc not in (EMB_OK, 8):
        raise EmbError(rc, emb_last_error())
    return f.value


def emb_debug_fail_device_alloc(after: int) -> None:
    """Fault injection: the next `after` device allocations succeed, later ones fail (negative: never)."""
    _check(lib().emb_debug_fail_device_alloc(int(after)))


def emb_debug_live_device_allocs() -> int:
    return int(lib().emb_debug_live_device_allocs())


def emb_debug_set_probe_bound(table: Table, bound: int) -> None:
    """Fault injection: lower the table's probe bound (as a corrupted table would)."""
    _check(lib().emb_debug_set_probe_bound(table.handle, int(bound)))
    table.stats = emb_table_get_stats(table)


class Pipeline:
    """emb_pipeline: overlaps the next batch's host-to-device copy (and the
    pooled output's copy back) with the current step.  Host tensors should be
    pinned.  Per batch: submit -> forward -> backward_adagrad/ftrl (or
    release) -> wait; submit may run up to depth - 1 batches ahead."""

    def __init__(self, table: Table, max_bags: int, max_nnz: int, depth: int = 2, upload_grad: bool = False,
                 stream=None):
        self.table = table
        self._keep = []
        h = _vp()
        _check(lib().emb_pipeline_create(table.handle, int(max_bags), int(max_nnz), int(depth), int(upload_grad),
                                         _stream(stream), ctypes.byref(h)))
        self._h = h

    def submit(self, offsets_h: torch.Tensor, keys_h: torch.Tensor, grad_h: Optional[torch.Tensor] = None) -> int:
        for t, n in ((offsets_h, "offsets"), (keys_h, "keys"), (grad_h, "grad_out")):
            if t is not None and t.is_cuda:
                raise ValueError(f"{n} must be host memory")
        tk = ctypes.c_int64()
        _check(lib().emb_pipeline_submit(self._h, _ptr(offsets_h, torch.int64, "offsets"), offsets_h.numel() - 1,
                                         _ptr(keys_h, torch.int64, "keys"), keys_h.numel(),
                                         _ptr(grad_h, torch.float32, "grad_out"), ctypes.byref(tk)))
        self._keep.append((offsets_h, keys_h, grad_h))   # host memory must outlive the copy
        self._keep = self._keep[-8:]
        return tk.value

    def forward(self, ticket: int, pool: str, out: Optional[torch.Tensor] = None,
                out_h: Optional[torch.Tensor] = None) -> int:
        """Returns the device address of the pooled output (out, or the set's own buffer)."""
        used = _vp()
        _check(lib().emb_pipeline_forward(self._h, int(ticket), _POOL[pool], _ptr(out, torch.float32, "out"),
                                          _ptr(out_h, torch.float32, "out_h"), ctypes.byref(used)))
        return used.value

    def backward_adagrad(self, ticket: int, lr: float, eps: float, grad_out: Optional[torch.Tensor] = None):
        _check(lib().emb_pipeline_backward_adagrad(self._h, int(ticket), _ptr(grad_out, torch.float32, "grad_out"),
                                                   ctypes.c_float(lr), ctypes.c_float(eps)))

    def backward_ftrl(self, ticket: int, alpha, beta, lambda1, lambda2, grad_out: Optional[torch.Tensor] = None):
        p = _ftrl(alpha, beta, lambda1, lambda2)
        _check(lib().emb_pipeline_backward_ftrl(self._h, int(ticket), _ptr(grad_out, torch.float32, "grad_out"),
                                                ctypes.byref(p)))

    def release(self, ticket: int):
        _check(lib().emb_pipeline_release(self._h, int(ticket)))

    def wait(self, ticket: int):
        _check(lib().emb_pipeline_wait(self._h, int(ticket)))

    def close(self):
        if self._h:
            lib().emb_pipeline_destroy(self._h)
            self._h = _vp()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
