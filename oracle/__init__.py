"""CPU oracle for the unified-hash-table embedding step (ctypes wrapper).

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this package.  The product
path (``sparse_ctr_embedding_gb300``) never imports it and the two share no
code; see ``oracle.cpp`` for the passages each function restates.

Pins (what ties the oracle to something other than itself) live in
``tests/test_oracle_pins.py``: the MurmurHash3 x64-128 verification value
through this ``fmix64``, brute-force probe layouts on tiny tables,
order-independence of the occupied-slot set, brute-force pooling and
gradient sums, closed-form Adagrad and numpy's float16 rounding; FTRL
against torch.optim.Adagrad in the regularisation-free case it reduces to,
and its weight against a numerical minimisation of the proximal objective.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import numpy as np

from .build import LIB_PATH, build

_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_f64p = ctypes.POINTER(ctypes.c_double)
_vp = ctypes.c_void_p

ERR = {0: "ok", 1: "invalid", 2: "duplicate key", 3: "reserved key", 4: "bad slot",
       5: "probe walk and key map disagree", 6: "row values not provided"}


class OracleError(RuntimeError):
    pass


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            build()
        L = ctypes.CDLL(LIB_PATH)
        L.orc_fmix64.restype = ctypes.c_uint64
        L.orc_fmix64.argtypes = [ctypes.c_uint64]
        L.orc_build.argtypes = [_vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _vp, ctypes.POINTER(_vp)]
        L.orc_free.argtypes = [_vp]
        L.orc_free.restype = None
        L.orc_info.argtypes = [_vp, _vp]
        L.orc_layout.argtypes = [_vp, _vp, _vp]
        L.orc_elem_offsets.argtypes = [_vp, _vp]
        L.orc_resolve.argtypes = [_vp, _vp, ctypes.c_int64, _vp, _vp]
        L.orc_forward.argtypes = [_vp, _vp, ctypes.c_int64, _vp, ctypes.c_int, ctypes.c_int, _vp, _vp,
                                  _vp, ctypes.c_int64, _vp, _vp]
        L.orc_backward.argtypes = [_vp, _vp, ctypes.c_int64, _vp, ctypes.c_int, _vp, _vp, ctypes.c_int64,
                                   ctypes.POINTER(_vp)]
        L.orc_grad_info.argtypes = [_vp, _vp, _vp]
        L.orc_grad_copy.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp]
        L.orc_grad_free.argtypes = [_vp]
        L.orc_grad_free.restype = None
        L.orc_adagrad.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, _vp, _vp, ctypes.c_float, ctypes.c_float]
        L.orc_f32_to_f16.argtypes = [_vp, ctypes.c_int64, _vp]
        L.orc_rowwise_adagrad.argtypes = [_vp, _vp, ctypes.c_int64, ctypes.c_int, _vp, _vp, ctypes.c_float,
                                          ctypes.c_float]
        L.orc_ftrl.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, _vp, _vp, _vp, ctypes.c_float, ctypes.c_float,
                               ctypes.c_float, ctypes.c_float]
        _lib = L
    return _lib


def _p(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(_vp)


def _check(rc: int):
    if rc != 0:
        raise OracleError(ERR.get(rc, str(rc)))


def fmix64(k: int) -> int:
    return int(lib().orc_fmix64(ctypes.c_uint64(k & ((1 << 64) - 1))))


def f32_to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _check(lib().orc_f32_to_f16(_p(x), x.size, _p(out)))
    return out


def f16_copy(master: np.ndarray) -> np.ndarray:
    """The rows the forward reads from a master-copy table (JD article 3.2.3:
    FP16 storage and compute, an FP32 copy of the weights for the update):
    each f32 master element rounded to nearest-even, as float16."""
    return f32_to_f16_bits(master).view(np.float16)


WDTYPE = {"f32": 0, "f16": 1}
POOL = {"sum": 0, "mean": 1}


class Table:
    """The prepared insert-free table: key->row map plus simulated slot layout."""

    def __init__(self, keys: np.ndarray, cap: int, dims) -> None:
        self.keys = np.ascontiguousarray(keys, dtype=np.int64)
        self.dims = np.ascontiguousarray(dims, dtype=np.int32)
        self.cap = int(cap)
        h = _vp()
        _check(lib().orc_build(_p(self.keys), self.keys.size, self.cap, len(self.dims), _p(self.dims),
                               ctypes.byref(h)))
        self._h = h
        info = np.zeros(6, dtype=np.int64)
        lib().orc_info(self._h, _p(info))
        (self.n, _, self.max_probe, self.sum_probe, self.max_cluster, self.n_elems) = (int(v) for v in info)

    def __del__(self):
        if getattr(self, "_h", None):
            lib().orc_free(self._h)
            self._h = None

    @property
    def n_slots(self) -> int:
        return len(self.dims)

    def layout(self) -> Tuple[np.ndarray, np.ndarray]:
        sk = np.empty(self.cap, dtype=np.int64)
        sr = np.empty(self.cap, dtype=np.int64)
        lib().orc_layout(self._h, _p(sk), _p(sr))
        return sk, sr

    def elem_offsets(self) -> np.ndarray:
        off = np.empty(self.n + 1, dtype=np.int64)
        lib().orc_elem_offsets(self._h, _p(off))
        return off

    def resolve(self, q: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
        q = np.ascontiguousarray(q, dtype=np.int64)
        slot = np.empty(q.size, dtype=np.int64)
        row = np.empty(q.size, dtype=np.int64)
        _check(lib().orc_resolve(self._h, _p(q), q.size, _p(slot), _p(row)))
        return slot, row

    def forward(self, offsets, qkeys, pool: str, wdtype: str, values: np.ndarray,
                row_map: Optional[np.ndarray] = None, bags: Optional[np.ndarray] = None):
        """Pooled output (float64) and sum|terms| for all bags, or the listed ones.

        All bags: arrays shaped [B, sum(dims)].  Listed bags: flat, each bag's
        dims[slot] values in list order."""
        offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        qkeys = np.ascontiguousarray(qkeys, dtype=np.int64)
        values = np.ascontiguousarray(values)
        n_bags = offsets.size - 1
        S = self.n_slots
        if bags is None:
            n_out = (n_bags // S) * int(self.dims.sum())
        else:
            bags = np.ascontiguousarray(bags, dtype=np.int64)
            n_out = int(self.dims[bags % S].sum())
        out = np.empty(n_out, dtype=np.float64)
        ab = np.empty(n_out, dtype=np.float64)
        rm = None if row_map is None else np.ascontiguousarray(row_map, dtype=np.int64)
        _check(lib().orc_forward(self._h, _p(offsets), n_bags, _p(qkeys), POOL[pool], WDTYPE[wdtype],
                                 _p(values), _p(rm), _p(bags), -1 if bags is None else bags.size,
                                 _p(out), _p(ab)))
        if bags is None:
            return out.reshape(n_bags // S, -1), ab.reshape(n_bags // S, -1)
        return out, ab

    def backward(self, offsets, qkeys, pool: str, grad: np.ndarray, key_filter: Optional[np.ndarray] = None):
        """Per-key gradients: (unique keys ascending, their rows, offsets, G, sum|terms|)."""
        offsets = np.ascontiguousarray(offsets, dtype=np.int64)
        qkeys = np.ascontiguousarray(qkeys, dtype=np.int64)
        grad = np.ascontiguousarray(grad, dtype=np.float32)
        kf = None if key_filter is None else np.ascontiguousarray(key_filter, dtype=np.int64)
        h = _vp()
        _check(lib().orc_backward(self._h, _p(offsets), offsets.size - 1, _p(qkeys), POOL[pool], _p(grad),
                                  _p(kf), 0 if kf is None else kf.size, ctypes.byref(h)))
        try:
            nu = ctypes.c_int64()
            ne = ctypes.c_int64()
            lib().orc_grad_info(h, ctypes.byref(nu), ctypes.byref(ne))
            keys = np.empty(nu.value, dtype=np.int64)
            rows = np.empty(nu.value, dtype=np.int64)
            goff = np.empty(nu.value + 1, dtype=np.int64)
            G = np.empty(ne.value, dtype=np.float64)
            A = np.empty(ne.value, dtype=np.float64)
            lib().orc_grad_copy(h, _p(keys), _p(rows), _p(goff), _p(G), _p(A))
        finally:
            lib().orc_grad_free(h)
        return keys, rows, goff, G, A


def adagrad(G: np.ndarray, w: np.ndarray, acc: np.ndarray, lr: float, eps: float) -> Tuple[np.ndarray, np.ndarray]:
    """Element-wise Adagrad on copies of (w, acc); w float32 or float16."""
    G = np.ascontiguousarray(G, dtype=np.float64)
    w = np.array(w, copy=True)
    acc = np.array(acc, dtype=np.float32, copy=True)
    wd = 1 if w.dtype == np.float16 else 0
    if wd == 0:
        w = w.astype(np.float32)
    assert G.size == w.size == acc.size
    _check(lib().orc_adagrad(_p(G), G.size, wd, _p(w), _p(acc), ctypes.c_float(lr), ctypes.c_float(eps)))
    return w, acc


def rowwise_adagrad(G: np.ndarray, goff: np.ndarray, w: np.ndarray, acc_rows: np.ndarray, lr: float,
                    eps: float) -> Tuple[np.ndarray, np.ndarray]:
    """Row-wise Adagrad on copies of (w, acc_rows): rows r = G[goff[r]:goff[r+1]], one
    accumulator per row; w float32 or float16.  Returns (w', acc_rows')."""
    G = np.ascontiguousarray(G, dtype=np.float64)
    goff = np.ascontiguousarray(goff, dtype=np.int64)
    w = np.array(w, copy=True)
    acc = np.array(acc_rows, dtype=np.float32, copy=True)
    wd = 1 if w.dtype == np.float16 else 0
    if wd == 0:
        w = w.astype(np.float32)
    assert G.size == w.size == goff[-1] and acc.size == goff.size - 1
    _check(lib().orc_rowwise_adagrad(_p(G), _p(goff), acc.size, wd, _p(w), _p(acc), ctypes.c_float(lr),
                                     ctypes.c_float(eps)))
    return w, acc


def ftrl(G: np.ndarray, w: np.ndarray, n: np.ndarray, z: np.ndarray, alpha: float, beta: float, lambda1: float,
         lambda2: float) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Element-wise FTRL-Proximal on copies of (w, n, z); w float32 or float16.
    Returns (w', n', z')."""
    G = np.ascontiguousarray(G, dtype=np.float64)
    w = np.array(w, copy=True)
    n = np.array(n, dtype=np.float32, copy=True)
    z = np.array(z, dtype=np.float32, copy=True)
    wd = 1 if w.dtype == np.float16 else 0
    if wd == 0:
        w = w.astype(np.float32)
    assert G.size == w.size == n.size == z.size
    _check(lib().orc_ftrl(_p(G), G.size, wd, _p(w), _p(n), _p(z), ctypes.c_float(alpha), ctypes.c_float(beta),
                          ctypes.c_float(lambda1), ctypes.c_float(lambda2)))
    return w, n, z
