"""Helpers for GPU-vs-oracle parity tests (test code only).

Tolerance gates, fixed before the first kernel was written (tol = 1e-5 for
float32 weight storage, 2e-3 for float16 storage):
  pooled output   |x - r| <= tol * max(|r|, A),  A = sum of |terms| of the bag
                  (a pooled sum of N(0,1)-like rows can cancel to ~0, so its
                  error is measured against the size of its terms)
  accumulator     |x - r| <= tol * r             (acc is positive)
  weight          |x - r| <= tol * max(|r|, |w_old|)
These plain gates hold for every element of a key whose gradient terms do not
cancel much: kappa = A_g / |g| <= KAPPA (A_g = sum of |terms| of the key, g
their sum).  Where they cancel more, no float32 evaluation can give g to a
relative 1e-5: each term grad_out * (1/L) is a float32 product, rounded once,
with 1/L itself a rounded float32, so g carries an error of order u * A_g
(u = 2^-24) whatever the summation.  The library sums with TwoSum
compensation (groups of at most 4 products summed plainly, then folded in
exactly), which bounds the whole error by
  |dg| <= DG_ULPS * u * A_g + u * |g|
(3u for the roundings of each term: 1/L, its product with the count of a run
of equal (row, bag) pairs, and the product with grad_out; 3u for a plain
4-term group sum; u for the float32 partial of a row cut by a sub-chunk edge;
u for a folded block of such partials; DG_ULPS = 8 covers these 8u).  For keys with
kappa > KAPPA the gates add that bound propagated through the update:
  accumulator  + 2 |g| dg + dg^2         (acc' = acc + g^2)
  weight       + lr * dg / sqrt(acc')    (|d/dg (g / sqrt(acc + g^2))| <= 1/sqrt(acc'))
The plain maximum relative error |x - r| / |r| is reported for both classes.
Index work (slots, rows, unique keys) and untouched rows are compared
bit-exactly.
"""
from __future__ import annotations

import dataclasses
import json
import os
from typing import Optional

import numpy as np
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E

TOL = {"f32": 1e-5, "f16": 2e-3, "f16m": 1e-5}   # f16m: the updated weights are the f32 masters


def tol_of(cfg) -> float:
    return TOL[cfg.wdtype]


def gate(name, x, r, scale, tol):
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    scale = np.asarray(scale, dtype=np.float64)
    err = np.abs(x - r)
    bad = err > tol * scale
    rel = float((err / np.maximum(scale, 1e-300)).max()) if err.size else 0.0
    if bad.any():
        i = int(np.argmax(bad))
        raise AssertionError(f"{name}: {int(bad.sum())}/{bad.size} outside tol {tol}; first at {i}: "
                             f"x={x.flat[i]!r} r={r.flat[i]!r} scale={scale.flat[i]!r}; max rel {rel:.3g}")
    return rel


KAPPA = 16.0       # cancellation A_g / |g| up to which the plain gates apply unchanged
DG_ULPS = 8.0      # bound on the float32 gradient's error, in units of u * A_g
U32 = 2.0 ** -24   # float32 unit roundoff


def grad_err(G, Ag):
    """Per-element bound on |g_gpu - g| for keys whose terms cancel (kappa >
    KAPPA), 0 elsewhere (see the module docstring)."""
    G = np.abs(np.asarray(G, dtype=np.float64))
    Ag = np.asarray(Ag, dtype=np.float64)
    dg = DG_ULPS * U32 * Ag + U32 * G
    return np.where(Ag > KAPPA * G, dg, 0.0)


def acc_scale(acc_r, G=None, Ag=None, tol=1.0):
    """Accumulators are positive: a plain relative gate, plus (kappa > KAPPA)
    the propagated gradient bound expressed in units of tol."""
    s = acc_r.astype(np.float64)
    if G is not None:
        dg = grad_err(G, Ag)
        s = s + (2 * np.abs(np.asarray(G, np.float64)) * dg + dg * dg) / tol
    return s


def w_scale(w_r, w_old, acc_r=None, G=None, Ag=None, lr=0.0, tol=1.0):
    """Weights: relative to the larger of the new and the old weight (an
    update can move a weight through zero), plus (kappa > KAPPA) the
    propagated gradient bound in units of tol."""
    s = np.maximum(np.abs(w_r.astype(np.float64)), np.abs(w_old.astype(np.float64)))
    if G is not None:
        s = s + lr * grad_err(G, Ag) / np.sqrt(acc_r.astype(np.float64)) / tol
    return s


def split_plain_rel(x, r, G, Ag):
    """Plain max relative error for elements of keys with kappa <= KAPPA and > KAPPA."""
    x = np.asarray(x, np.float64)
    r = np.asarray(r, np.float64)
    hi = np.asarray(Ag, np.float64) > KAPPA * np.abs(np.asarray(G, np.float64))
    return (plain_rel(x[~hi], r[~hi]) if (~hi).any() else 0.0,
            plain_rel(x[hi], r[hi]) if hi.any() else 0.0, int(hi.sum()))


def report(key: str, **fields) -> None:
    """Append measured errors to the JSON-lines file named by EMB_PARITY_REPORT
    (nothing when it is unset): the numbers the design notes quote."""
    path = os.environ.get("EMB_PARITY_REPORT")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"case": key, **fields}) + "\n")


def plain_rel(x, r):
    """max |x - r| / |r| over elements with |r| >= 1e-3 * max |r| (information only)."""
    x = np.asarray(x, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    if r.size == 0 or not np.any(r):
        return 0.0
    m = np.abs(r) >= 1e-3 * np.abs(r).max()
    return float((np.abs(x - r)[m] / np.abs(r)[m]).max())


@dataclasses.dataclass
class GpuStep:
    table: E.Table
    out: torch.Tensor
    slots: torch.Tensor
    rows: torch.Tensor
    unique: np.ndarray
    keys_out: np.ndarray
    values_out: np.ndarray
    acc_out: np.ndarray
    flags: int
    ws: torch.Tensor


def make_table(cfg, wl, values_dev=True):
    vals = wl.values.cuda() if values_dev else wl.values.cpu()
    return E.emb_table_create(cfg.dims, cfg.wdtype, wl.keys.cpu(), values=vals, acc=None,
                              capacity=cfg.capacity, acc_init=cfg.acc0)


def gpu_step(cfg, wl, values_dev=True, recorded=False) -> GpuStep:
    """One step through the C ABI.  recorded=True uses the forward that
    records (row, bag) pairs and the backward that starts from them."""
    tbl = make_table(cfg, wl, values_dev)
    off, q, g = wl.offsets.cuda(), wl.qkeys.cuda(), wl.grad.cuda()
    n_bags, nnz = off.numel() - 1, q.numel()
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, n_bags, nnz), dtype=torch.uint8, device="cuda")
    if recorded:
        out = E.emb_lookup_fwd_record(tbl, off, q, cfg.pool, ws)
    else:
        out = E.emb_lookup_fwd(tbl, off, q, cfg.pool)
    slots, rows = E.emb_resolve(tbl, q)
    if recorded:
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws)
    else:
        E.emb_bwd_adagrad(tbl, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
    uk = torch.empty(max(nnz, 1), dtype=torch.int64, device="cuda")
    nu = torch.zeros(1, dtype=torch.int64, device="cuda")
    E.emb_bwd_unique_keys(tbl, ws, uk, nu)
    n_el = tbl.stats["n_elems"]
    ko = torch.empty(cfg.n_keys, dtype=torch.int64, device="cuda")
    vo = torch.empty(n_el, dtype=wl.values.dtype, device="cuda")
    ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, ko, vo, ao)
    flags = E.emb_check_device_flag(tbl)
    torch.cuda.synchronize()
    return GpuStep(tbl, out, slots, rows, uk[:int(nu.item())].cpu().numpy(), ko.cpu().numpy(),
                   vo.cpu().numpy(), ao.cpu().numpy(), flags, ws)


def elem_index(elem_off: np.ndarray, rows: np.ndarray) -> np.ndarray:
    starts = elem_off[rows]
    lens = elem_off[rows + 1] - starts
    rep = np.repeat(starts, lens)
    within = np.arange(int(lens.sum())) - np.repeat(np.cumsum(lens) - lens, lens)
    return rep + within


def check_step(cfg, wl, gs: GpuStep, T: Optional[oracle.Table] = None) -> dict:
    """Full element-wise parity of one step against the oracle."""
    tol = tol_of(cfg)
    keys = wl.keys.cpu().numpy()
    off = wl.offsets.cpu().numpy()
    q = wl.qkeys.cpu().numpy()
    values = wl.values.cpu().numpy()
    grad = wl.grad.cpu().numpy()
    if T is None:
        T = oracle.Table(keys, cfg.capacity, cfg.dims)
    rep = {}
    assert gs.flags == 0, f"device flag {gs.flags}"
    # slot resolution and hit mask: bit-exact
    slot_r, row_r = T.resolve(q)
    assert np.array_equal(gs.slots.cpu().numpy(), slot_r)
    assert np.array_equal(gs.rows.cpu().numpy(), row_r)
    # pooled output
    out_r, A = T.forward(off, q, cfg.pool, cfg.wdtype, values)
    rep["fwd_gate"] = gate("pooled", gs.out.cpu().numpy(), out_r, np.maximum(np.abs(out_r), A), tol)
    rep["fwd_plain_rel"] = plain_rel(gs.out.cpu().numpy(), out_r)
    # unique keys: bit-exact as a set
    uk_r, rows_u, goff, G, Ag = T.backward(off, q, cfg.pool, grad)
    assert np.array_equal(np.sort(gs.unique), uk_r)
    rep["n_unique"] = int(uk_r.size)
    # checkpoint keys come back in keys-array order
    assert np.array_equal(gs.keys_out, keys)
    # updated rows
    eoff = T.elem_offsets()
    idx = elem_index(eoff, rows_u)
    acc0 = np.full(idx.size, cfg.acc0, dtype=np.float32)
    w_r, acc_r = oracle.adagrad(G, values[idx], acc0, cfg.lr, cfg.eps)
    rep["acc_gate"] = gate("acc", gs.acc_out[idx], acc_r, acc_scale(acc_r, G, Ag, tol), tol)
    rep["acc_plain_rel"], rep["acc_plain_rel_cancelling"], rep["n_cancelling"] = \
        split_plain_rel(gs.acc_out[idx], acc_r, G, Ag)
    w_r64 = w_r.astype(np.float64)
    rep["w_gate"] = gate("weight", gs.values_out[idx].astype(np.float64), w_r64,
                         w_scale(w_r, values[idx], acc_r, G, Ag, cfg.lr, tol), tol)
    rep["w_plain_rel"], rep["w_plain_rel_cancelling"], _ = split_plain_rel(gs.values_out[idx], w_r64, G, Ag)
    rep["max_cancellation"] = float((Ag / np.maximum(np.abs(G), 1e-300)).max()) if G.size else 0.0
    # rows not hit: bit-identical weights and accumulators
    untouched = np.ones(values.size, dtype=bool)
    untouched[idx] = False
    assert np.array_equal(gs.values_out[untouched].view(np.int16 if values.dtype == np.float16 else np.int32),
                          values[untouched].view(np.int16 if values.dtype == np.float16 else np.int32))
    assert np.all(gs.acc_out[untouched] == np.float32(cfg.acc0))
    return rep
