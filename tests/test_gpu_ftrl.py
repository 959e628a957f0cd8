"""GPU parity of the FTRL-Proximal update (emb_bwd_ftrl / emb_bwd_ftrl_recorded)
against the oracle's FTRL, over several steps in a row so that the state
(w, n, z) carried from step to step is checked too.

Gates (tol as for Adagrad; see parity_util for dg, the bound on the float32
per-key gradient's error, nonzero only for keys whose terms cancel):
  n        |x - r| <= tol * r + 2|g| dg + dg^2                (n' = n + g^2, as Adagrad's acc)
  z        |x - r| <= tol * max(|r|, |z_old| + |g| + |sigma w_old|) + dg + ds
           (z' = z + g - sigma w is a sum whose terms can cancel)
  weight   |x - r| <= tol * max(|r|, |w_old|, |z'| / den) + (dg + ds) / den,
           den = (beta + sqrt(n')) / alpha + lambda2
           (w' = -(z' - sign(z') lambda1) / den: near the threshold |z'| = lambda1 the
           shrunk weight is small, so its error is measured against the unshrunk |z'| / den)
ds is the conditioning of sigma itself: sigma = (sqrt(n') - sqrt(n)) / alpha is a
difference of two nearly equal square roots when g^2 << n, so the last bit of
n' (which follows g's last bit) moves sigma by about u sqrt(n') / alpha, and z
by that times |w|; both sides evaluate the same float32 formula, so
  ds = 4 u sqrt(n') |w_old| / alpha + |g| dg' |w_old| / (alpha sqrt(n'))
bounds the difference that g's own error dg' = DG_ULPS u A_g + u |g| (every
key, cancelling or not) and the roundings of n' and the square roots can make
(u = 2^-24).
"""
import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import DG_ULPS, U32, elem_index, gate, grad_err, report, tol_of

pytestmark = pytest.mark.gpu

ALPHA, BETA, L1, L2 = 0.05, 1.0, 0.5, 0.1


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CASES = [
    W.config(1),                                    # 4 slots, dim 16 f32, sum
    W.scaled(W.config(2), 100, 16),                 # 26 slots, dim 64 f32, mean, absent keys
    W.scaled(W.config(3), 500, 64),                 # 100 slots, dim 32 f16, sum
    W.scaled(W.config(4), 250, 32),                 # ragged dims
]
MASTER = W.scaled(W.config(5), 1000, 256)           # dim 128, run with f32 masters + f16 copy


def _table(cfg, wl, wdtype=None):
    wd = wdtype or cfg.wdtype
    vals = wl.values.float() if wd == "f16m" else wl.values
    return E.emb_table_create(cfg.dims, wd, wl.keys.cpu(), values=vals.cuda(), capacity=cfg.capacity,
                              acc_init=cfg.acc0, optimizer="ftrl")


def _state(tbl, n_el, wdt):
    vo = torch.empty(n_el, dtype=wdt, device="cuda")
    no = torch.empty(n_el, dtype=torch.float32, device="cuda")
    zo = torch.empty(n_el, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, None, vo, no)
    E.emb_table_export_z(tbl, zo)
    return vo.cpu().numpy(), no.cpu().numpy(), zo.cpu().numpy()


def _run(cfg, wdtype=None, steps=3):
    wd = wdtype or cfg.wdtype
    wl = W.make(cfg, device="cuda")
    off, q = wl.offsets, wl.qkeys
    n_bags, nnz = off.numel() - 1, q.numel()
    rec, unr = _table(cfg, wl, wd), _table(cfg, wl, wd)
    ws = torch.empty(E.emb_bwd_workspace_size(rec, n_bags, nnz), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws)
    n_el = rec.stats["n_elems"]
    wdt = torch.float16 if wd == "f16" else torch.float32
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    eoff = T.elem_offsets()
    offn, qn = off.cpu().numpy(), q.cpu().numpy()
    w = wl.values.cpu().numpy().copy()
    if wd == "f16m":
        w = w.astype(np.float32)
    n = np.full(n_el, cfg.acc0, np.float32)
    z = np.zeros(n_el, np.float32)
    tol = tol_of(cfg) if wd != "f16m" else 1e-5
    zeros = 0
    for k in range(steps):
        g = torch.roll(wl.grad, shifts=k, dims=0) * (1.0, -0.5, 2.0)[k % 3]   # a different gradient each step
        E.emb_lookup_fwd_record(rec, off, q, cfg.pool, ws)
        E.emb_bwd_ftrl_recorded(rec, n_bags, nnz, cfg.pool, g, ALPHA, BETA, L1, L2, ws)
        E.emb_bwd_ftrl(unr, off, q, cfg.pool, g, ALPHA, BETA, L1, L2, ws2)
        assert E.emb_check_device_flag(rec) == 0 and E.emb_check_device_flag(unr) == 0
        w_x, n_x, z_x = _state(rec, n_el, wdt)
        w_u, n_u, z_u = _state(unr, n_el, wdt)
        for a, b in ((w_x, w_u), (n_x, n_u), (z_x, z_u)):    # both backward paths: bit-identical
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        # the oracle's step on the rows the batch hits
        _, rows_u, _, G, Ag = T.backward(offn, qn, cfg.pool, g.cpu().numpy())
        idx = elem_index(eoff, rows_u)
        w_old, n_old, z_old = w[idx].copy(), n[idx].copy(), z[idx].copy()
        w_r, n_r, z_r = oracle.ftrl(G, w_old, n_old, z_old, ALPHA, BETA, L1, L2)
        w[idx], n[idx], z[idx] = w_r, n_r, z_r
        dg = grad_err(G, Ag)
        absg = np.abs(G)
        sn1 = np.sqrt(n_r.astype(np.float64))
        absw = np.abs(w_old.astype(np.float64))
        sigma = (sn1 - np.sqrt(n_old.astype(np.float64))) / ALPHA
        den = (BETA + sn1) / ALPHA + L2
        dg_all = DG_ULPS * U32 * Ag + U32 * absg             # the gradient's error bound, every key
        ds = 4 * U32 * sn1 * absw / ALPHA + absg * dg_all * absw / (ALPHA * sn1)
        gate(f"n, step {k + 1}", n_x[idx], n_r, n_r.astype(np.float64) + (2 * absg * dg + dg * dg) / tol, tol)
        gate(f"z, step {k + 1}", z_x[idx], z_r,
             np.maximum(np.abs(z_r.astype(np.float64)),
                        np.abs(z_old.astype(np.float64)) + absg + np.abs(sigma * w_old.astype(np.float64)))
             + (dg + ds) / tol, tol)
        gate(f"weights, step {k + 1}", w_x[idx].astype(np.float64), w_r.astype(np.float64),
             np.maximum(np.maximum(np.abs(w_r.astype(np.float64)), absw),
                        np.abs(z_r.astype(np.float64)) / den) + (dg + ds) / den / tol, tol)
        # rows the batch does not hit: bit-identical to the oracle's (unchanged) state
        untouched = np.ones(n_el, bool)
        untouched[idx] = False
        assert np.array_equal(w_x[untouched].view(np.uint8), w[untouched].astype(w_x.dtype).view(np.uint8))
        assert np.array_equal(n_x[untouched], n[untouched]) and np.array_equal(z_x[untouched], z[untouched])
        zeros += int((w_x[idx] == 0).sum())
        # the next step starts both sides from the GPU's state: each step is checked
        # from identical inputs (independent roundings would otherwise compound)
        w[idx], n[idx], z[idx] = w_x[idx], n_x[idx], z_x[idx]
        report(f"ftrl/{cfg.name}/{wd}/step{k + 1}", n_elems=int(idx.size), zero_weights=int((w_x[idx] == 0).sum()),
               oracle_zero_weights=int((w_r == 0).sum()))
    assert zeros > 0                                   # lambda1 made weights exactly 0 (sparsity)
    return rec, w, wl


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_ftrl_steps_match_the_oracle(cfg):
    _run(cfg)


def test_ftrl_on_master_copy_tables_refreshes_the_forward_copy():
    """f32 masters updated by FTRL; the forward's f16 copy is written from the
    new masters in the same kernel: a forward after the steps reads exactly the
    masters rounded to nearest-even."""
    cfg = MASTER
    tbl, w, wl = _run(cfg, "f16m", steps=2)
    out = E.emb_lookup_fwd(tbl, wl.offsets, wl.qkeys, cfg.pool)
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    ref, A = T.forward(wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy(), cfg.pool, "f16", oracle.f16_copy(w))
    gate("forward on the refreshed f16 copy", out.cpu().numpy(), ref, np.maximum(np.abs(ref), A), 2e-3)


def test_optimizer_mismatch_and_bad_parameters_are_refused():
    cfg = CASES[0]
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    ftrl = _table(cfg, wl)
    with pytest.raises(E.EmbError) as ei:                          # Adagrad on an FTRL table
        E.emb_bwd_adagrad(ftrl, off, q, cfg.pool, g, 0.01, 1e-8, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    with pytest.raises(E.EmbError) as ei:                          # alpha must be > 0
        E.emb_bwd_ftrl(ftrl, off, q, cfg.pool, g, 0.0, 1.0, 0.0, 0.0, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    ada = E.emb_table_create(cfg.dims, cfg.wdtype, wl.keys.cpu(), values=wl.values, capacity=cfg.capacity,
                             acc_init=cfg.acc0)
    with pytest.raises(E.EmbError) as ei:                          # FTRL on an Adagrad table
        E.emb_bwd_ftrl(ada, off, q, cfg.pool, g, ALPHA, BETA, L1, L2, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    with pytest.raises(E.EmbError):                                # an Adagrad table has no z
        E.emb_table_export_z(ada, torch.empty(ada.stats["n_elems"], dtype=torch.float32, device="cuda"))


def test_ftrl_z_checkpoint_round_trip():
    """export (weights, n) + export_z, then create + import_z: the resumed table
    continues exactly like the original."""
    cfg = CASES[1]
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    a = _table(cfg, wl)
    ws = torch.empty(E.emb_bwd_workspace_size(a, n_bags, nnz), dtype=torch.uint8, device="cuda")
    E.emb_bwd_ftrl(a, off, q, cfg.pool, g, ALPHA, BETA, L1, L2, ws)
    n_el = a.stats["n_elems"]
    w0, n0, z0 = _state(a, n_el, torch.float32)
    b = E.emb_table_create(cfg.dims, cfg.wdtype, wl.keys.cpu(), values=torch.from_numpy(w0),
                           acc=torch.from_numpy(n0), capacity=cfg.capacity, optimizer="ftrl")
    E.emb_table_import_z(b, torch.from_numpy(z0))
    for t in (a, b):
        E.emb_bwd_ftrl(t, off, q, cfg.pool, -g, ALPHA, BETA, L1, L2, ws)
    sa, sb = _state(a, n_el, torch.float32), _state(b, n_el, torch.float32)
    for x, y in zip(sa, sb):
        assert np.array_equal(x.view(np.uint8), y.view(np.uint8))
