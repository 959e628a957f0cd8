"""The forward with a within-batch dedupe (emb_lookup_fwd_dedup): pooled output
against the oracle, and the recorded backward that follows it (which skips its
sort) bit-identical to the one that follows the recording forward."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import gate, make_table, tol_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CASES = [
    W.config(1),
    W.scaled(W.config(2), 100, 16),
    W.scaled(W.config(3), 500, 64),
    W.scaled(W.config(4), 250, 32),
    W.scaled(W.config(5), 1000, 256),
]


def _export(tbl, n_el, dt):
    vo = torch.empty(n_el, dtype=dt, device="cuda")
    ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, None, vo, ao)
    return vo, ao


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_dedupe_forward_and_the_backward_after_it(cfg):
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    a, b = make_table(cfg, wl), make_table(cfg, wl)
    ws_a = torch.empty(E.emb_bwd_workspace_size(a, n_bags, nnz), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty_like(ws_a)
    out_d = E.emb_lookup_fwd_dedup(a, off, q, cfg.pool, ws_a)
    out_r = E.emb_lookup_fwd_record(b, off, q, cfg.pool, ws_b)
    assert E.emb_check_device_flag(a) == 0
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    ref, A = T.forward(off.cpu().numpy(), q.cpu().numpy(), cfg.pool, cfg.wdtype, wl.values.cpu().numpy())
    tol = tol_of(cfg)
    gate("dedupe forward vs oracle", out_d.cpu().numpy(), ref, np.maximum(np.abs(ref), A), tol)
    gate("dedupe forward vs fused forward", out_d.cpu().numpy(), out_r.cpu().numpy().astype(np.float64),
         np.maximum(np.abs(ref), A), 2 * tol)          # each within tol of the oracle
    E.emb_bwd_adagrad_recorded(a, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws_a)
    E.emb_bwd_adagrad_recorded(b, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws_b)
    n_el = a.stats["n_elems"]
    (va, aa), (vb, ab) = _export(a, n_el, wl.values.dtype), _export(b, n_el, wl.values.dtype)
    it = torch.int16 if va.dtype == torch.float16 else torch.int32
    assert torch.equal(va.view(it), vb.view(it)) and torch.equal(aa, ab)
    keys = []
    for t, ws in ((a, ws_a), (b, ws_b)):
        uk = torch.empty(max(nnz, 1), dtype=torch.int64, device="cuda")
        nu = torch.zeros(1, dtype=torch.int64, device="cuda")
        E.emb_bwd_unique_keys(t, ws, uk, nu)
        keys.append(torch.sort(uk[:int(nu.item())]).values)
    assert torch.equal(keys[0], keys[1])
    assert E.emb_check_device_flag(a) == 0


def test_dedupe_forward_on_master_copy_tables_reads_the_f16_copy():
    cfg = CASES[4]
    wl = W.make(cfg, device="cuda")
    tbl = E.emb_table_create(cfg.dims, "f16m", wl.keys.cpu(), values=wl.values.float().cuda(),
                             capacity=cfg.capacity, acc_init=cfg.acc0)
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, wl.offsets.numel() - 1, wl.qkeys.numel()), dtype=torch.uint8,
                     device="cuda")
    out = E.emb_lookup_fwd_dedup(tbl, wl.offsets, wl.qkeys, cfg.pool, ws)
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    ref, A = T.forward(wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy(), cfg.pool, "f16",
                       oracle.f16_copy(wl.values.float().cpu().numpy()))
    gate("dedupe forward, master-copy table", out.cpu().numpy(), ref, np.maximum(np.abs(ref), A), 2e-3)
