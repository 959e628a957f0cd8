"""emb_bwd_adagrad_noalloc: the backward + Adagrad step for callers that cannot
allocate device memory (a framework's caching allocator already owns the GPU,
or a serving loop that forbids allocation during a step).  It must give the
same table update as emb_bwd_adagrad with a caller workspace, call after call,
through the C ABI.  This file sorts last so a stop-at-first-failure run has
already run every other test."""
import numpy as np
import pytest
import torch

import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import gate, make_table, tol_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _export(cfg, tbl, n_el, dt):
    vo = torch.empty(n_el, dtype=dt, device="cuda")
    ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, None, vo, ao)
    return vo.double().cpu().numpy(), ao.double().cpu().numpy()


@pytest.mark.parametrize("cfg", [W.config(1), W.scaled(W.config(5), 1000, 256)], ids=lambda c: c.name)
def test_noalloc_matches_workspace_path_on_two_calls(cfg):
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    assert E.emb_bwd_workspace_size(make_table(cfg, wl), n_bags, nnz) <= E.EMB_NOALLOC_SCRATCH_BYTES
    ref = make_table(cfg, wl)
    new = make_table(cfg, wl)
    ws = torch.empty(E.emb_bwd_workspace_size(ref, n_bags, nnz), dtype=torch.uint8, device="cuda")
    n_el = ref.stats["n_elems"]
    tol = tol_of(cfg)
    for call in range(2):
        E.emb_bwd_adagrad(ref, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
        E.emb_bwd_adagrad_noalloc(new, off, q, cfg.pool, g, cfg.lr, cfg.eps)
        assert E.emb_check_device_flag(new) == 0
        w_r, a_r = _export(cfg, ref, n_el, wl.values.dtype)
        w_x, a_x = _export(cfg, new, n_el, wl.values.dtype)
        gate(f"weights after call {call + 1}", w_x, w_r, np.maximum(np.abs(w_r), 1e-30), tol)
        gate(f"accumulators after call {call + 1}", a_x, a_r, a_r, tol)
        assert not np.array_equal(a_r, np.full_like(a_r, cfg.acc0))   # the step did update rows


def test_noalloc_rejects_batches_beyond_its_scratch():
    cfg = W.config(1)
    wl = W.make(cfg, device="cuda")
    tbl = make_table(cfg, wl)
    huge_nnz = 10_000_000            # far beyond the fixed scratch; rejected on the host, nothing queued
    need = E.emb_bwd_workspace_size(tbl, wl.offsets.numel() - 1, huge_nnz)
    assert need > E.EMB_NOALLOC_SCRATCH_BYTES
    fake_keys = torch.empty(1, dtype=torch.int64, device="cuda").expand(huge_nnz)
    with pytest.raises(E.EmbError) as ei:
        rc = E.lib().emb_bwd_adagrad_noalloc(tbl.handle, wl.offsets.data_ptr(), wl.offsets.numel() - 1,
                                             fake_keys.data_ptr(), huge_nnz, 0, wl.grad.data_ptr(),
                                             0.01, 1e-8, None)
        E._check(rc)
    assert ei.value.name == "EMB_ERR_UNSUPPORTED"
    assert "scratch" in ei.value.message
