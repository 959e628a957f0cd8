"""Failure paths on the GPU, with every failure injected on the host (no kernel
is made to fault or hang):

* a probe that gives up: a table whose probe bound is lowered, as a corrupted
  table would have it, must make every lookup stop at the bound, treat keys
  further from their home as misses and raise EMB_FLAG_PROBE_BOUND;
* a device allocation that fails at any point of emb_table_create must give
  EMB_ERR_OOM and leave none of the library's device memory allocated, and the
  library must keep working afterwards.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import gate, make_table

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _probe_lengths(keys, slots, cap):
    """Slots inspected to find each key: from its home (fmix64 mod cap) to its slot."""
    home = np.array([oracle.fmix64(int(k)) & (cap - 1) for k in keys], dtype=np.int64)
    return (slots - home) % cap + 1


def test_probe_gives_up_at_a_lowered_bound():
    cfg = W.config(1)
    wl = W.make(cfg, device="cuda")
    tbl = make_table(cfg, wl)
    keys = wl.keys.cpu().numpy()
    T = oracle.Table(keys, cfg.capacity, cfg.dims)
    slot_r, row_r = T.resolve(keys)
    plen = _probe_lengths(keys, slot_r, cfg.capacity)
    bound = 2
    near = plen <= bound
    assert (~near).sum() > 100 and near.sum() > 100
    E.emb_debug_set_probe_bound(tbl, bound)
    slot_x, row_x = E.emb_resolve(tbl, wl.keys.cuda())
    assert E.emb_check_device_flag(tbl) & E.EMB_FLAG_PROBE_BOUND
    slot_x, row_x = slot_x.cpu().numpy(), row_x.cpu().numpy()
    assert np.array_equal(slot_x[near], slot_r[near]) and np.array_equal(row_x[near], row_r[near])
    assert np.all(slot_x[~near] == -1) and np.all(row_x[~near] == -1)
    # the forward stops at the bound too: it pools exactly what the oracle pools
    # when every key beyond the bound is replaced by an absent key of its slot
    q = wl.qkeys.cpu().numpy()
    far = set(keys[~near].tolist())
    q2 = np.array([((k >> 48) << 48) | ((1 << 47) + i) if k in far else k for i, k in enumerate(q.tolist())],
                  dtype=np.int64)
    out = E.emb_lookup_fwd(tbl, wl.offsets, wl.qkeys, cfg.pool)
    assert E.emb_check_device_flag(tbl) & E.EMB_FLAG_PROBE_BOUND
    ref, A = T.forward(wl.offsets.cpu().numpy(), q2, cfg.pool, cfg.wdtype, wl.values.cpu().numpy())
    gate("pooled with far keys missing", out.cpu().numpy(), ref, np.maximum(np.abs(ref), A), 1e-5)
    # back to the table's own bound: every key resolves, no flag
    E.emb_debug_set_probe_bound(tbl, tbl.stats["max_cluster"] + 1)
    slot_y, _ = E.emb_resolve(tbl, wl.keys.cuda())
    assert E.emb_check_device_flag(tbl) == 0
    assert np.array_equal(slot_y.cpu().numpy(), slot_r)
    with pytest.raises(E.EmbError):
        E.emb_debug_set_probe_bound(tbl, 0)


@pytest.mark.parametrize("cfg,wdtype,host_values", [(W.scaled(W.config(4), 250, 32), None, True),
                                                     (W.scaled(W.config(5), 1000, 256), "f16m", False)],
                         ids=["ragged-host-values", "master-copy-device-values"])
def test_allocation_failure_at_every_point_of_create(cfg, wdtype, host_values):
    wl = W.make(cfg, device="cuda")
    wd = wdtype or cfg.wdtype
    vals = wl.values.float() if wd == "f16m" else wl.values
    vals = vals.cpu() if host_values else vals.cuda()
    torch.cuda.synchronize()
    keys_h = wl.keys.cpu()
    gc.collect()                      # tables of earlier tests are freed now, not during the counts
    gc.disable()
    try:
        live0 = E.emb_debug_live_device_allocs()
        created_after = None
        for after in range(0, 32):
            E.emb_debug_fail_device_alloc(after)
            try:
                tbl = E.emb_table_create(cfg.dims, wd, keys_h, values=vals, capacity=cfg.capacity,
                                         acc_init=cfg.acc0)
            except E.EmbError as e:
                assert e.name == "EMB_ERR_OOM", e
                assert E.emb_debug_live_device_allocs() == live0, f"leak after failing allocation {after}"
                continue
            finally:
                E.emb_debug_fail_device_alloc(-1)
            created_after = after
            break
    finally:
        gc.enable()
    assert created_after is not None and created_after >= 8      # every allocation point was failed once
    # the library still works: the table that was created runs a step
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    out = E.emb_lookup_fwd(tbl, off, q, cfg.pool)
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, off.numel() - 1, q.numel()), dtype=torch.uint8, device="cuda")
    E.emb_bwd_adagrad(tbl, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
    assert E.emb_check_device_flag(tbl) == 0 and torch.isfinite(out).all()
    gc.disable()
    try:
        tbl.close()
        assert E.emb_debug_live_device_allocs() == live0
    finally:
        gc.enable()
