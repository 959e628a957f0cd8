"""emb_bwd_adagrad_noalloc: the backward + Adagrad step for callers that cannot
allocate device memory (a framework's caching allocator already owns the GPU,
or a serving loop that forbids allocation during a step).  It runs the same
kernels as emb_bwd_adagrad with a caller workspace, so it must give a
bitwise-identical table update, call after call, through the C ABI, whatever
an earlier call left in the library's shared scratch array.  This file sorts
last so a stop-at-first-failure run has already run every other test."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import acc_scale, elem_index, gate, make_table, tol_of, w_scale

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _export(tbl, n_el, dt):
    vo = torch.empty(n_el, dtype=dt, device="cuda")
    ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, None, vo, ao)
    return vo.cpu().numpy(), ao.cpu().numpy()


def _bits(a):
    return np.ascontiguousarray(a).view(np.uint8)


LARGE = W.scaled(W.config(5), 1000, 256)   # 64 slots, dim 128 f16, long bags, hot keys
SMALL = W.config(1)                        # 4 slots, dim 16 f32


@pytest.mark.parametrize("cfg", [SMALL, LARGE], ids=lambda c: c.name)
def test_noalloc_matches_workspace_path_on_two_calls(cfg):
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    ref = make_table(cfg, wl)
    new = make_table(cfg, wl)
    assert E.emb_bwd_workspace_size(ref, n_bags, nnz) <= E.EMB_NOALLOC_SCRATCH_BYTES
    ws = torch.empty(E.emb_bwd_workspace_size(ref, n_bags, nnz), dtype=torch.uint8, device="cuda")
    n_el = ref.stats["n_elems"]
    for call in range(2):
        E.emb_bwd_adagrad(ref, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
        E.emb_bwd_adagrad_noalloc(new, off, q, cfg.pool, g, cfg.lr, cfg.eps)
        assert E.emb_check_device_flag(new) == 0
        w_r, a_r = _export(ref, n_el, wl.values.dtype)
        w_x, a_x = _export(new, n_el, wl.values.dtype)
        assert np.array_equal(_bits(w_x), _bits(w_r)), f"weights differ after call {call + 1}"
        assert np.array_equal(_bits(a_x), _bits(a_r)), f"accumulators differ after call {call + 1}"
        assert not np.array_equal(a_r, np.full_like(a_r, cfg.acc0))   # the step did update rows


def _oracle_step(cfg, wl):
    """The oracle's table after one step from the initial state: (weights, accumulators)."""
    keys, off, q = wl.keys.cpu().numpy(), wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy()
    values, grad = wl.values.cpu().numpy(), wl.grad.cpu().numpy()
    T = oracle.Table(keys, cfg.capacity, cfg.dims)
    _, rows_u, _, G, Ag = T.backward(off, q, cfg.pool, grad)
    idx = elem_index(T.elem_offsets(), rows_u)
    w_r, acc_r = oracle.adagrad(G, values[idx], np.full(idx.size, cfg.acc0, np.float32), cfg.lr, cfg.eps)
    return idx, w_r, acc_r, G, Ag


def test_large_call_then_smaller_call_in_the_shared_scratch():
    """A large batch fills much of the shared array; a smaller one after it must
    not read anything the large one left there (every region it reads is
    written first).  Each is checked bitwise against the workspace path on its
    own table and against the oracle."""
    for cfg in (LARGE, SMALL):
        wl = W.make(cfg, device="cuda")
        off, q, g = wl.offsets, wl.qkeys, wl.grad
        n_bags, nnz = off.numel() - 1, q.numel()
        ref, new = make_table(cfg, wl), make_table(cfg, wl)
        ws = torch.empty(E.emb_bwd_workspace_size(ref, n_bags, nnz), dtype=torch.uint8, device="cuda")
        E.emb_bwd_adagrad(ref, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
        E.emb_bwd_adagrad_noalloc(new, off, q, cfg.pool, g, cfg.lr, cfg.eps)
        assert E.emb_check_device_flag(new) == 0
        n_el = ref.stats["n_elems"]
        w_r, a_r = _export(ref, n_el, wl.values.dtype)
        w_x, a_x = _export(new, n_el, wl.values.dtype)
        assert np.array_equal(_bits(w_x), _bits(w_r)) and np.array_equal(_bits(a_x), _bits(a_r)), cfg.name
        idx, w_o, a_o, G, Ag = _oracle_step(cfg, wl)
        tol = tol_of(cfg)
        gate(f"{cfg.name} accumulators", a_x[idx], a_o, acc_scale(a_o, G, Ag, tol), tol)
        gate(f"{cfg.name} weights", w_x[idx].astype(np.float64), w_o.astype(np.float64),
             w_scale(w_o, wl.values.cpu().numpy()[idx], a_o, G, Ag, cfg.lr, tol), tol)
        ref.close()
        new.close()


def test_malformed_offsets_after_a_full_call_update_nothing():
    """After a normal call has left its (row, bag) pairs in the shared array, a
    call whose offsets end before nnz (every bag empty) must update no row:
    positions outside every bag are absent pairs, never the earlier call's."""
    cfg = LARGE
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    tbl = make_table(cfg, wl)
    E.emb_bwd_adagrad_noalloc(tbl, off, q, cfg.pool, g, cfg.lr, cfg.eps)
    assert E.emb_check_device_flag(tbl) == 0
    n_el = tbl.stats["n_elems"]
    w0, a0 = _export(tbl, n_el, wl.values.dtype)
    empty = torch.zeros_like(off)                     # offsets[n_bags] = 0 < nnz: flagged, all bags empty
    E.emb_bwd_adagrad_noalloc(tbl, empty, q, cfg.pool, g, cfg.lr, cfg.eps)
    assert E.emb_check_device_flag(tbl) & E.EMB_FLAG_BAD_OFFSETS
    w1, a1 = _export(tbl, n_el, wl.values.dtype)
    assert np.array_equal(_bits(w1), _bits(w0)) and np.array_equal(_bits(a1), _bits(a0))


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
