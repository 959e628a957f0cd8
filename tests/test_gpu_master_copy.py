"""Master-copy tables (EMB_F16_MASTER): the forward gathers the f16 copy of
each row, the update works on the f32 master rows, and after the step the f16
copy of every updated row is its master rounded to nearest-even (JD article
3.2.3: FP16 storage and compute, an FP32 copy of the weights for the update).
Parity against the oracle composed the same way: its forward on the rounded
masters, its f32 Adagrad on the masters."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import acc_scale, elem_index, gate, gpu_step, tol_of, w_scale
from test_gpu_parity import _handmade, _key

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _master_cfg(cfg):
    return dataclasses.replace(cfg, wdtype="f16m", name=cfg.name + "/f16m")


def _check_master_step(cfg, wl, gs):
    tol = tol_of(cfg)
    keys = wl.keys.cpu().numpy()
    off, q = wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy()
    master0 = wl.values.cpu().numpy()
    assert master0.dtype == np.float32
    grad = wl.grad.cpu().numpy()
    T = oracle.Table(keys, cfg.capacity, cfg.dims)
    assert gs.flags == 0
    # the forward reads the f16 copy of the initial masters
    out_r, A = T.forward(off, q, cfg.pool, "f16", oracle.f16_copy(master0))
    gate("pooled (f16 copy)", gs.out.cpu().numpy(), out_r, np.maximum(np.abs(out_r), A), tol)
    # the update works on the f32 masters
    uk_r, rows_u, goff, G, Ag = T.backward(off, q, cfg.pool, grad)
    assert np.array_equal(np.sort(gs.unique), uk_r)
    idx = elem_index(T.elem_offsets(), rows_u)
    acc0 = np.full(idx.size, cfg.acc0, dtype=np.float32)
    w_r, acc_r = oracle.adagrad(G, master0[idx], acc0, cfg.lr, cfg.eps)
    assert gs.values_out.dtype == np.float32                     # export returns the masters
    gate("accumulators", gs.acc_out[idx], acc_r, acc_scale(acc_r, G, Ag, tol), tol)
    gate("master weights", gs.values_out[idx].astype(np.float64), w_r.astype(np.float64),
         w_scale(w_r, master0[idx], acc_r, G, Ag, cfg.lr, tol), tol)
    untouched = np.ones(master0.size, dtype=bool)
    untouched[idx] = False
    assert np.array_equal(gs.values_out[untouched].view(np.int32), master0[untouched].view(np.int32))
    assert np.all(gs.acc_out[untouched] == np.float32(cfg.acc0))
    # the f16 copy followed the updated masters: a second forward over the same
    # batch reads exactly the masters the step left, rounded
    out2 = E.emb_lookup_fwd(gs.table, wl.offsets.cuda(), wl.qkeys.cuda(), cfg.pool)
    out2_r, A2 = T.forward(off, q, cfg.pool, "f16", oracle.f16_copy(gs.values_out))
    gate("pooled after the update", out2.cpu().numpy(), out2_r, np.maximum(np.abs(out2_r), A2), tol)
    assert not np.array_equal(out2.cpu().numpy(), gs.out.cpu().numpy())   # the copy did change


@pytest.mark.parametrize("cfg", [_master_cfg(W.scaled(W.config(5), 1000, 256)),
                                 _master_cfg(W.scaled(W.config(3), 500, 64))], ids=lambda c: c.name)
@pytest.mark.parametrize("recorded", [False, True], ids=["unrecorded", "recorded"])
def test_master_copy_step_parity(cfg, recorded):
    wl = W.make(cfg, device="cuda")
    gs = gpu_step(cfg, wl, recorded=recorded)
    _check_master_step(cfg, wl, gs)


def test_master_copy_hot_key_across_reduce_chunks():
    # a key repeated 100k times: its update goes through the cross-chunk fixup,
    # and its f16 copy must still be refreshed
    hot = _key(0, 3)
    bags = [[[hot] * 200 + [_key(0, 1 + b % 40)]] for b in range(500)]
    cfg, wl = _handmade(64, [128], "f16m", bags, "mean")
    assert wl.values.dtype == torch.float32
    gs = gpu_step(cfg, wl)
    _check_master_step(cfg, wl, gs)
