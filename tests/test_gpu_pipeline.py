"""The batch pipeline (emb_pipeline_*): uploads of the next batches overlapped
with the current step, pooled outputs copied back on a second stream.  A
pipelined run over several different batches must match the oracle step by
step (the table after each step, and each step's pooled output computed from
the table the previous steps left), and be bit-identical to the same steps
made with direct calls one after the other."""
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


def _batches(cfg, wl, n):
    """n different CSR batches from the workload: the samples in rotated order,
    each with its own grad_out (host, pinned)."""
    off, q = wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy()
    S, B = cfg.n_slots, cfg.batch
    g = wl.grad.cpu()
    out = []
    for k in range(n):
        order = np.roll(np.arange(B), 17 * k)
        segs, lens = [], []
        for b in order:
            lo, hi = off[b * S], off[(b + 1) * S]
            segs.append(q[lo:hi])
            lens.append(np.diff(off[b * S:(b + 1) * S + 1]))
        o = np.concatenate([[0], np.cumsum(np.concatenate(lens))]).astype(np.int64)
        qq = np.concatenate(segs).astype(np.int64)
        gk = (g[torch.from_numpy(order)] * (1.0 - 0.3 * k)).contiguous()
        out.append((torch.from_numpy(o).pin_memory(), torch.from_numpy(qq).pin_memory(), gk.pin_memory()))
    return out


@pytest.mark.parametrize("cfg", [W.scaled(W.config(2), 100, 16), W.scaled(W.config(5), 1000, 256)],
                         ids=lambda c: c.name)
def test_pipelined_steps_match_the_oracle_and_direct_calls(cfg):
    steps, depth = 4, 2
    wl = W.make(cfg, device="cuda")
    batches = _batches(cfg, wl, steps)
    max_bags = cfg.batch * cfg.n_slots
    max_nnz = max(b[1].numel() for b in batches)
    # direct calls, one step after the other
    direct = make_table(cfg, wl)
    ws = torch.empty(E.emb_bwd_workspace_size(direct, max_bags, max_nnz), dtype=torch.uint8, device="cuda")
    outs_direct = []
    for o, q, g in batches:
        od, qd, gd = o.cuda(), q.cuda(), g.cuda()
        outs_direct.append(E.emb_lookup_fwd_record(direct, od, qd, cfg.pool, ws).cpu())
        E.emb_bwd_adagrad_recorded(direct, od.numel() - 1, qd.numel(), cfg.pool, gd, cfg.lr, cfg.eps, ws)
    # the pipeline, submitting one batch ahead of the step
    tbl = make_table(cfg, wl)
    pipe = E.Pipeline(tbl, max_bags, max_nnz, depth=depth, upload_grad=True)
    outs_h = [torch.empty((cfg.batch, cfg.sum_dims), dtype=torch.float32).pin_memory() for _ in range(steps)]
    keys = wl.keys.cpu().numpy()
    T = oracle.Table(keys, cfg.capacity, cfg.dims)
    eoff = T.elem_offsets()
    w = wl.values.cpu().numpy().copy()
    acc = np.full(w.size, cfg.acc0, np.float32)
    n_el = tbl.stats["n_elems"]
    tol = tol_of(cfg)
    tickets = [pipe.submit(*batches[0])]
    for k in range(steps):
        if k + 1 < steps:
            tickets.append(pipe.submit(*batches[k + 1]))          # the next upload overlaps this step
        pipe.forward(tickets[k], cfg.pool, out_h=outs_h[k])
        pipe.backward_adagrad(tickets[k], cfg.lr, cfg.eps)
        pipe.wait(tickets[k])
        o, q, g = (x.numpy() for x in batches[k])
        # pooled output: the oracle's forward on the table as the previous steps left it
        ref, A = T.forward(o, q, cfg.pool, cfg.wdtype, w)
        gate(f"pooled, step {k + 1}", outs_h[k].numpy(), ref, np.maximum(np.abs(ref), A), tol)
        assert torch.equal(outs_h[k], outs_direct[k])
        # the update
        _, rows_u, _, G, Ag = T.backward(o, q, cfg.pool, g)
        idx = elem_index(eoff, rows_u)
        w_old = w[idx].copy()
        w[idx], acc[idx] = oracle.adagrad(G, w_old, acc[idx], cfg.lr, cfg.eps)
        vo = torch.empty(n_el, dtype=wl.values.dtype, device="cuda")
        ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
        E.emb_table_export(tbl, None, vo, ao)
        vx, ax = vo.cpu().numpy(), ao.cpu().numpy()
        gate(f"accumulators, step {k + 1}", ax[idx], acc[idx], acc_scale(acc[idx], G, Ag, tol), tol)
        gate(f"weights, step {k + 1}", vx[idx].astype(np.float64), w[idx].astype(np.float64),
             w_scale(w[idx], w_old, acc[idx], G, Ag, cfg.lr, tol), tol)
        w[idx], acc[idx] = vx[idx], ax[idx]       # continue from the GPU's state (errors do not compound)
    # bit-identical to the direct calls
    va = torch.empty(n_el, dtype=wl.values.dtype, device="cuda")
    vb = torch.empty_like(va)
    aa = torch.empty(n_el, dtype=torch.float32, device="cuda")
    ab = torch.empty_like(aa)
    E.emb_table_export(direct, None, va, aa)
    E.emb_table_export(tbl, None, vb, ab)
    assert torch.equal(va.view(torch.int16 if va.dtype == torch.float16 else torch.int32),
                       vb.view(torch.int16 if vb.dtype == torch.float16 else torch.int32))
    assert torch.equal(aa, ab)
    assert E.emb_check_device_flag(tbl) == 0
    pipe.close()


def test_pipeline_order_rules():
    cfg = W.config(1)
    wl = W.make(cfg, device="cuda")
    tbl = make_table(cfg, wl)
    o, q = wl.offsets.cpu().pin_memory(), wl.qkeys.cpu().pin_memory()
    pipe = E.Pipeline(tbl, o.numel() - 1, q.numel(), depth=2)
    t0 = pipe.submit(o, q)
    t1 = pipe.submit(o, q)
    with pytest.raises(E.EmbError):                  # both sets held: a third batch must wait for a backward
        pipe.submit(o, q)
    with pytest.raises(E.EmbError):                  # backward before forward
        pipe.backward_adagrad(t0, cfg.lr, cfg.eps, grad_out=wl.grad)
    pipe.forward(t0, cfg.pool)
    with pytest.raises(E.EmbError):                  # no grad_out given and none uploaded
        pipe.backward_adagrad(t0, cfg.lr, cfg.eps)
    pipe.backward_adagrad(t0, cfg.lr, cfg.eps, grad_out=wl.grad)
    pipe.forward(t1, cfg.pool)
    pipe.release(t1)                                 # forward-only use of a batch
    pipe.wait(t1)
    t2 = pipe.submit(o, q)                           # sets are free again
    assert t2 == 2
    pipe.forward(t2, cfg.pool)
    pipe.release(t2)
    pipe.wait(t0)                                    # a ticket whose set was reused
    pipe.wait(t2)
    assert E.emb_check_device_flag(tbl) == 0
    pipe.close()
