"""GPU parity at the five workloads' full sizes, in the benchmark's launch
configuration (the recording forward emb_lookup_fwd_record + the recorded
backward emb_bwd_adagrad_recorded, as the benchmark times them; the
unrecorded pair emb_lookup_fwd + emb_bwd_adagrad on the 26-slot workload and
on the 100-slot one, whose batch takes the 4-lane forward teams),
on outputs the oracle computes one by one:

* slot resolution and hit/miss: bit-exact on a random sample of occurrences;
* pooled output: sampled bags (random and the longest ones);
* unique-key set: the whole set, against its definition written with torch
  library routines (isin + unique of the hit keys), plus oracle membership on
  a sample;
* per-key gradient + Adagrad: the hottest keys and a random sample of unique
  keys, through the oracle's per-key gradient map restricted to them;
* untouched rows: a random sample of rows outside the unique set stays
  bit-identical.
"""
import gc

import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import acc_scale, gate, plain_rel, report, split_plain_rel, tol_of, w_scale

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


class FullRun:
    def __init__(self, i, recorded=True):
        cfg = W.config(i)
        self.cfg = cfg
        dev = torch.device("cuda")
        rng = np.random.default_rng(100 + i)
        keys = W.table_keys(cfg, dev)
        off, q = W.batch(cfg, dev)
        grad = W.grad_out(cfg, dev)
        n_el = int(sum(cfg.vocab[s] * cfg.dims[s] for s in range(cfg.n_slots)))
        vals = W.w0_values(cfg, n_el, dev)
        self.keys_h = keys.cpu()
        tbl = E.emb_table_create(cfg.dims, cfg.wdtype, self.keys_h, values=vals, capacity=cfg.capacity,
                                 acc_init=cfg.acc0)
        del vals, keys
        torch.cuda.empty_cache()
        nnz, n_bags = q.numel(), off.numel() - 1
        # sampled rows (keys-array indices) read before the step, for the untouched-row check
        self.rand_rows = torch.from_numpy(rng.choice(cfg.n_keys, size=min(cfg.n_keys, 200_000),
                                                     replace=False)).cuda()
        self.w_before, self.a_before = E.emb_table_export_rows(tbl, self.rand_rows)
        out = torch.empty((cfg.batch, cfg.sum_dims), dtype=torch.float32, device=dev)
        ws = torch.empty(E.emb_bwd_workspace_size(tbl, n_bags, nnz), dtype=torch.uint8, device=dev)
        if recorded:   # the benchmark's step
            E.emb_lookup_fwd_record(tbl, off, q, cfg.pool, ws, out=out)
            E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, grad, cfg.lr, cfg.eps, ws)
        else:
            E.emb_lookup_fwd(tbl, off, q, cfg.pool, out=out)
            E.emb_bwd_adagrad(tbl, off, q, cfg.pool, grad, cfg.lr, cfg.eps, ws)
        self.path = "recorded" if recorded else "unrecorded"
        uk = torch.empty(nnz, dtype=torch.int64, device=dev)
        nu = torch.zeros(1, dtype=torch.int64, device=dev)
        E.emb_bwd_unique_keys(tbl, ws, uk, nu)
        self.flags = E.emb_check_device_flag(tbl)
        self.unique = uk[:int(nu.item())].clone()
        del ws, uk
        # occurrence sample for slot resolution
        occ = torch.from_numpy(rng.choice(nnz, size=min(nnz, 1_000_000), replace=False)).cuda()
        self.occ_keys = q[occ]
        self.occ_slots, self.occ_rows = E.emb_resolve(tbl, self.occ_keys)
        # the unique set by definition, with library routines: distinct table keys
        # among the occurrences whose slot field equals their bag's slot
        bag_of = torch.repeat_interleave(torch.arange(n_bags, device=dev), off[1:] - off[:-1])
        same_slot = (q >> 48) == (bag_of % cfg.n_slots)
        del bag_of
        present = torch.isin(q, self.keys_h.cuda())
        self.unique_def = torch.unique(q[present & same_slot])
        del present, same_slot
        self.out, self.tbl = out, tbl
        self.off_h, self.q_h, self.grad_h = off.cpu().numpy(), q.cpu().numpy(), grad.cpu().numpy()
        del off, q, grad
        torch.cuda.empty_cache()
        self.T = oracle.Table(self.keys_h.numpy(), cfg.capacity, cfg.dims)
        self.rng = rng

    def close(self):
        self.tbl.close()


@pytest.fixture(scope="module", params=[(1, True), (2, True), (2, False), (3, True), (3, False), (4, True), (5, True)],
                ids=lambda p: f"config{p[0]}-{'recorded' if p[1] else 'unrecorded'}")
def run(request):
    r = FullRun(*request.param)
    yield r
    r.close()
    del r
    gc.collect()
    torch.cuda.empty_cache()


def test_flags_clean(run):
    assert run.flags == 0


def test_resolve_bit_exact_on_sample(run):
    s_r, r_r = run.T.resolve(run.occ_keys.cpu().numpy())
    assert np.array_equal(run.occ_slots.cpu().numpy(), s_r)
    assert np.array_equal(run.occ_rows.cpu().numpy(), r_r)


def test_unique_key_set(run):
    got = torch.sort(run.unique).values
    assert torch.equal(got, run.unique_def)
    n = run.unique.numel()
    sample = run.unique[torch.randperm(n, device="cuda")[:min(n, 100_000)]].cpu().numpy()
    _, rows = run.T.resolve(sample)
    assert np.all(rows >= 0)


def _bag_sample(run, k=3000):
    cfg, rng = run.cfg, run.rng
    L = np.diff(run.off_h)
    longest = np.argsort(L)[-200:]
    rand = rng.choice(cfg.n_bags, size=min(k, cfg.n_bags), replace=False)
    return np.unique(np.concatenate([rand, longest]))


def _row_values(run, rows_ext):
    """Initial weights of keys-array rows from the generator, in compact form + row map."""
    cfg = run.cfg
    keys = run.keys_h.numpy()
    dims_rows = np.array(cfg.dims, dtype=np.int64)[keys[rows_ext] >> 48]
    eoff = torch.from_numpy(run.T.elem_offsets())
    vals = W.w0_rows(cfg, eoff, torch.from_numpy(rows_ext), torch.from_numpy(dims_rows)).numpy()
    row_map = np.full(keys.size, -1, dtype=np.int64)
    row_map[rows_ext] = np.concatenate([[0], np.cumsum(dims_rows)[:-1]]).astype(np.int64)
    return vals, row_map


def test_pooled_output_on_sampled_bags(run):
    cfg = run.cfg
    bags = _bag_sample(run)
    qs = np.concatenate([run.q_h[run.off_h[b]:run.off_h[b + 1]] for b in bags])
    _, rows = run.T.resolve(qs)
    rows = np.unique(rows[rows >= 0])
    vals, row_map = _row_values(run, rows)
    ref, A = run.T.forward(run.off_h, run.q_h, cfg.pool, cfg.wdtype, vals, row_map=row_map, bags=bags)
    out = run.out.cpu().numpy()
    cols = np.concatenate([[0], np.cumsum(cfg.dims)])
    got = np.concatenate([out[b // cfg.n_slots, cols[b % cfg.n_slots]:cols[b % cfg.n_slots + 1]] for b in bags])
    rel = gate("pooled", got, ref, np.maximum(np.abs(ref), A), tol_of(cfg))
    report(f"full/{cfg.name}/{run.path}", pooled_gate=rel, pooled_plain_rel=plain_rel(got, ref), bags=int(bags.size))


def test_adagrad_on_hot_and_sampled_keys(run):
    cfg, rng = run.cfg, run.rng
    uq = run.unique.cpu().numpy()
    vals_c, counts = np.unique(run.q_h, return_counts=True)
    hot = vals_c[np.argsort(counts)[-16:]]
    hot = hot[np.isin(hot, uq)]
    pick = np.unique(np.concatenate([hot, rng.choice(uq, size=min(uq.size, 2000), replace=False)]))
    uk, rows, goff, G, Ag = run.T.backward(run.off_h, run.q_h, cfg.pool, run.grad_h, key_filter=pick)
    assert np.array_equal(uk, pick)
    vals, row_map = _row_values(run, rows)
    md = max(cfg.dims)
    d = goff[1:] - goff[:-1]
    idx = np.concatenate([np.arange(row_map[r], row_map[r] + d[i]) for i, r in enumerate(rows)])
    w_r, acc_r = oracle.adagrad(G, vals[idx], np.full(idx.size, cfg.acc0, np.float32), cfg.lr, cfg.eps)
    wg, ag = E.emb_table_export_rows(run.tbl, torch.from_numpy(rows).cuda())
    mask = (np.arange(md)[None, :] < d[:, None]).reshape(-1)
    w_x = wg.cpu().numpy().reshape(-1)[mask].astype(np.float64)
    a_x = ag.cpu().numpy().reshape(-1)[mask]
    tol = tol_of(cfg)
    ga = gate("acc", a_x, acc_r, acc_scale(acc_r, G, Ag, tol), tol)
    gw = gate("weight", w_x, w_r.astype(np.float64), w_scale(w_r, vals[idx], acc_r, G, Ag, cfg.lr, tol), tol)
    cond = float((Ag / np.maximum(np.abs(G), 1e-300)).max())   # A_g / |g|: how much the key's terms cancel
    ap, apc, ncan = split_plain_rel(a_x, acc_r, G, Ag)
    wp, wpc, _ = split_plain_rel(w_x, w_r, G, Ag)
    report(f"full/{cfg.name}/{run.path}", keys=int(pick.size), hottest=int(hot.size), acc_gate=ga, w_gate=gw,
           acc_plain_rel=ap, acc_plain_rel_cancelling=apc, w_plain_rel=wp, w_plain_rel_cancelling=wpc,
           n_cancelling=ncan, n_elems=int(idx.size), max_cancellation=cond)


def test_untouched_rows_bit_identical(run):
    keys_rand = run.keys_h.numpy()[run.rand_rows.cpu().numpy()]
    untouched = torch.from_numpy(~np.isin(keys_rand, run.unique.cpu().numpy())).cuda()
    w_after, a_after = E.emb_table_export_rows(run.tbl, run.rand_rows)
    assert untouched.sum() > 1000
    itype = torch.int16 if run.w_before.dtype == torch.float16 else torch.int32
    assert torch.equal(w_after[untouched].contiguous().view(itype), run.w_before[untouched].contiguous().view(itype))
    assert torch.equal(a_after[untouched], run.a_before[untouched])
    touched = ~untouched
    if touched.any():
        assert not torch.equal(a_after[touched], run.a_before[touched])   # hit rows did move
