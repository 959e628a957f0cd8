"""GPU parity of row-wise Adagrad (tables created with
optimizer="rowwise_adagrad": one float32 accumulator per key,
a += sum_d g_d^2 / D, then w_d -= lr g_d / (sqrt(a) + eps) on each of the
row's D elements) against the oracle's row-wise Adagrad, over several steps in
a row, through both backward paths (recorded and unrecorded, bit-identical to
each other), on master-copy tables, on rows wide enough for several column
blocks per lane, and on a batch of more than 2^24 lookups whose hot rows take
the fold kernel.

Gates (u = 2^-24; per element dg = DG_ULPS u A_g + u |g|, the bound on the
float32 per-key gradient's error from parity_util, taken for every key; per
row D its dim and m = sum_d g_d^2 / D):
  accumulator  |x - r| <= tol r + 2 gamma_D m + sum_d (2 |g_d| dg_d + dg_d^2) / D
               (the two sides sum the D float32 squares in different orders,
               each within gamma_D = D u / (1 - D u) of the exact sum, relative;
               the gradient's error moves each square by 2 |g| dg + dg^2)
  weight       |x - r| <= tol max(|w'|, |w_old|) + 10 u |s| + lr dg / den + |s| da / (2 a')
               (s = lr g / den the step, den = sqrt(a') + eps; 10 u the step's
               roundings: 4 on the oracle's side (product, sqrt, add, divide),
               6 on the kernel's (product, rsqrtf's 2 ulp and its product, add,
               __fdividef's 2 ulp); da the accumulator's bound above: a relative
               change da / a' of a' moves sqrt(a') by half of it)
"""
import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import DG_ULPS, U32, elem_index, gate, report, tol_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


CASES = [
    W.config(1),                                    # 4 slots, dim 16 f32, sum: 4-lane groups
    W.scaled(W.config(2), 100, 16),                 # 26 slots, dim 64 f32, mean, absent keys
    W.scaled(W.config(3), 500, 64),                 # 100 slots, dim 32 f16, sum
    W.scaled(W.config(4), 250, 32),                 # ragged dims 8..128
    W.scaled(W.config(1), 4, 1, name="4slot-256d-f32", dims=(256,) * 4),   # two column blocks per lane
    W.scaled(W.config(1), 4, 1, name="4slot-512d-f32", dims=(512,) * 4),   # four
]
MASTER = W.scaled(W.config(5), 1000, 256)           # dim 128, f32 masters + f16 copy
FOLD = W.scaled(W.config(5), 16, 16)                # > 2^24 lookups: the fold kernel runs


def _table(cfg, keys_h, values, wdtype=None, acc=None):
    wd = wdtype or cfg.wdtype
    vals = values.float() if wd == "f16m" else values
    return E.emb_table_create(cfg.dims, wd, keys_h, values=vals, acc=acc, capacity=cfg.capacity,
                              acc_init=cfg.acc0, optimizer="rowwise_adagrad")


def _state(tbl, n_el, n_keys, wdt):
    vo = torch.empty(n_el, dtype=wdt, device="cuda")
    ao = torch.empty(n_keys, dtype=torch.float32, device="cuda")
    E.emb_table_export(tbl, None, vo, ao)
    return vo.cpu().numpy(), ao.cpu().numpy()


def _check_rows(name, tol, lr, eps, G, goff, Ag, w_old, a_old, w_x, a_x):
    """The oracle's row-wise step on (w_old, a_old) against the kernel's
    (w_x, a_x), rows given by goff; returns the oracle's (w', a')."""
    w_r, a_r = oracle.rowwise_adagrad(G, goff, w_old, a_old, lr, eps)
    D = np.diff(goff).astype(np.float64)
    assert D.min() > 0
    starts = goff[:-1]
    rowid = np.repeat(np.arange(D.size), np.diff(goff))
    absg = np.abs(G)
    dg = DG_ULPS * U32 * np.asarray(Ag, np.float64) + U32 * absg
    gam = D * U32 / (1 - D * U32)
    m = np.add.reduceat(G * G, starts) / D
    da = 2 * gam * m + np.add.reduceat(2 * absg * dg + dg * dg, starts) / D
    ar = a_r.astype(np.float64)
    ga = gate(f"{name}: accumulator", a_x, ar, ar + da / tol, tol)
    den = (np.sqrt(ar) + eps)[rowid]
    s = np.abs(lr * G / den)
    wsc = np.maximum(np.abs(w_r.astype(np.float64)), np.abs(w_old.astype(np.float64)))
    wsc = wsc + (10 * U32 * s + lr * dg / den + s * (da + 4 * U32 * ar)[rowid] / (2 * ar[rowid])) / tol
    gw = gate(f"{name}: weights", np.asarray(w_x, np.float64), w_r.astype(np.float64), wsc, tol)
    return w_r, a_r, ga, gw


def _run(cfg, wdtype=None, steps=3):
    wd = wdtype or cfg.wdtype
    wl = W.make(cfg, device="cuda")
    off, q = wl.offsets, wl.qkeys
    n_bags, nnz = off.numel() - 1, q.numel()
    keys_h = wl.keys.cpu()
    rec, unr = _table(cfg, keys_h, wl.values, wd), _table(cfg, keys_h, wl.values, wd)
    ws = torch.empty(E.emb_bwd_workspace_size(rec, n_bags, nnz), dtype=torch.uint8, device="cuda")
    ws2 = torch.empty_like(ws)
    n_el, n_keys = rec.stats["n_elems"], cfg.n_keys
    wdt = torch.float16 if wd == "f16" else torch.float32
    T = oracle.Table(keys_h.numpy(), cfg.capacity, cfg.dims)
    eoff = T.elem_offsets()
    offn, qn = off.cpu().numpy(), q.cpu().numpy()
    w = wl.values.cpu().numpy().copy()
    if wd == "f16m":
        w = w.astype(np.float32)
    a = np.full(n_keys, cfg.acc0, np.float32)
    tol = tol_of(cfg) if wd != "f16m" else 1e-5
    for k in range(steps):
        g = torch.roll(wl.grad, shifts=k, dims=0) * (1.0, -0.5, 2.0)[k % 3]   # a different gradient each step
        E.emb_lookup_fwd_record(rec, off, q, cfg.pool, ws)
        E.emb_bwd_adagrad_recorded(rec, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws)
        E.emb_bwd_adagrad(unr, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws2)
        assert E.emb_check_device_flag(rec) == 0 and E.emb_check_device_flag(unr) == 0
        w_x, a_x = _state(rec, n_el, n_keys, wdt)
        w_u, a_u = _state(unr, n_el, n_keys, wdt)
        assert np.array_equal(w_x.view(np.uint8), w_u.view(np.uint8))      # both backward paths: bit-identical
        assert np.array_equal(a_x.view(np.uint8), a_u.view(np.uint8))
        _, rows_u, goff, G, Ag = T.backward(offn, qn, cfg.pool, g.cpu().numpy())
        idx = elem_index(eoff, rows_u)
        w_r, a_r, ga, gw = _check_rows(f"{cfg.name}/{wd} step {k + 1}", tol, cfg.lr, cfg.eps, G, goff, Ag,
                                       w[idx], a[rows_u], w_x[idx], a_x[rows_u])
        # keys the batch does not hit: weights and accumulator bit-identical to before
        untouched = np.ones(n_el, bool)
        untouched[idx] = False
        assert np.array_equal(w_x[untouched].view(np.uint8), w[untouched].astype(w_x.dtype).view(np.uint8))
        cold = np.ones(n_keys, bool)
        cold[rows_u] = False
        assert np.array_equal(a_x[cold], a[cold])
        # the next step starts both sides from the kernel's state, so that each
        # step is checked from identical inputs
        w[idx], a[rows_u] = w_x[idx], a_x[rows_u]
        report(f"rowwise/{cfg.name}/{wd}/step{k + 1}", acc_gate=ga, w_gate=gw, rows=int(rows_u.size),
               n_elems=int(idx.size))
    return rec, w, wl


@pytest.mark.parametrize("cfg", CASES, ids=lambda c: c.name)
def test_rowwise_steps_match_the_oracle(cfg):
    _run(cfg)


def test_rowwise_on_master_copy_tables_refreshes_the_forward_copy():
    cfg = MASTER
    tbl, w, wl = _run(cfg, "f16m", steps=2)
    out = E.emb_lookup_fwd(tbl, wl.offsets, wl.qkeys, cfg.pool)
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    ref, A = T.forward(wl.offsets.cpu().numpy(), wl.qkeys.cpu().numpy(), cfg.pool, "f16", oracle.f16_copy(w))
    gate("forward on the refreshed f16 copy", out.cpu().numpy(), ref, np.maximum(np.abs(ref), A), 2e-3)


def test_rowwise_hot_rows_through_the_fold():
    """More than 2^24 lookups: rows that span whole blocks of sub-chunks have
    them folded before the fixup applies the row-wise update.  Checked on the
    hottest keys (the folded ones) and a random sample, from weights read
    before the step."""
    cfg = FOLD
    rng = np.random.default_rng(7)
    keys = W.table_keys(cfg, "cuda")
    off, q = W.batch(cfg, "cuda")
    nnz, n_bags = q.numel(), off.numel() - 1
    assert nnz >= 1 << 24
    grad = W.grad_out(cfg, "cuda")
    n_el = int(sum(cfg.vocab[s] * cfg.dims[s] for s in range(cfg.n_slots)))
    keys_h = keys.cpu()
    tbl = _table(cfg, keys_h, W.w0_values(cfg, n_el, "cuda"))
    T = oracle.Table(keys_h.numpy(), cfg.capacity, cfg.dims)
    q_h = q.cpu().numpy()
    vals_c, counts = np.unique(q_h, return_counts=True)
    cand = np.unique(np.concatenate([vals_c[np.argsort(counts)[-16:]], rng.choice(vals_c, 2000, replace=False)]))
    _, rows_c = T.resolve(cand)
    cand, rows_c = cand[rows_c >= 0], rows_c[rows_c >= 0]
    w_before, a_before = E.emb_table_export_rows(tbl, torch.from_numpy(rows_c).cuda())
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, n_bags, nnz), dtype=torch.uint8, device="cuda")
    E.emb_lookup_fwd_record(tbl, off, q, cfg.pool, ws)
    E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, grad, cfg.lr, cfg.eps, ws)
    assert E.emb_check_device_flag(tbl) == 0
    w_after, a_after = E.emb_table_export_rows(tbl, torch.from_numpy(rows_c).cuda())
    uk, rows, goff, G, Ag = T.backward(off.cpu().numpy(), q_h, cfg.pool, grad.cpu().numpy(), key_filter=cand)
    # below 2^27 lookups a sub-chunk holds 128 positions: the hottest row spans
    # at least one folded block of 32 of them
    assert counts.max() >= 32 * 128
    pos = {int(r): i for i, r in enumerate(rows_c)}
    sel = np.array([pos[int(r)] for r in rows], dtype=np.int64)
    d = np.diff(goff)
    md = max(cfg.dims)
    mask = (np.arange(md)[None, :] < d[:, None]).reshape(-1)
    w_old = w_before.cpu().numpy()[sel].reshape(-1)[mask]
    w_x = w_after.cpu().numpy()[sel].reshape(-1)[mask]
    _, _, ga, gw = _check_rows(f"{cfg.name} hot + sampled rows", tol_of(cfg), cfg.lr, cfg.eps, G, goff, Ag, w_old,
                               a_before.cpu().numpy()[sel], w_x, a_after.cpu().numpy()[sel])
    # keys of the sample that the batch did not hit keep their state bit for bit
    cold = ~np.isin(cand, uk)
    assert torch.equal(a_after[torch.from_numpy(cold).cuda()], a_before[torch.from_numpy(cold).cuda()])
    report(f"rowwise/{cfg.name}/fold", acc_gate=ga, w_gate=gw, rows=int(rows.size), nnz=int(nnz))
    tbl.close()


def test_rowwise_state_round_trip_and_no_alloc_entry():
    """export (weights, per-key accumulators), create from them, step both:
    bit-identical; the allocation-free backward gives the same bits as the one
    with a caller workspace; export_rows returns one accumulator per row."""
    cfg = CASES[1]
    wl = W.make(cfg, device="cuda")
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    keys_h = wl.keys.cpu()
    a = _table(cfg, keys_h, wl.values)
    ws = torch.empty(E.emb_bwd_workspace_size(a, n_bags, nnz), dtype=torch.uint8, device="cuda")
    E.emb_bwd_adagrad(a, off, q, cfg.pool, g, cfg.lr, cfg.eps, ws)
    n_el = a.stats["n_elems"]
    w0, a0 = _state(a, n_el, cfg.n_keys, torch.float32)
    rows = torch.arange(0, cfg.n_keys, 7, device="cuda")
    wr, ar = E.emb_table_export_rows(a, rows)
    assert ar.shape == (rows.numel(),) and torch.equal(ar.cpu(), torch.from_numpy(a0)[rows.cpu()])
    b = _table(cfg, keys_h, torch.from_numpy(w0), acc=torch.from_numpy(a0))
    c = _table(cfg, keys_h, torch.from_numpy(w0), acc=torch.from_numpy(a0).cuda())
    E.emb_bwd_adagrad(a, off, q, cfg.pool, -g, cfg.lr, cfg.eps, ws)
    E.emb_bwd_adagrad(b, off, q, cfg.pool, -g, cfg.lr, cfg.eps, ws)
    E.emb_bwd_adagrad_noalloc(c, off, q, cfg.pool, -g, cfg.lr, cfg.eps)
    sa = _state(a, n_el, cfg.n_keys, torch.float32)
    for t in (b, c):
        st = _state(t, n_el, cfg.n_keys, torch.float32)
        for x, y in zip(sa, st):
            assert np.array_equal(x.view(np.uint8), y.view(np.uint8))


def test_rowwise_table_refuses_ftrl_and_z():
    cfg = CASES[0]
    wl = W.make(cfg, device="cuda")
    t = _table(cfg, wl.keys.cpu(), wl.values)
    ws = torch.empty(1 << 22, dtype=torch.uint8, device="cuda")
    with pytest.raises(E.EmbError) as ei:
        E.emb_bwd_ftrl(t, wl.offsets, wl.qkeys, cfg.pool, wl.grad, 0.05, 1.0, 0.0, 0.0, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    with pytest.raises(E.EmbError):
        E.emb_table_export_z(t, torch.empty(t.stats["n_elems"], dtype=torch.float32, device="cuda"))
