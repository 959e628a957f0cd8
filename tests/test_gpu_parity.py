"""GPU parity: the sm_103a library against the CPU oracle, element by element,
at sizes the oracle finishes in seconds (several sort tiles, reduce chunks and
32-key probe rounds, with ragged tails), plus edge cases and determinism."""
import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E
from parity_util import check_step, gpu_step, make_table, report, tol_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


SMALL = [
    W.config(1),                                    # the tiny config, full size
    W.scaled(W.config(2), 100, 16),                 # 26 slots, f32 d64, mean, 2% absent
    W.scaled(W.config(3), 500, 64),                 # 100 slots, f16 d32, Zipf 1.2
    W.scaled(W.config(4), 250, 32),                 # 40 slots, ragged dims
    W.scaled(W.config(5), 1000, 256),               # 64 slots, f16 d128, mean, long bags, hot keys
]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_step_parity_small(cfg):
    wl = W.make(cfg, device="cuda")
    gs = gpu_step(cfg, wl)
    rep = check_step(cfg, wl, gs)
    report(f"small/{cfg.name}/unrecorded", **rep)


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_recorded_step_parity_and_identity(cfg):
    """The forward that records (row, bag) pairs + the backward that starts
    from them: oracle parity, and bit-identical to the unrecorded path."""
    wl = W.make(cfg, device="cuda")
    rec = gpu_step(cfg, wl, recorded=True)
    report(f"small/{cfg.name}/recorded", **check_step(cfg, wl, rec))
    ref = gpu_step(cfg, wl)
    assert torch.equal(rec.out, ref.out)
    assert np.array_equal(rec.values_out.view(np.uint8), ref.values_out.view(np.uint8))
    assert np.array_equal(rec.acc_out.view(np.uint8), ref.acc_out.view(np.uint8))
    assert np.array_equal(np.sort(rec.unique), np.sort(ref.unique))


# The 100M-key workload's structure (Zipf bag lengths up to 256, so many
# repeated keys within a bag; 5% absent keys; mean pooling) with rows of 4 and
# 8 elements: one and two lanes per row in the reduce, whose windows then hold
# one and two positions.
NARROW = [
    W.scaled(W.config(5), 1000, 256, name="64slot-4d-f32-mean", dims=(4,) * 64, wdtype="f32"),
    W.scaled(W.config(5), 1000, 256, name="64slot-8d-f16-mean", dims=(8,) * 64),
]


@pytest.mark.parametrize("cfg", NARROW, ids=lambda c: c.name)
def test_narrow_rows_parity_both_paths(cfg):
    wl = W.make(cfg, device="cuda")
    rec = gpu_step(cfg, wl, recorded=True)
    report(f"narrow/{cfg.name}/recorded", **check_step(cfg, wl, rec))
    ref = gpu_step(cfg, wl)
    assert torch.equal(rec.out, ref.out)
    assert np.array_equal(rec.values_out.view(np.uint8), ref.values_out.view(np.uint8))
    assert np.array_equal(rec.acc_out.view(np.uint8), ref.acc_out.view(np.uint8))


def test_recorded_backward_needs_its_forward():
    cfg = SMALL[0]
    wl = W.make(cfg, device="cuda")
    tbl = make_table(cfg, wl)
    off, q, g = wl.offsets, wl.qkeys, wl.grad
    n_bags, nnz = off.numel() - 1, q.numel()
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, n_bags, nnz), dtype=torch.uint8, device="cuda")
    with pytest.raises(E.EmbError) as ei:                         # nothing recorded yet
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    E.emb_lookup_fwd_record(tbl, off, q, cfg.pool, ws)
    other = torch.empty_like(ws)
    with pytest.raises(E.EmbError):                               # another workspace
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, other)
    with pytest.raises(E.EmbError):                               # another batch shape
        E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz - 1, cfg.pool, g, cfg.lr, cfg.eps, ws)
    E.emb_bwd_adagrad_recorded(tbl, n_bags, nnz, cfg.pool, g, cfg.lr, cfg.eps, ws)
    assert E.emb_check_device_flag(tbl) == 0


@pytest.mark.parametrize("cfg", [SMALL[1], SMALL[4]], ids=lambda c: c.name)
def test_host_values_upload_matches_device_upload(cfg):
    wl = W.make(cfg, device="cuda")
    a = gpu_step(cfg, wl, values_dev=True)
    b = gpu_step(cfg, wl, values_dev=False)
    assert torch.equal(a.out, b.out)
    assert np.array_equal(a.values_out, b.values_out) and np.array_equal(a.acc_out, b.acc_out)


@pytest.mark.parametrize("cfg", [SMALL[2], SMALL[4]], ids=lambda c: c.name)
def test_step_is_bitwise_deterministic(cfg):
    wl = W.make(cfg, device="cuda")
    a = gpu_step(cfg, wl)
    b = gpu_step(cfg, wl)
    assert torch.equal(a.out, b.out)
    assert np.array_equal(a.values_out.view(np.uint8), b.values_out.view(np.uint8))
    assert np.array_equal(a.acc_out.view(np.uint8), b.acc_out.view(np.uint8))


def _handmade(keys_per_slot, dims, wdtype, bags, pool="sum", seed=0, acc0=0.1):
    """A workload from explicit bag contents: bags[b][s] = list of keys."""
    rng = np.random.default_rng(seed)
    S = len(dims)
    keys = np.concatenate([(np.int64(s) << 48) | np.arange(1, keys_per_slot + 1, dtype=np.int64) * 1009
                           for s in range(S)])
    keys = keys[rng.permutation(keys.size)]
    cfg = W.Config("handmade", S, (keys_per_slot,) * S, tuple(dims), wdtype, len(bags), ("uniform", 1, 1),
                   1.0, 0.0, pool, 0.05, 1e-8, acc0, 1.0)
    lens = [len(bags[b][s]) for b in range(len(bags)) for s in range(S)]
    off = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    q = np.array([k for b in range(len(bags)) for s in range(S) for k in bags[b][s]], dtype=np.int64)
    n_el = keys_per_slot * sum(dims)
    dt = torch.float16 if wdtype == "f16" else torch.float32
    values = torch.from_numpy(rng.uniform(-0.05, 0.05, n_el).astype(np.float32)).to(dt)
    grad = torch.from_numpy(rng.standard_normal((len(bags), sum(dims))).astype(np.float32))
    wl = W.Workload(cfg, torch.from_numpy(keys), torch.from_numpy(off), torch.from_numpy(q), values, grad)
    return cfg, wl


def _key(s, i):
    return int((np.int64(s) << 48) | np.int64(i * 1009))


@pytest.mark.parametrize("wdtype,dims", [("f32", [16, 16]), ("f16", [128, 128]), ("f32", [8, 128])])
@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_edge_cases(wdtype, dims, pool):
    absent0 = _key(0, 5000)           # slot 0, never in the table
    bags = [
        [[], []],                                                 # empty bags
        [[absent0, absent0], [_key(1, 3)]],                       # all-miss bag; L=1 bag
        [[_key(0, 7)] * 3 + [absent0], [_key(1, 3), _key(1, 4)]],  # duplicates within a bag
        [[_key(0, i % 50 + 1) for i in range(1000)], []],         # a long bag (many 32-key rounds)
        [[_key(0, 1)] * 70, [_key(1, 9)] * 33],                    # key shared with the long bag
    ]
    cfg, wl = _handmade(200, dims, wdtype, bags, pool)
    gs = gpu_step(cfg, wl)
    rep = check_step(cfg, wl, gs)
    out = gs.out.cpu().numpy()
    assert np.all(out[0] == 0)                                    # empty bags pool to zero
    assert np.all(out[1, :dims[0]] == 0)                          # all-miss bag pools to zero
    print(rep)


@pytest.mark.parametrize("wdtype,D", [("f32", 64), ("f16", 128)])
def test_hot_key_spanning_many_reduce_chunks(wdtype, D):
    # one key repeated 100k times across 500 bags: its gradient segment spans
    # hundreds of reduce chunks and goes through the cross-chunk fixup
    hot = _key(0, 3)
    bags = [[[hot] * 200 + [_key(0, 1 + b % 40)]] for b in range(500)]
    cfg, wl = _handmade(64, [D], wdtype, bags, "mean")
    gs = gpu_step(cfg, wl)
    check_step(cfg, wl, gs)


@pytest.mark.parametrize("wdtype,D", [("f32", 64), ("f16", 128)])
@pytest.mark.parametrize("pool", ["sum", "mean"])
def test_reduce_windows_of_distinct_rows(wdtype, D, pool):
    # 4000 distinct keys, one occurrence each, then a hot key: every 32-position
    # window of the sorted pairs starts 32 rows (the reduce's crowded-window
    # path), and chunk edges cut both singleton runs and the hot segment
    bags = [[[_key(0, b * 40 + j + 1) for j in range(40)]] for b in range(100)]
    bags += [[[_key(0, 7)] * 300] for _ in range(4)]
    cfg, wl = _handmade(4096, [D], wdtype, bags, pool)
    gs = gpu_step(cfg, wl)
    check_step(cfg, wl, gs)


def test_nnz_zero_and_single_bag():
    cfg, wl = _handmade(16, [8], "f32", [[[]]])
    gs = gpu_step(cfg, wl)
    assert gs.unique.size == 0 and np.all(gs.out.cpu().numpy() == 0)
    check_step(cfg, wl, gs)


def test_slot_mismatch_and_bad_offsets_raise_device_flags():
    cfg, wl = _handmade(16, [8, 8], "f32", [[[_key(1, 2)], [_key(1, 3)]]])   # slot-1 key in a slot-0 bag
    tbl = make_table(cfg, wl)
    out = E.emb_lookup_fwd(tbl, wl.offsets.cuda(), wl.qkeys.cuda(), "sum")
    assert E.emb_check_device_flag(tbl) == E.EMB_FLAG_SLOT_MISMATCH
    assert np.all(out.cpu().numpy()[0, :8] == 0)                  # the mismatched key was skipped
    assert E.emb_check_device_flag(tbl) == 0                      # the flag word was cleared
    bad = torch.tensor([0, 5, 2], dtype=torch.int64, device="cuda")  # decreasing, and past nnz
    E.emb_lookup_fwd(tbl, bad, wl.qkeys.cuda(), "sum")
    assert E.emb_check_device_flag(tbl) & E.EMB_FLAG_BAD_OFFSETS


def test_host_side_rejections():
    cfg, wl = _handmade(16, [8, 8], "f32", [[[_key(0, 1)], [_key(1, 1)]]])
    tbl = make_table(cfg, wl)
    off, q = wl.offsets.cuda(), wl.qkeys.cuda()
    with pytest.raises(E.EmbError) as ei:
        E.emb_lookup_fwd(tbl, off[:2], q, "sum")                  # 1 bag: not a multiple of 2 slots
    assert ei.value.name == "EMB_ERR_INVALID_ARG"
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(E.EmbError) as ei:
        E.emb_bwd_adagrad(tbl, off, q, "sum", wl.grad.cuda(), 0.1, 1e-8, ws)
    assert ei.value.name == "EMB_ERR_WORKSPACE"
    with pytest.raises(E.EmbError) as ei:
        E.emb_table_create([8], "f32", torch.tensor([3, 3]), capacity=8)
    assert ei.value.name == "EMB_ERR_DUP_KEY"
    # pooled rows are written, and grad_out rows read, with 16-byte vector
    # accesses: a pointer 4 bytes past a 16-byte boundary is refused on the host
    buf = torch.empty(16 + 1, dtype=torch.float32, device="cuda")
    with pytest.raises(E.EmbError) as ei:
        E.emb_lookup_fwd(tbl, off, q, "sum", out=buf[1:])
    assert ei.value.name == "EMB_ERR_INVALID_ARG" and "aligned" in ei.value.message
    ws = torch.empty(E.emb_bwd_workspace_size(tbl, off.numel() - 1, q.numel()), dtype=torch.uint8, device="cuda")
    with pytest.raises(E.EmbError) as ei:
        E.emb_bwd_adagrad(tbl, off, q, "sum", buf[1:], 0.1, 1e-8, ws)
    assert ei.value.name == "EMB_ERR_INVALID_ARG" and "aligned" in ei.value.message


def test_resolve_sentinel_and_absent_keys():
    cfg, wl = _handmade(32, [8], "f32", [[[_key(0, 1)]]])
    tbl = make_table(cfg, wl)
    q = torch.tensor([-1, _key(0, 1), _key(0, 999), 0], dtype=torch.int64, device="cuda")
    slots, rows = E.emb_resolve(tbl, q)
    T = oracle.Table(wl.keys.numpy(), cfg.capacity, cfg.dims)
    s_r, r_r = T.resolve(q.cpu().numpy())
    assert np.array_equal(slots.cpu().numpy(), s_r) and np.array_equal(rows.cpu().numpy(), r_r)
    assert rows[0].item() == -1 and rows[1].item() >= 0


def test_slots_layout_and_export_roundtrip():
    cfg = SMALL[3]
    wl = W.make(cfg, device="cuda")
    gs = gpu_step(cfg, wl)
    T = oracle.Table(wl.keys.cpu().numpy(), cfg.capacity, cfg.dims)
    sk = torch.empty(cfg.capacity, dtype=torch.int64)
    sr = torch.empty(cfg.capacity, dtype=torch.int64)
    E.emb_table_slots(gs.table, sk, sr)                           # host destinations
    ok_, or_ = T.layout()
    assert np.array_equal(sk.numpy(), ok_) and np.array_equal(sr.numpy(), or_)
    # resume: a table created from the export pools exactly like the original
    t2 = E.emb_table_create(cfg.dims, cfg.wdtype, torch.from_numpy(gs.keys_out),
                            values=torch.from_numpy(gs.values_out), acc=torch.from_numpy(gs.acc_out),
                            capacity=cfg.capacity)
    off, q = wl.offsets.cuda(), wl.qkeys.cuda()
    o1 = E.emb_lookup_fwd(gs.table, off, q, cfg.pool)
    o2 = E.emb_lookup_fwd(t2, off, q, cfg.pool)
    assert torch.equal(o1, o2)
    ko = torch.empty(cfg.n_keys, dtype=torch.int64)
    vo = torch.empty(gs.values_out.size, dtype=wl.values.dtype)
    ao = torch.empty(gs.acc_out.size, dtype=torch.float32)
    E.emb_table_export(t2, ko, vo, ao)                            # host destinations
    assert np.array_equal(vo.numpy().view(np.uint8), gs.values_out.view(np.uint8))
    assert np.array_equal(ao.numpy(), gs.acc_out)
