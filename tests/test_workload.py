"""The seeded synthetic input generator (CPU only)."""
import numpy as np
import pytest
import torch

import workload as W


def _np_mix(seed, stream, ctr):
    M = np.uint64
    with np.errstate(over="ignore"):
        x = ctr.astype(np.uint64) + M((seed * 0xD1B54A32D192ED03 + stream * 0xAEF17502108EF2D9
                                       + 0x9E3779B97F4A7C15) & ((1 << 64) - 1))
        x = (x ^ (x >> M(30))) * M(0xBF58476D1CE4E5B9)
        x = (x ^ (x >> M(27))) * M(0x94D049BB133111EB)
        return x ^ (x >> M(31))


def test_mixer_wraps_like_uint64():
    c = np.arange(0, 200000, dtype=np.int64) * 104729 - 7
    a = W.mix64(5, 3, torch.from_numpy(c)).numpy().view(np.uint64)
    assert np.array_equal(a, _np_mix(5, 3, c))
    u = W.uniform01(5, 3, torch.from_numpy(c)).numpy()
    assert u.min() >= 0.0 and u.max() < 1.0 and abs(u.mean() - 0.5) < 0.01


SMALL = [W.config(1), W.scaled(W.config(2), 200, 64), W.scaled(W.config(3), 1000, 256),
         W.scaled(W.config(4), 1000, 128), W.scaled(W.config(5), 1000, 512)]


@pytest.mark.parametrize("cfg", SMALL, ids=lambda c: c.name)
def test_workload_structure(cfg):
    a = W.make(cfg)
    b = W.make(cfg)
    for x, y in [(a.keys, b.keys), (a.offsets, b.offsets), (a.qkeys, b.qkeys), (a.values, b.values), (a.grad, b.grad)]:
        assert torch.equal(x, y)                                     # deterministic
    keys = a.keys.numpy()
    assert np.unique(keys).size == keys.size == cfg.n_keys
    slot = keys >> 48
    assert np.array_equal(np.bincount(slot, minlength=cfg.n_slots), np.array(cfg.vocab))
    off = a.offsets.numpy()
    L = np.diff(off)
    assert off[0] == 0 and np.all(L >= 1) and off.size == cfg.n_bags + 1
    kind = cfg.bag_len[0]
    hi = cfg.bag_len[2] if kind in ("uniform", "geometric") else cfg.bag_len[3]
    assert L.max() <= hi
    q = a.qkeys.numpy()
    bag_slot = np.repeat(np.arange(cfg.n_bags) % cfg.n_slots, L)
    assert np.array_equal(q >> 48, bag_slot)                         # bag (b, s) holds slot-s keys
    present = np.isin(q, keys)
    if cfg.absent == 0:
        assert present.all()
    else:
        assert abs((~present).mean() - cfg.absent) < 0.35 * cfg.absent + 0.01
    v = a.values.float().numpy()
    assert v.size == sum(cfg.vocab[s] * cfg.dims[s] for s in range(cfg.n_slots))
    assert v.min() >= -0.05 and v.max() <= 0.05
    g = a.grad.numpy()
    assert g.shape == (cfg.batch, cfg.sum_dims)
    assert abs(g.std() - cfg.grad_std) < 0.05 * cfg.grad_std


def test_zipf_head_frequency():
    cfg = W.scaled(W.config(1), 1, 1, batch=4096)
    _, q = W.batch(cfg)
    q = q.numpy()
    s0 = q[(q >> 48) == 0]
    V, s = cfg.vocab[0], cfg.zipf_s
    p1 = 1.0 / np.sum(np.arange(1, V + 1, dtype=np.float64) ** -s)
    a, c = W._slot_affine(cfg, "cpu")
    top = int(((a[0] * 0 + c[0]) & ((1 << 48) - 1)).item())        # rank 0 of slot 0
    f = np.mean(s0 == top)
    assert abs(f - p1) < 0.15 * p1


def test_w0_rows_match_full_array():
    cfg = W.config(4)
    cfg = W.scaled(cfg, 2000, 64)
    keys = W.table_keys(cfg)
    off = W.elem_offsets(cfg, keys)
    full = W.w0_values(cfg, int(off[-1]))
    rows = torch.tensor([0, 5, 17, keys.numel() - 1])
    dims = torch.tensor(cfg.dims)[keys[rows] >> 48]
    got = W.w0_rows(cfg, off, rows, dims)
    exp = torch.cat([full[off[r]:off[r + 1]] for r in rows.tolist()])
    assert torch.equal(got, exp)
