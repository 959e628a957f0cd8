"""emb_table_create_device: the table prepared on the GPU must be exactly the
host-prepared one (emb_table_plan / emb_table_create): the slot layout (key and
keys-array index per slot), the statistics, the row numbering (checked through
the export and a forward), and the same errors.  Besides the five workloads'
tables (scaled), tables built from keys chosen by their hash: many homes just
before the end of the table (the layout wraps), runs longer than one warp
replays, and a run longer than the device build takes."""
import gc

import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E

pytestmark = pytest.mark.gpu

STAT_KEYS = ("n_keys", "capacity", "n_elems", "n_slots", "sum_dims", "max_dim", "wdtype", "max_probe", "sum_probe",
             "max_cluster", "probe_bound", "load_factor", "max_slot_keys")


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"


def _layout(tbl):
    cap = tbl.stats["capacity"]
    sk = torch.empty(cap, dtype=torch.int64, device="cuda")
    sr = torch.empty(cap, dtype=torch.int64, device="cuda")
    E.emb_table_slots(tbl, sk, sr)
    return sk.cpu().numpy(), sr.cpu().numpy()


def _same_as_host(dims, wdtype, keys, capacity=0, values=None):
    keys_h = torch.as_tensor(keys, dtype=torch.int64)
    st_h, sk_h, sr_h = E.emb_table_plan(dims, wdtype, keys_h.numpy(), capacity=capacity, layout=True)
    dev = E.emb_table_create_device(dims, wdtype, keys_h.cuda(), values=values, capacity=capacity, acc_init=0.1)
    for k in STAT_KEYS:
        assert dev.stats[k] == st_h[k], (k, dev.stats[k], st_h[k])
    sk, sr = _layout(dev)
    assert np.array_equal(sk, sk_h) and np.array_equal(sr, sr_h)
    return dev, st_h


def _keys_with_homes(rng, slot, n, cap, lo, hi):
    """n distinct keys of `slot` whose home fmix64(key) mod cap lies in [lo, hi] (wrapping)."""
    out = []
    seen = set()
    while len(out) < n:
        raw = rng.integers(1, 1 << 47, size=1 << 20, dtype=np.int64)
        k = (np.int64(slot) << 48) | raw
        hh = _fmix64_np(k.view(np.uint64)) & np.uint64(cap - 1)
        sel = ((hh - np.uint64(lo)) & np.uint64(cap - 1)) <= np.uint64((hi - lo) & (cap - 1))
        for x in k[sel]:
            if int(x) not in seen:
                seen.add(int(x))
                out.append(int(x))
                if len(out) == n:
                    break
    return np.array(out, dtype=np.int64)


def _fmix64_np(k):
    """MurmurHash3's 64-bit finaliser on a uint64 array (numpy wraps modulo 2^64), checked
    against the oracle's fmix64 below before use."""
    k = k.copy()
    k ^= k >> np.uint64(33)
    k *= np.uint64(0xFF51AFD7ED558CCD)
    k ^= k >> np.uint64(33)
    k *= np.uint64(0xC4CEB9FE1A85EC53)
    k ^= k >> np.uint64(33)
    return k


def test_numpy_hash_helper_agrees_with_the_oracle():
    rng = np.random.default_rng(3)
    k = rng.integers(-(1 << 62), 1 << 62, size=1000, dtype=np.int64)
    got = _fmix64_np(k.view(np.uint64))
    assert all(int(g) == oracle.fmix64(int(x)) for g, x in zip(got, k))


@pytest.mark.parametrize("cfg", [W.config(1), W.scaled(W.config(2), 100, 4), W.scaled(W.config(3), 500, 16),
                                 W.scaled(W.config(4), 250, 8), W.scaled(W.config(5), 1000, 64)],
                         ids=lambda c: c.name)
def test_device_build_equals_host_build(cfg):
    wl = W.make(cfg, device="cuda")
    dev, _ = _same_as_host(cfg.dims, cfg.wdtype, wl.keys.cpu().numpy(), cfg.capacity, values=wl.values.cuda())
    host = E.emb_table_create(cfg.dims, cfg.wdtype, wl.keys.cpu(), values=wl.values.cuda(), capacity=cfg.capacity,
                              acc_init=0.1)
    # row numbering: the export (keys-array order) and a forward are identical
    n_el = host.stats["n_elems"]
    outs = []
    for t in (dev, host):
        ko = torch.empty(cfg.n_keys, dtype=torch.int64, device="cuda")
        vo = torch.empty(n_el, dtype=wl.values.dtype, device="cuda")
        ao = torch.empty(n_el, dtype=torch.float32, device="cuda")
        E.emb_table_export(t, ko, vo, ao)
        outs.append((ko, vo, ao, E.emb_lookup_fwd(t, wl.offsets, wl.qkeys, cfg.pool)))
    for a, b in zip(*outs):
        assert torch.equal(a, b)
    assert E.emb_check_device_flag(dev) == 0


def test_full_size_26_slot_table_equals_host_build():
    cfg = W.config(2)
    keys = W.table_keys(cfg, torch.device("cuda"))
    _same_as_host(cfg.dims, cfg.wdtype, keys.cpu().numpy(), cfg.capacity)


def test_layout_that_wraps_around_the_end():
    rng = np.random.default_rng(5)
    cap = 1 << 12
    near_end = _keys_with_homes(rng, 0, 600, cap, cap - 40, cap - 1)      # spill past the last slot
    rest = _keys_with_homes(rng, 1, 1200, cap, 0, cap - 1)
    keys = np.concatenate([near_end, rest])
    keys = keys[rng.permutation(keys.size)]
    dev, st = _same_as_host([8, 8], "f32", keys, cap)
    assert st["max_cluster"] > 500


def test_runs_longer_than_a_warp_and_the_too_long_refusal():
    rng = np.random.default_rng(6)
    cap = 1 << 14
    window = _keys_with_homes(rng, 0, 1500, cap, 5000, 5020)              # one run of about 1500 keys
    rest = _keys_with_homes(rng, 1, 3000, cap, 0, cap - 1)
    keys = np.concatenate([window, rest])
    keys = keys[rng.permutation(keys.size)]
    _, st = _same_as_host([8, 16], "f32", keys, cap)
    assert st["max_cluster"] > 1000
    huge = _keys_with_homes(rng, 0, 4200, cap, 9000, 9010)                # a run beyond 4096: refused
    with pytest.raises(E.EmbError) as ei:
        E.emb_table_create_device([8], "f32", torch.from_numpy(huge).cuda(), capacity=cap)
    assert ei.value.name == "EMB_ERR_UNSUPPORTED"
    E.emb_table_plan([8], "f32", huge, capacity=cap)                      # the host build takes it


@pytest.mark.parametrize("case", ["dup", "reserved", "badslot"])
def test_device_build_errors_match_the_host(case):
    rng = np.random.default_rng(7)
    keys = (np.int64(0) << 48) | rng.choice(1 << 40, size=5000, replace=False).astype(np.int64)
    if case == "dup":
        keys[4000] = keys[123]
        keys[2500] = keys[77]
    elif case == "reserved":
        keys[3000] = -1
        keys[4000] = np.int64(3) << 48
    else:
        keys[3000] = np.int64(3) << 48
        keys[4000] = -1
    with pytest.raises(E.EmbError) as eh:
        E.emb_table_plan([8], "f32", keys)
    keys_d = torch.from_numpy(keys).cuda()
    gc.collect()                      # tables of earlier tests are freed now, not during the count
    gc.disable()
    try:
        live0 = E.emb_debug_live_device_allocs()
        with pytest.raises(E.EmbError) as ed:
            E.emb_table_create_device([8], "f32", keys_d)
        live1 = E.emb_debug_live_device_allocs()
    finally:
        gc.enable()
    assert ed.value.name == eh.value.name
    if case == "dup":
        assert ed.value.message == eh.value.message              # the same keys-array index
    assert live1 == live0                                       # nothing left allocated
