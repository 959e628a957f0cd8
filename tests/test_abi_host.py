"""The C-ABI library without a GPU: symbols, host-side table preparation and
input validation (emb_table_plan makes no CUDA call)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workload as W
import sparse_ctr_embedding_gb300 as E


@pytest.fixture(scope="module", autouse=True)
def built():
    E.build()


def test_library_exports_every_declared_symbol():
    declared = E.declared_symbols()
    assert len(declared) >= 14
    L = E.lib()
    for name in declared:
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value
    assert E.emb_status_string(0) == "ok"


def test_binding_constants_match_the_header():
    import re
    text = open(E.HEADER).read()
    defs = {m.group(1): m.group(2) for m in re.finditer(r"^#define (EMB_\w+)\s+\(?([0-9]+u?(?: << [0-9]+)?)\)?", text, re.M)}
    val = lambda v: eval(v.replace("u", ""))
    assert val(defs["EMB_NOALLOC_SCRATCH_BYTES"]) == E.EMB_NOALLOC_SCRATCH_BYTES
    assert val(defs["EMB_SORT_DIGIT_BITS"]) == E.EMB_SORT_DIGIT_BITS
    assert val(defs["EMB_BWD_PHASES"]) == len(E.BWD_PHASES)
    for f in ["EMB_FLAG_PROBE_BOUND", "EMB_FLAG_BAD_OFFSETS", "EMB_FLAG_SLOT_MISMATCH", "EMB_FLAG_BAD_ROW"]:
        assert val(defs[f]) == getattr(E, f)


@pytest.mark.parametrize("cfg", [W.config(1), W.scaled(W.config(2), 100, 1), W.scaled(W.config(4), 200, 1),
                                 W.scaled(W.config(5), 1000, 1)], ids=lambda c: c.name)
def test_host_layout_matches_oracle_bit_exact(cfg):
    keys = W.table_keys(cfg).numpy()
    st, sk, sr = E.emb_table_plan(cfg.dims, cfg.wdtype, keys, cfg.capacity, layout=True)
    T = oracle.Table(keys, cfg.capacity, cfg.dims)
    ok_, or_ = T.layout()
    assert np.array_equal(sk, ok_)
    assert np.array_equal(sr, or_)
    assert st["max_probe"] == T.max_probe
    assert st["sum_probe"] == T.sum_probe
    assert st["max_cluster"] == T.max_cluster
    assert st["probe_bound"] == T.max_cluster + 1
    assert st["n_elems"] == T.n_elems
    assert st["capacity"] == cfg.capacity and st["sum_dims"] == cfg.sum_dims


def test_auto_capacity_is_smallest_power_of_two_at_half_load():
    for n in [1, 2, 3, 1000, 65536, 65537]:
        keys = np.arange(n, dtype=np.int64)
        st, _, _ = E.emb_table_plan([4], "f32", keys, 0)
        cap = st["capacity"]
        assert cap >= 2 * n and cap & (cap - 1) == 0 and (cap // 2 < 2 * n or cap == 2)


@pytest.mark.parametrize("keys,dims,wd,cap,err", [
    ([1, 2, 1], [4], "f32", 8, "EMB_ERR_DUP_KEY"),
    ([1, -1], [4], "f32", 8, "EMB_ERR_RESERVED_KEY"),
    ([(2 << 48) | 5], [4, 4], "f32", 8, "EMB_ERR_INVALID_ARG"),   # slot field >= n_slots
    ([1, 2, 3], [4], "f32", 4, "EMB_ERR_LOAD_FACTOR"),             # 3 keys need 8 slots
    ([1, 2], [4], "f32", 12, "EMB_ERR_LOAD_FACTOR"),               # not a power of two
    ([1, 2], [6], "f32", 8, "EMB_ERR_UNSUPPORTED"),                # f32 dim not multiple of 4
    ([1, 2], [4], "f16", 8, "EMB_ERR_UNSUPPORTED"),                # f16 dim not multiple of 8
    ([1, 2], [1024], "f32", 8, "EMB_ERR_UNSUPPORTED"),             # above EMB_MAX_DIM
])
def test_plan_rejects_bad_tables(keys, dims, wd, cap, err):
    with pytest.raises(E.EmbError) as ei:
        E.emb_table_plan(dims, wd, np.array(keys, dtype=np.int64), cap)
    assert ei.value.name == err
    assert E.emb_last_error()


def test_plan_stats_count_probes():
    # every key of a tiny table lands at probe length >= 1; the sum counts them
    keys = (np.arange(40, dtype=np.int64) * 7919) | (1 << 48)
    st, sk, sr = E.emb_table_plan([8, 8], "f32", keys, 128, layout=True)
    assert st["n_keys"] == 40 and (sk != -1).sum() == 40
    assert st["sum_probe"] >= 40 and st["max_probe"] >= 1
    assert sorted(sr[sr >= 0].tolist()) == list(range(40))


def test_master_copy_tables_plan_like_f16_tables():
    cfg = W.scaled(W.config(5), 2000, 1)
    keys = W.table_keys(cfg).numpy()
    st16, sk16, sr16 = E.emb_table_plan(cfg.dims, "f16", keys, cfg.capacity, layout=True)
    stm, skm, srm = E.emb_table_plan(cfg.dims, "f16m", keys, cfg.capacity, layout=True)
    assert np.array_equal(sk16, skm) and np.array_equal(sr16, srm)
    assert stm["wdtype"] == 2 and stm["n_elems"] == st16["n_elems"]
    with pytest.raises(E.EmbError):
        E.emb_table_plan([12], "f16m", keys[:4] & ((1 << 48) - 1), 16)     # f16 rows need dims % 8 == 0



def test_plan_accepts_each_optimizer_and_rejects_an_unknown_one():
    keys = (np.arange(20, dtype=np.int64) * 7919) | (1 << 48)
    base, sk0, _ = E.emb_table_plan([8, 8], "f32", keys, 64, layout=True)
    for opt in ("ftrl", "rowwise_adagrad"):          # the optimizer changes no part of the layout
        st, sk, _ = E.emb_table_plan([8, 8], "f32", keys, 64, layout=True, optimizer=opt)
        assert np.array_equal(sk, sk0) and st["n_elems"] == base["n_elems"]
    d, _keep = E._desc([8, 8], "f32", 64, 0.0)
    d.optimizer = 3
    s = E._Stats()
    with pytest.raises(E.EmbError) as ei:
        E._check(E.lib().emb_table_plan(ctypes.byref(d), keys.ctypes.data, keys.size, ctypes.byref(s), None, None))
    assert ei.value.name == "EMB_ERR_INVALID_ARG"


def test_failed_create_returns_oom_and_leaves_nothing_allocated():
    """Fault injection on the host: the table's first device allocation fails;
    create must return EMB_ERR_OOM (not abort) and hold no device memory.
    Nothing reaches CUDA, so this runs without a GPU."""
    import gc
    keys = torch.tensor([(0 << 48) | 5, (1 << 48) | 7], dtype=torch.int64)
    gc.collect()
    gc.disable()
    live0 = E.emb_debug_live_device_allocs()
    E.emb_debug_fail_device_alloc(0)
    try:
        with pytest.raises(E.EmbError) as ei:
            E.emb_table_create([8, 8], "f32", keys, capacity=8, stream=0)   # no torch stream on a CPU machine
    finally:
        E.emb_debug_fail_device_alloc(-1)
        gc.enable()
    assert ei.value.name == "EMB_ERR_OOM"
    assert E.emb_debug_live_device_allocs() == live0
